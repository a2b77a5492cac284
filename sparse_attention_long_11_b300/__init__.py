"""DeepSeek Sparse Attention (DSA) hot path for NVIDIA B300 (sm_103a).

The compute lives in ``libdsa.so`` (hand-written CUDA behind a C ABI, see
``include/dsa.h``); ``api`` is a thin ctypes binding over it.  Importing the
package does not load the library; the first call into ``api`` does, and it
raises if the library has not been built.
"""
