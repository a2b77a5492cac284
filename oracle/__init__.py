"""CPU oracle for the DSA hot path -- test infrastructure only.

Imported by the tests, the smoke check and the benchmark's CPU-baseline leg;
never by the library.
"""
from .dsa_oracle import (decode_bf16, decode_e4m3, dense_causal_mqa, dsa_query,  # noqa: F401
                         index_scores, sparse_attention, topk_select)
