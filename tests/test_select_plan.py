"""Host logic of the streamed selection's sizing: the shared list of the
select kernel holds a row's candidates plus its samples at or above the
threshold, exactly r = threshold_rank(S, n, k) of them.  The library sizes
that part of the list by a closed-form bound on r (csrc/select.cu,
plan_select); this test checks the bound against every row length n of
several cache sizes, with r and S computed as the kernels compute them."""
import math

import pytest

SAMPLE_TILES = 32   # sampled key tiles per row at most (128 keys each)


def _plan_m(max_kv):
    t = (max_kv + 127) // 128
    return max(1, (t + SAMPLE_TILES - 1) // SAMPLE_TILES)


def _threshold_rank(s, n, k):
    f = s * k / n
    r = math.ceil(f + 6.0 * math.sqrt(f) + 16.0)
    return s if r >= s else r


def _samples(pos, m):
    slots = (pos // (m * 128) + 1) * 128
    return slots - 128 + min(128, pos - (slots // 128 - 1) * m * 128 + 1)


@pytest.mark.parametrize("max_kv,k", [(4096, 2048), (32768, 2048), (65536, 2048), (131072, 2048),
                                      (32768, 8192), (131072, 8192), (20000, 100)])
def test_sample_rank_bound_covers_every_row(max_kv, k):
    m = _plan_m(max_kv)
    t = (max_kv + 127) // 128
    lds = ((t + m - 1) // m) * 128
    big_f = k / m + 128.0
    bound = min(lds, math.ceil(big_f + 6.0 * math.sqrt(big_f) + 16.0))
    worst = max(_threshold_rank(_samples(n - 1, m), n, k) for n in range(k + 1, max_kv + 1))
    assert worst <= bound, (worst, bound)
