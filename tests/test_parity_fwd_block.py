"""Forward parity of the per-block kernel on small shapes (GPU).

The forward has two tcgen05 kernels: a persistent one for items that
average at most 16 kv steps per 256-row query block, and one CTA per query
block above that.  Small parity shapes all fall below the limit, so these
cases are sized to exceed it: dense causal N >= 4096 (N / 256 + 1 > 16 steps),
non-causal N > 2048 (N / 128 > 16), a causal band no narrower than 1920 keys
((w + 256) / 128 + 1 > 16).  Each covers a path of the per-block kernel the
full-size workloads do not: d = 64, no mask, ALiBi without a mask, a band,
and a ragged last query block whose second tile is partly or wholly past the
sequence end.  Tolerances as in test_parity_fwd (O stored fp32).
"""
import numpy as np
import pytest

from oracle import attention_fp64 as A
from exact_io_aware_36_gb300 import inputs as I
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE = 1e-2, 1e-3


def avg_kv_steps(w):
    """Average kv steps of a query block, as the forward's dispatch counts them."""
    steps = w.N // 256 + 1 if w.causal else (w.N + 127) // 128
    if w.causal and w.window is not None:
        steps = min(steps, (w.window + 256) // 128 + 1)
    return steps


CASES = [
    # B, Hq, Hkv, N, d, causal, alibi, window
    (1, 2, 1, 4100, 64, True, False, None),      # second tile of the last block: 4 rows
    (1, 1, 1, 4097, 128, True, True, None),      # last block: one row
    (1, 2, 1, 2100, 64, False, False, None),
    (1, 1, 1, 2200, 128, False, True, None),
    (1, 1, 1, 4500, 128, True, False, 2000),
    (2, 1, 1, 4224, 128, True, False, None),     # last block: first tile only
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal,alibi,window", CASES)
def test_block_forward(B, Hq, Hkv, N, d, causal, alibi, window):
    w = I.small_case("bf16", causal=causal, B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, alibi=alibi,
                     window=window, backward=False)
    assert avg_kv_steps(w) > 16                  # the per-block kernel takes this shape
    x = I.make_inputs(w, seed=N + d)
    O, lse = G.forward(x)
    O_ref, lse_ref = A.attention_forward(x.q, x.k, x.v, x.scale, causal, x.cu_seqlens,
                                         x.alibi_slopes, window=window)
    eo, el = np.max(np.abs(O - O_ref)), np.max(np.abs(lse - lse_ref))
    assert eo <= TOL_O, f"O max abs err {eo}"
    assert el <= TOL_LSE, f"LSE max abs err {el}"
