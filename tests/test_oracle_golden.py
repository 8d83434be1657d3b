"""The oracle still reproduces its committed fixtures (CPU only), and the
softmax-gradient invariant sum_j dS_ij = 0 (so the dK rows of a sequence and
kv head sum to zero) holds on them."""
import json
import os

import numpy as np

from oracle import attention_fp64 as A
from exact_io_aware_36_gb300 import inputs as I
from tests.golden import make_golden as G

HERE = os.path.join(os.path.dirname(__file__), "golden")


def test_c1_fixture_reproduced():
    ref = json.load(open(os.path.join(HERE, "c1_fp32_rows.json")))
    now = G.c1_fixture()
    np.testing.assert_allclose(now["O"], ref["O"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(now["LSE"], ref["LSE"], rtol=0, atol=1e-14)
    assert abs(now["O_sum"] - ref["O_sum"]) < 1e-10


def test_small_backward_fixture_reproduced():
    ref = json.load(open(os.path.join(HERE, "small_bwd_sums.json")))
    now = G.small_bwd_fixture()
    for k, v in ref["sums"].items():
        assert abs(now["sums"][k] - v) <= 1e-9 * max(1.0, abs(v)), k
    for k, v in ref["absmax"].items():
        assert abs(now["absmax"][k] - v) <= 1e-12 * max(1.0, abs(v)), k


def test_dk_rows_sum_to_zero():
    w = I.small_case("bf16", causal=True, Hq=4, Hkv=2, d=32, alibi=True, seqlens=(9, 40))
    x = I.make_inputs(w, seed=3)
    dq, dk, dv, *_ = A.attention_backward(x.q, x.k, x.v, x.do, w.scale, True,
                                          x.cu_seqlens, x.alibi_slopes)
    cu = x.cu_seqlens
    for b in range(len(cu) - 1):
        s = dk[cu[b]:cu[b + 1]].sum(0)
        assert np.abs(s).max() < 1e-12 * max(1.0, np.abs(dk).max())
