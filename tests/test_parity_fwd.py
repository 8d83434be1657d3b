"""Forward parity: the CUDA path against the fp64 oracle (GPU).

Tolerances: fp32 workload: max abs error <= 1e-5 on O and LSE.  bf16
workloads: max abs error <= 1e-2 on O and <= 1e-3 on LSE, with O stored as
fp32 (inputs are bf16-exact on both sides, so the error is the kernel's
arithmetic: bf16 P in the PV product, fp32 accumulation).  When O is stored
as bf16, the storage itself rounds by up to half a bf16 ulp (<= 2^-8 |O|),
which that test adds to the 1e-2 bound.
"""
import json
import os

import numpy as np
import pytest

from oracle import attention_fp64 as A
from exact_io_aware_36_gb300 import inputs as I
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

TOL_O_BF16, TOL_LSE_BF16, TOL_FP32 = 1e-2, 1e-3, 1e-5


def check_full(x, O, lse, tol_o, tol_lse, o_storage_rel=0.0):
    w = x.workload
    O_ref, lse_ref = A.attention_forward(x.q, x.k, x.v, x.scale, w.causal, x.cu_seqlens,
                                         x.alibi_slopes)
    if O.size:
        excess = np.abs(O - O_ref) - (tol_o + o_storage_rel * np.abs(O_ref))
        eo = np.max(np.abs(O - O_ref))
        assert excess.max() <= 0, f"O max abs err {eo} (excess {excess.max()})"
    if lse.size:
        el = np.max(np.abs(lse - lse_ref))
        assert el <= tol_lse, f"LSE max abs err {el}"


def test_fp32_workload_matches_oracle():
    w = I.workload("c1_fp32_fwd")
    x = I.make_inputs(w, seed=0)
    O, lse = G.forward(x)
    check_full(x, O, lse, TOL_FP32, TOL_FP32)
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "c1_fp32_rows.json")))
    for n, t in enumerate(gold["rows"]):
        assert np.max(np.abs(O[t, 0] - np.array(gold["O"][n]))) <= TOL_FP32
        assert abs(lse[0, t] - gold["LSE"][n]) <= TOL_FP32


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d,Hq,Hkv", [(1, 64, 1, 1), (33, 32, 2, 1), (200, 128, 4, 2),
                                         (77, 100, 2, 2)])
def test_fp32_shapes(causal, N, d, Hq, Hkv):
    w = I.small_case("fp32", causal=causal, B=2, Hq=Hq, Hkv=Hkv, N=N, d=d, backward=False)
    x = I.make_inputs(w, seed=11)
    O, lse = G.forward(x)
    check_full(x, O, lse, TOL_FP32, TOL_FP32)


@pytest.mark.parametrize("causal", [False, True])
def test_fp32_alibi_packed_odd_d(causal):
    # packed lengths around the 32-key tile and the 4-row block (1, 3, 31..33,
    # 100), GQA, ALiBi, and d = 37: rows and head columns with ragged tails
    w = I.small_case("fp32", causal=causal, Hq=4, Hkv=2, d=37, alibi=True,
                     seqlens=(1, 3, 31, 32, 33, 100), backward=False)
    x = I.make_inputs(w, seed=12)
    O, lse = G.forward(x)
    check_full(x, O, lse, TOL_FP32, TOL_FP32)


BF16_CASES = [
    # B, Hq, Hkv, N, d, causal, alibi
    (1, 1, 1, 128, 64, True, False),
    (1, 2, 2, 256, 128, True, False),
    (2, 2, 2, 129, 64, True, False),
    (1, 1, 1, 1, 128, True, False),
    (1, 2, 2, 17, 64, False, False),
    (1, 2, 1, 255, 128, False, False),
    (2, 4, 2, 300, 64, True, True),
    (1, 4, 1, 513, 128, True, True),
    (1, 2, 2, 640, 128, False, True),
    (3, 3, 3, 384, 64, True, False),
    (1, 8, 1, 1000, 128, True, False),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal,alibi", BF16_CASES)
def test_bf16_dense(B, Hq, Hkv, N, d, causal, alibi):
    w = I.small_case("bf16", causal=causal, B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, alibi=alibi)
    x = I.make_inputs(w, seed=N + d)
    O, lse = G.forward(x)
    check_full(x, O, lse, TOL_O_BF16, TOL_LSE_BF16)


@pytest.mark.parametrize("seqlens,d,causal,alibi", [
    ((5, 300, 1, 128, 129), 128, True, False),
    ((256, 255, 257), 64, True, True),
    ((17, 600, 3), 128, False, False),
    ((0, 40, 0, 1), 64, True, False),       # empty sequences
])
def test_bf16_varlen(seqlens, d, causal, alibi):
    w = I.small_case("bf16", causal=causal, Hq=4, Hkv=2, d=d, alibi=alibi, seqlens=seqlens)
    x = I.make_inputs(w, seed=3)
    O, lse = G.forward(x)
    check_full(x, O, lse, TOL_O_BF16, TOL_LSE_BF16)


@pytest.mark.parametrize("d,alibi", [(64, True), (128, False)])
def test_bf16_output_storage(d, alibi):
    """O stored as bf16: within 1e-2 plus half a bf16 ulp of O."""
    t = pytest.importorskip("torch")
    w = I.small_case("bf16", causal=True, B=2, Hq=4, Hkv=2, N=300, d=d, alibi=alibi)
    x = I.make_inputs(w, seed=9)
    O, lse = G.forward(x, out_dtype=t.bfloat16)
    check_full(x, O, lse, TOL_O_BF16, TOL_LSE_BF16, o_storage_rel=2.0 ** -8)


def test_qk_gain_workload_small():
    """The long-context recipe (q, k scaled by 0.5) at a size the oracle runs whole."""
    w = I.small_case("bf16", causal=True, B=1, Hq=2, Hkv=2, N=2048, d=128, qk_gain=0.5)
    x = I.make_inputs(w, seed=0)
    O, lse = G.forward(x)
    check_full(x, O, lse, TOL_O_BF16, TOL_LSE_BF16)
