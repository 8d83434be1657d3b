"""Backward parity: the CUDA path against the fp64 oracle (GPU).

Tolerances: O <= 1e-2 and LSE <= 1e-3 max abs error (O stored fp32);
dQ, dK, dV: max abs error <= 2e-2 x max|grad| of that tensor in the oracle.
"""
import numpy as np
import pytest

from oracle import attention_fp64 as A
from exact_io_aware_36_gb300 import inputs as I
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE, TOL_GRAD = 1e-2, 1e-3, 2e-2


def check(x, res):
    w = x.workload
    O, lse, dq, dk, dv = res
    dq_r, dk_r, dv_r, O_r, lse_r, _ = A.attention_backward(
        x.q, x.k, x.v, x.do, x.scale, w.causal, x.cu_seqlens, x.alibi_slopes, window=w.window)
    errs = {}
    if O.size:
        errs["O"] = np.abs(O - O_r).max()
        errs["LSE"] = np.abs(lse - lse_r).max()
        for name, a, r in (("dQ", dq, dq_r), ("dK", dk, dk_r), ("dV", dv, dv_r)):
            errs[name] = np.abs(a - r).max() / max(np.abs(r).max(), 1e-30)
    assert errs.get("O", 0) <= TOL_O, errs
    assert errs.get("LSE", 0) <= TOL_LSE, errs
    for name in ("dQ", "dK", "dV"):
        assert errs.get(name, 0) <= TOL_GRAD, errs
    return errs


CASES = [
    # B, Hq, Hkv, N, d, causal, alibi
    (1, 1, 1, 128, 128, True, False),
    (1, 1, 1, 128, 64, True, False),
    (1, 2, 2, 256, 128, False, False),
    (2, 2, 1, 200, 64, True, False),
    (1, 4, 2, 333, 128, True, True),
    (1, 1, 1, 1, 128, True, False),
    (1, 2, 2, 65, 64, False, True),
    (2, 8, 1, 520, 128, True, False),
    (1, 3, 3, 1024, 64, True, True),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal,alibi", CASES)
def test_bwd_dense(B, Hq, Hkv, N, d, causal, alibi):
    w = I.small_case("bf16", causal=causal, B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, alibi=alibi)
    x = I.make_inputs(w, seed=100 + N)
    check(x, G.backward(x))


@pytest.mark.parametrize("seqlens,d,causal,alibi", [
    ((5, 300, 1, 128, 129), 128, True, False),
    ((256, 255, 257), 64, True, True),
    ((17, 600, 3), 128, False, False),
    ((0, 40, 0, 1), 64, True, False),
])
def test_bwd_varlen(seqlens, d, causal, alibi):
    w = I.small_case("bf16", causal=causal, Hq=4, Hkv=2, d=d, alibi=alibi, seqlens=seqlens)
    x = I.make_inputs(w, seed=5)
    check(x, G.backward(x))


def test_bwd_bf16_output_o():
    """The backward also accepts O stored as bf16 (D = dO . O from bf16 O)."""
    t = pytest.importorskip("torch")
    w = I.small_case("bf16", causal=True, B=1, Hq=2, Hkv=2, N=256, d=128)
    x = I.make_inputs(w, seed=8)
    O, lse, dq, dk, dv = G.backward(x, out_dtype=t.bfloat16)
    dq_r, dk_r, dv_r, *_ = A.attention_backward(x.q, x.k, x.v, x.do, x.scale, True)
    for a, r in ((dq, dq_r), (dk, dk_r), (dv, dv_r)):
        assert np.abs(a - r).max() <= TOL_GRAD * np.abs(r).max()


def test_bwd_repeatable_within_tolerance():
    """Two runs agree to the fp32 reduction-order noise of dQ."""
    w = I.small_case("bf16", causal=True, B=1, Hq=4, Hkv=1, N=700, d=128)
    x = I.make_inputs(w, seed=2)
    r1 = G.backward(x)
    r2 = G.backward(x)
    np.testing.assert_array_equal(r1[3], r2[3])   # dK: fixed order in TMEM
    np.testing.assert_array_equal(r1[4], r2[4])   # dV
    assert np.abs(r1[2] - r2[2]).max() <= 1e-2 * np.abs(r1[2]).max()


def _bwd_with_workspace(x, ws_bytes, deterministic):
    """fa_fwd + fa_bwd with a workspace of exactly ws_bytes; torch tensors."""
    t = G.torch()
    from exact_io_aware_36_gb300 import fa
    w = x.workload
    q, k, v, do = (G.to_dev(x, n) for n in ("q", "k", "v", "do"))
    cu = t.from_numpy(x.cu_seqlens).cuda() if w.varlen else None
    slopes = t.from_numpy(x.alibi_slopes).cuda() if x.alibi_slopes is not None else None
    kw = dict(causal=w.causal, scale=x.scale, cu_seqlens=cu, max_seqlen=w.N if w.varlen else None,
              batch=None if w.varlen else w.B, alibi_slopes=slopes, window=w.window, check=True)
    o, lse = fa.attention_forward(q, k, v, out_dtype=t.float32, **kw)
    ws = t.empty(ws_bytes, dtype=t.uint8, device="cuda")
    dq, dk, dv = fa.attention_backward(q, k, v, o, do, lse, workspace=ws,
                                       deterministic=deterministic, **kw)
    t.cuda.synchronize()
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,N,d,alibi,seqlens,window", [
    (2, 8, 1, 700, 128, True, None, None),       # MQA: the group of 8 in two halves
    (1, 8, 2, 513, 64, False, None, None),
    (1, 4, 2, 0, 128, False, (300, 1, 129), None),
    (1, 8, 4, 900, 128, False, None, 200),
])
def test_gqa_split_dkdv(B, Hq, Hkv, N, d, alibi, seqlens, window, deterministic):
    """With fa_bwd_workspace_size_gqa bytes the dK/dV work of each GQA group
    is split in two blocks whose sums the last stage adds in a fixed order:
    the oracle's tolerances hold, repeats are bit-identical (dK, dV; dQ too
    in the deterministic mode), and the result stays within rounding of the
    unsplit one (the base workspace size)."""
    from exact_io_aware_36_gb300 import fa
    w = I.small_case("bf16", causal=True, B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, alibi=alibi,
                     seqlens=seqlens, window=window)
    x = I.make_inputs(w, seed=17)
    base = fa.fa_bwd_workspace_size(w.B, w.Hq, w.N, w.d, x.T)
    big = fa.fa_bwd_workspace_size_gqa(w.B, w.Hq, w.Hkv, w.N, w.d, x.T)
    assert big > base
    r1 = _bwd_with_workspace(x, big, deterministic)
    r2 = _bwd_with_workspace(x, big, deterministic)
    r0 = _bwd_with_workspace(x, base, deterministic)
    t = G.torch()
    for i in (3, 4) + ((2,) if deterministic else ()):
        assert t.equal(r1[i], r2[i]), i
    res = [G.as_f64(a) for a in r1]
    check(x, res)
    for i in (2, 3, 4):
        a, b = res[i], G.as_f64(r0[i])
        assert np.abs(a - b).max() <= 1e-2 * max(np.abs(b).max(), 1e-30), i
