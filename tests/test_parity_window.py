"""Sliding-window (causal band) parity: the CUDA path against the fp64 oracle (GPU).

Key j is visible to query i iff i - w <= j <= i.  Tolerances as in the other
parity tests: fp32 forward 1e-5; bf16 O 1e-2 (stored fp32), LSE 1e-3, each
gradient 2e-2 x max|grad| of that tensor in the oracle.

Windows are chosen around the tile edges of the kernels: the forward visits
K/V in tiles of 128 keys for query tiles of 128 rows, the backward query
tiles of 64 rows per key tile of 128.  w = 0 (each query sees only itself),
w = N - 1 (the plain causal mask) and w >= N are included.
"""
import numpy as np
import pytest

from oracle import attention_fp64 as A
from exact_io_aware_36_gb300 import inputs as I
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE, TOL_GRAD, TOL_FP32 = 1e-2, 1e-3, 2e-2, 1e-5


def _oracle_fwd(x):
    w = x.workload
    return A.attention_forward(x.q, x.k, x.v, x.scale, True, x.cu_seqlens, x.alibi_slopes,
                               window=w.window)


@pytest.mark.parametrize("N,d,window", [
    (300, 64, 0), (300, 128, 1), (513, 64, 63), (513, 128, 64), (640, 64, 127),
    (640, 128, 128), (700, 64, 129), (1000, 128, 255), (1000, 64, 256), (1100, 128, 300),
    (257, 64, 255), (257, 128, 256), (257, 64, 5000),
])
def test_fwd_window(N, d, window):
    w = I.small_case("bf16", causal=True, B=2, Hq=4, Hkv=2, N=N, d=d, window=window)
    x = I.make_inputs(w, seed=N + window)
    O, lse = G.forward(x)
    O_r, lse_r = _oracle_fwd(x)
    assert np.abs(O - O_r).max() <= TOL_O
    assert np.abs(lse - lse_r).max() <= TOL_LSE


@pytest.mark.parametrize("alibi,seqlens,window", [
    (True, None, 100), (True, None, 383),
    (False, (5, 300, 1, 700, 129), 200), (True, (256, 255, 600), 64),
])
def test_fwd_window_alibi_varlen(alibi, seqlens, window):
    if seqlens is None:
        w = I.small_case("bf16", causal=True, B=1, Hq=4, Hkv=1, N=900, d=128, alibi=alibi,
                         window=window)
    else:
        w = I.small_case("bf16", causal=True, Hq=4, Hkv=2, d=64, alibi=alibi, seqlens=seqlens,
                         window=window)
    x = I.make_inputs(w, seed=3)
    O, lse = G.forward(x)
    O_r, lse_r = _oracle_fwd(x)
    assert np.abs(O - O_r).max() <= TOL_O
    assert np.abs(lse - lse_r).max() <= TOL_LSE


@pytest.mark.parametrize("N,d,window", [(200, 64, 0), (333, 100, 37), (500, 128, 64),
                                        (129, 32, 128)])
def test_fp32_window(N, d, window):
    w = I.small_case("fp32", causal=True, B=2, Hq=2, Hkv=1, N=N, d=d, window=window,
                     backward=False)
    x = I.make_inputs(w, seed=21)
    O, lse = G.forward(x)
    O_r, lse_r = _oracle_fwd(x)
    assert np.abs(O - O_r).max() <= TOL_FP32
    assert np.abs(lse - lse_r).max() <= TOL_FP32


# Floor of the gradient scale: with w = 0 each query sees only its own key,
# so P = 1, dS = P o (dP - D) = 0 and dQ = dK = 0 exactly; the kernel's values
# are then rounding noise (dP_ii and D_i are the same dot product dO_i . v_i
# summed in different orders, ~1e-6), which a scale of 0 would turn into an
# unbounded relative error.
GRAD_SCALE_FLOOR = 1e-3


def check_bwd(x, res):
    w = x.workload
    O, lse, dq, dk, dv = res
    dq_r, dk_r, dv_r, O_r, lse_r, _ = A.attention_backward(
        x.q, x.k, x.v, x.do, x.scale, True, x.cu_seqlens, x.alibi_slopes, window=w.window)
    errs = {"O": np.abs(O - O_r).max(), "LSE": np.abs(lse - lse_r).max()}
    for name, a, r in (("dQ", dq, dq_r), ("dK", dk, dk_r), ("dV", dv, dv_r)):
        errs[name] = np.abs(a - r).max() / max(np.abs(r).max(), GRAD_SCALE_FLOOR)
    assert errs["O"] <= TOL_O and errs["LSE"] <= TOL_LSE, errs
    assert max(errs["dQ"], errs["dK"], errs["dV"]) <= TOL_GRAD, errs


@pytest.mark.parametrize("B,Hq,Hkv,N,d,window,alibi", [
    (1, 2, 2, 300, 128, 0, False),
    (1, 2, 1, 513, 64, 63, False),
    (2, 4, 2, 640, 128, 64, True),
    (1, 2, 2, 700, 64, 127, False),
    (1, 4, 1, 1000, 128, 191, False),
    (1, 2, 2, 1024, 128, 1023, True),     # w = N - 1: the plain causal mask
    (1, 3, 3, 450, 64, 256, True),
])
def test_bwd_window(B, Hq, Hkv, N, d, window, alibi):
    w = I.small_case("bf16", causal=True, B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, alibi=alibi,
                     window=window)
    x = I.make_inputs(w, seed=7 + window)
    check_bwd(x, G.backward(x))


def test_bwd_window_varlen():
    w = I.small_case("bf16", causal=True, Hq=4, Hkv=2, d=128, seqlens=(5, 300, 1, 700, 129),
                     window=150)
    x = I.make_inputs(w, seed=9)
    check_bwd(x, G.backward(x))


def test_window_wider_than_sequence_equals_causal():
    """w >= N - 1 masks nothing beyond causality: results equal the unbanded
    causal run bit for bit (both take the same kernel path)."""
    base = I.small_case("bf16", causal=True, B=1, Hq=2, Hkv=2, N=400, d=128)
    x = I.make_inputs(base, seed=4)
    r0 = G.backward(x)
    for wnd in (399, 400, 10 ** 6):
        xw = I.make_inputs(I.small_case("bf16", causal=True, B=1, Hq=2, Hkv=2, N=400, d=128,
                                        window=wnd), seed=4)
        r1 = G.backward(xw)
        for a, b in zip(r0[:2] + r0[3:], r1[:2] + r1[3:]):   # dQ order is not fixed
            np.testing.assert_array_equal(a, b)


def _sub_inputs(x, a, b):
    """Tokens [a, b) of a one-sequence workload as a problem of their own."""
    w = x.workload
    sub = I.with_seqlens(w, [b - a])
    return I.Inputs(sub, x.seed, np.array([b - a]), np.array([0, b - a], dtype=np.int32),
                    x.q[a:b], x.k[a:b], x.v[a:b], x.do[a:b], x.alibi_slopes, x.scale)


@pytest.mark.slow
def test_full_size_window_workload_sampled():
    """The sliding-window workload at full size (one sequence of 32768 tokens,
    w = 4095, GQA 32/8), run exactly as the benchmark runs it.

    O, LSE and dQ of sampled rows come from the oracle's row forms.  For dK and
    dV the band gives a shortcut that holds at any size: key j meets only
    queries j .. j + w, and those see only keys from j - w on, so the
    gradient of key j is the same in any sub-sequence [a, b) with
    a <= j - w and b > j + w (positions enter only as differences).  Key rows
    near the start are checked on the prefix [0, 2w + 2), rows near the end on
    the suffix [L - 2w - 2, L).
    """
    w = I.workload("swa_32k")
    x = I.make_inputs(w, seed=0)
    O, lse, dq, dk, dv = G.backward(x, guard=False)
    for t_ in (O, lse, dq, dk, dv):
        assert np.isfinite(t_).all()
    rng = np.random.Generator(np.random.PCG64(77))
    L, W = w.N, w.window
    toks = [0, 1, 127, 128, W - 1, W, W + 1, W + 128, L // 2, L - 129, L - 1]
    toks += [int(t) for t in rng.integers(0, L, size=13)]
    qrows = [(t, int(rng.integers(0, w.Hq))) for t in toks]
    O_r, lse_r = A.forward_rows(x.q, x.k, x.v, x.scale, True, qrows, window=W)
    dq_r = A.backward_query_rows(x.q, x.k, x.v, x.do, x.scale, True, qrows, window=W)
    e_o = np.abs(np.array([O[t, h] for t, h in qrows]) - O_r).max()
    e_l = np.abs(np.array([lse[h, t] for t, h in qrows]) - lse_r).max()
    e_dq = np.abs(np.array([dq[t, h] for t, h in qrows]) - dq_r).max() / np.abs(dq_r).max()
    span = 2 * W + 2
    dks, dvs, dk_rs, dv_rs = [], [], [], []
    for a, offs in ((0, (0, 1, 127, 128, W - 64, W)), (L - span, (W + 1, W + 64, span - 129,
                                                                  span - 1))):
        xs = _sub_inputs(x, a, a + span)
        g = int(rng.integers(0, w.Hkv))
        krows = [(o, g) for o in offs]
        dk_r, dv_r = A.backward_key_rows(xs.q, xs.k, xs.v, xs.do, xs.scale, True, krows,
                                         window=W)
        dks += [dk[a + o, g] for o, _ in krows]
        dvs += [dv[a + o, g] for o, _ in krows]
        dk_rs.append(dk_r)
        dv_rs.append(dv_r)
    dk_r, dv_r = np.concatenate(dk_rs), np.concatenate(dv_rs)
    e_dk = np.abs(np.array(dks) - dk_r).max() / np.abs(dk_r).max()
    e_dv = np.abs(np.array(dvs) - dv_r).max() / np.abs(dv_r).max()
    errs = {"O": e_o, "LSE": e_l, "dQ": e_dq, "dK": e_dk, "dV": e_dv}
    print("swa_32k", {k_: float(v_) for k_, v_ in errs.items()})
    assert e_o <= TOL_O and e_l <= TOL_LSE, errs
    assert e_dq <= TOL_GRAD and e_dk <= TOL_GRAD and e_dv <= TOL_GRAD, errs
