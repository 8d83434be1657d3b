"""Pins of the fp64 oracle to facts outside itself (CPU only).

Each test checks the oracle against something it does not compute itself: a
closed form, an invariant of softmax attention, a second algorithm the pages
give (the online recurrence), finite differences, or an independent library
routine (PyTorch's float64 CPU attention and autograd).  Together they are
chosen so that a dropped term, a wrong sign or index, a missing scale or a
transposed operand in the oracle fails at least one of them.
"""
import math

import numpy as np
import pytest

from oracle import attention_fp64 as A
from exact_io_aware_36_gb300 import inputs as I


def rnd(seed, *shape, scale=1.0):
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape) * scale


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("slope", [None, 0.37])
def test_probability_rows_sum_to_one(causal, slope):
    L, d = 37, 16
    q, k, v = rnd(1, L, d), rnd(2, L, d), rnd(3, L, d)
    O, lse, P = A.head_forward(q, k, v, 0.25, causal, slope)
    assert np.all(P >= 0)
    assert np.max(np.abs(P.sum(1) - 1)) <= 1e-12
    S = A.head_scores(q, k, 0.25, causal, slope)
    assert np.max(np.abs(np.exp(S - lse[:, None]).sum(1) - 1)) <= 1e-12
    if causal:
        assert np.all(P[np.triu_indices(L, 1)] == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_mean_of_visible_values(causal):
    """Q = 0 makes every visible score equal: O_i is the mean of the visible
    V rows and LSE_i = ln(#visible keys)."""
    L, d = 29, 8
    v = rnd(4, L, d)
    O, lse, _ = A.head_forward(np.zeros((L, d)), rnd(5, L, d), v, 0.3, causal)
    if causal:
        n = np.arange(1, L + 1)
        ref = np.cumsum(v, axis=0) / n[:, None]
    else:
        n = np.full(L, L)
        ref = np.broadcast_to(v.mean(0), (L, d))
    np.testing.assert_allclose(O, ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, np.log(n), rtol=0, atol=1e-13)


def test_causal_first_row_is_first_value():
    L, d = 11, 8
    q, k, v = rnd(6, L, d), rnd(7, L, d), rnd(8, L, d)
    O, lse, _ = A.head_forward(q, k, v, 0.5, True)
    np.testing.assert_allclose(O[0], v[0], rtol=0, atol=1e-15)
    assert abs(lse[0] - 0.5 * float(q[0] @ k[0])) <= 1e-14


def test_dominant_key_returns_its_value():
    """k_j = alpha * q_i / |q_i|^2 gives query i a score alpha/.. far above the
    others, so O_i -> V_j (gap > 60 nats => error < 1e-25 relative)."""
    L, d = 16, 8
    q, k, v = rnd(9, L, d), rnd(10, L, d, scale=0.01), rnd(11, L, d)
    i, j = 12, 5
    k[j] = 100.0 * q[i] / (q[i] @ q[i])
    O, _, _ = A.head_forward(q, k, v, 1.0, True)
    np.testing.assert_allclose(O[i], v[j], rtol=0, atol=1e-12)


def test_closed_form_two_keys():
    """One query, two keys, scale 1: P = (p, 1-p) with p = e^a / (e^a + e^b);
    O = p v0 + (1-p) v1; LSE = ln(e^a + e^b); dq = p(1-p) (dO.(v0-v1)) (k0-k1);
    dk0 = -dk1 = p(1-p) (dO.(v0-v1)) q; dv0 = p dO, dv1 = (1-p) dO."""
    q = np.array([[0.3, -1.2, 0.5]])
    k = np.array([[1.0, 0.2, -0.4], [-0.7, 0.1, 0.9]])
    v = np.array([[1.0, 2.0], [3.0, -4.0]])
    do = np.array([[0.25, -1.5]])
    a, b = float(q[0] @ k[0]), float(q[0] @ k[1])
    p = math.exp(a) / (math.exp(a) + math.exp(b))
    dq, dk, dv, O, lse, D = A.head_backward(q, k, v, do, 1.0, False)
    np.testing.assert_allclose(O[0], p * v[0] + (1 - p) * v[1], rtol=1e-15, atol=1e-15)
    assert abs(lse[0] - math.log(math.exp(a) + math.exp(b))) < 1e-15
    g = p * (1 - p) * float(do[0] @ (v[0] - v[1]))
    np.testing.assert_allclose(dq[0], g * (k[0] - k[1]), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dk[0], g * q[0], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dk[1], -g * q[0], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dv[0], p * do[0], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(dv[1], (1 - p) * do[0], rtol=1e-14, atol=1e-15)


def test_closed_form_scale_factor():
    """The same two-key case with scale s: scores scale by s and dq picks up
    one more factor s (chain rule), dv none."""
    q = np.array([[0.3, -1.2, 0.5]])
    k = np.array([[1.0, 0.2, -0.4], [-0.7, 0.1, 0.9]])
    v = np.array([[1.0, 2.0], [3.0, -4.0]])
    do = np.array([[0.25, -1.5]])
    s = 0.125
    a, b = s * float(q[0] @ k[0]), s * float(q[0] @ k[1])
    p = 1.0 / (1.0 + math.exp(b - a))
    dq, dk, dv, O, lse, D = A.head_backward(q, k, v, do, s, False)
    g = p * (1 - p) * float(do[0] @ (v[0] - v[1]))
    np.testing.assert_allclose(dq[0], s * g * (k[0] - k[1]), rtol=1e-13, atol=1e-16)
    np.testing.assert_allclose(dv[0], p * do[0], rtol=1e-14)
    assert abs(lse[0] - (a + math.log1p(math.exp(b - a)))) < 1e-15


def test_D_identity():
    """D_i = rowsum(P o dP) equals dO_i . O_i."""
    L, d = 23, 8
    q, k, v, do = rnd(12, L, d), rnd(13, L, d), rnd(14, L, d), rnd(15, L, d)
    _, _, _, O, _, D = A.head_backward(q, k, v, do, 0.35, True, 0.2)
    np.testing.assert_allclose(D, (do * O).sum(1), rtol=0, atol=1e-13)


# ------------------------------------------------ the pages' recurrences

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("slope", [None, 0.5])
@pytest.mark.parametrize("bq,bk", [(1, 1), (3, 7), (7, 3), (40, 40), (5, 40)])
def test_online_recurrence_equals_two_pass(causal, slope, bq, bk):
    """Key design 2's merge, run in the FA1 loop order with several block
    sizes, equals the materialised two-pass softmax (FA1 Theorem 1)."""
    L, d = 40, 8
    q, k, v = rnd(16, L, d, scale=2.0), rnd(17, L, d), rnd(18, L, d)
    O_ref, lse_ref, _ = A.head_forward(q, k, v, 0.4, causal, slope)
    O, lse = A.online_softmax_forward(q, k, v, 0.4, causal, slope, bq, bk)
    np.testing.assert_allclose(O, O_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("bk", [1, 3, 7, 40])
def test_normalised_recurrence_equals_two_pass(bk):
    L, d = 40, 8
    q, k, v = rnd(19, L, d, scale=2.0), rnd(20, L, d), rnd(21, L, d)
    O_ref, lse_ref, _ = A.head_forward(q, k, v, 0.4, True)
    O, lse = A.online_softmax_forward_normalised(q, k, v, 0.4, True, None, bk)
    np.testing.assert_allclose(O, O_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


# ------------------------------------------------------- finite differences

def _fd_case(causal, alibi, Hq, Hkv, seqlens, d=4, seed=22):
    T = sum(seqlens)
    q, k, v, do = rnd(seed, T, Hq, d), rnd(seed + 1, T, Hkv, d), rnd(seed + 2, T, Hkv, d), rnd(seed + 3, T, Hq, d)
    cu = np.concatenate([[0], np.cumsum(seqlens)])
    slopes = I.alibi_slopes(Hq).astype(np.float64) if alibi else None
    return q, k, v, do, cu, slopes


@pytest.mark.parametrize("causal,alibi,Hq,Hkv,seqlens", [
    (False, False, 1, 1, [6]),
    (True, False, 1, 1, [8]),
    (True, True, 2, 2, [5]),
    (True, False, 2, 1, [3, 5]),
    (False, True, 4, 2, [4, 2]),
])
def test_gradients_match_finite_differences(causal, alibi, Hq, Hkv, seqlens):
    """fp64 central differences of f = <dO, O> w.r.t. q, k, v agree with the
    oracle's gradients to 1e-6 relative (pins dQ, dK, dV and the scale)."""
    q, k, v, do, cu, slopes = _fd_case(causal, alibi, Hq, Hkv, seqlens)
    scale = 0.7

    def f(q_, k_, v_):
        O, _ = A.attention_forward(q_, k_, v_, scale, causal, cu, slopes)
        return float((do * O).sum())

    dq, dk, dv, *_ = A.attention_backward(q, k, v, do, scale, causal, cu, slopes)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            num[idx] = (f(*args_p) - f(*args_m)) / (2 * h)
        err = np.max(np.abs(num - g)) / max(np.max(np.abs(g)), 1e-30)
        assert err <= 1e-6, (name, err)


# ---------------------------------------------------------- bias and heads

def test_alibi_sign_and_index_by_row_shift():
    """bias -s(i-j) and bias +s*j differ by a per-row constant: same O, LSE
    shifted by -s*i.  The +s*j bias is realised without the oracle's bias
    code, as an extra feature column (q' = [q, 1], k' = [k, s*j/scale])."""
    L, d, s, scale = 19, 8, 0.3, 0.5
    q, k, v = rnd(30, L, d), rnd(31, L, d), rnd(32, L, d)
    j = np.arange(L, dtype=np.float64)
    q2 = np.concatenate([q, np.ones((L, 1))], axis=1)
    k2 = np.concatenate([k, (s * j / scale)[:, None]], axis=1)
    for causal in (False, True):
        O1, lse1, _ = A.head_forward(q, k, v, scale, causal, s)
        O2, lse2, _ = A.head_forward(q2, k2, v, scale, causal, None)
        np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse1, lse2 - s * j, rtol=0, atol=1e-12)


def test_alibi_huge_slope_picks_diagonal():
    L, d = 13, 8
    q, k, v = rnd(33, L, d), rnd(34, L, d), rnd(35, L, d)
    O, _, _ = A.head_forward(q, k, v, 0.1, True, 1e4)
    np.testing.assert_allclose(O, v, rtol=0, atol=1e-12)


def test_alibi_slopes_definition():
    s = I.alibi_slopes(32)
    assert s[0] == np.float32(2 ** -0.25) and s[31] == np.float32(2 ** -8)
    s8 = I.alibi_slopes(8)
    np.testing.assert_array_equal(s8, np.float32(2.0) ** -np.arange(1, 9, dtype=np.float32))


def test_gqa_equals_mha_with_repeated_kv():
    T, Hq, Hkv, d = 21, 6, 2, 8
    q, k, v, do = rnd(36, T, Hq, d), rnd(37, T, Hkv, d), rnd(38, T, Hkv, d), rnd(39, T, Hq, d)
    slopes = I.alibi_slopes(Hq).astype(np.float64)
    dq, dk, dv, O, lse, _ = A.attention_backward(q, k, v, do, 0.3, True, None, slopes)
    kr, vr = np.repeat(k, Hq // Hkv, axis=1), np.repeat(v, Hq // Hkv, axis=1)
    dq2, dk2, dv2, O2, lse2, _ = A.attention_backward(q, kr, vr, do, 0.3, True, None, slopes)
    np.testing.assert_allclose(O, O2, atol=1e-14)
    np.testing.assert_allclose(lse, lse2, atol=1e-14)
    np.testing.assert_allclose(dq, dq2, atol=1e-14)
    np.testing.assert_allclose(dk, dk2.reshape(T, Hkv, Hq // Hkv, d).sum(2), atol=1e-13)
    np.testing.assert_allclose(dv, dv2.reshape(T, Hkv, Hq // Hkv, d).sum(2), atol=1e-13)


def test_varlen_equals_independent_sequences():
    lens = [5, 1, 17, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, d = cu[-1], 2, 8
    q, k, v, do = rnd(40, T, H, d), rnd(41, T, H, d), rnd(42, T, H, d), rnd(43, T, H, d)
    dq, dk, dv, O, lse, _ = A.attention_backward(q, k, v, do, 0.3, True, cu)
    for b in range(len(lens)):
        s, e = cu[b], cu[b + 1]
        r = A.attention_backward(q[s:e], k[s:e], v[s:e], do[s:e], 0.3, True)
        np.testing.assert_allclose(O[s:e], r[3], atol=1e-14)
        np.testing.assert_allclose(lse[:, s:e], r[4], atol=1e-14)
        np.testing.assert_allclose(dq[s:e], r[0], atol=1e-14)
        np.testing.assert_allclose(dk[s:e], r[1], atol=1e-14)
        np.testing.assert_allclose(dv[s:e], r[2], atol=1e-14)


def test_noncausal_key_permutation_invariance():
    L, d = 17, 8
    q, k, v = rnd(44, L, d), rnd(45, L, d), rnd(46, L, d)
    perm = np.random.Generator(np.random.PCG64(47)).permutation(L)
    O1, lse1, _ = A.head_forward(q, k, v, 0.3, False)
    O2, lse2, _ = A.head_forward(q, k[perm], v[perm], 0.3, False)
    np.testing.assert_allclose(O1, O2, atol=1e-13)
    np.testing.assert_allclose(lse1, lse2, atol=1e-13)


# ------------------------------------------------- independent library check

@pytest.mark.parametrize("causal,alibi,Hq,Hkv", [
    (False, False, 2, 2), (True, False, 4, 4), (True, True, 4, 2), (True, True, 8, 1)])
def test_matches_torch_float64_sdpa_and_autograd(causal, alibi, Hq, Hkv):
    torch = pytest.importorskip("torch")
    L, d, scale = 33, 16, 0.2
    q, k, v, do = rnd(50, L, Hq, d), rnd(51, L, Hkv, d), rnd(52, L, Hkv, d), rnd(53, L, Hq, d)
    slopes = I.alibi_slopes(Hq).astype(np.float64) if alibi else None
    dq, dk, dv, O, lse, _ = A.attention_backward(q, k, v, do, scale, causal, None, slopes)

    tq = torch.tensor(q.transpose(1, 0, 2)[None], requires_grad=True)
    tk = torch.tensor(np.repeat(k, Hq // Hkv, 1).transpose(1, 0, 2)[None], requires_grad=True)
    tv = torch.tensor(np.repeat(v, Hq // Hkv, 1).transpose(1, 0, 2)[None], requires_grad=True)
    i = torch.arange(L, dtype=torch.float64)[:, None]
    j = torch.arange(L, dtype=torch.float64)[None, :]
    mask = torch.zeros(Hq, L, L, dtype=torch.float64)
    if alibi:
        mask = mask + torch.tensor(slopes)[:, None, None] * (j - i)[None]
    if causal:
        mask = mask.masked_fill((j > i)[None], float("-inf"))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask[None], scale=scale)
    out.backward(torch.tensor(do.transpose(1, 0, 2)[None]))
    np.testing.assert_allclose(O, out[0].detach().numpy().transpose(1, 0, 2), atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad[0].numpy().transpose(1, 0, 2), atol=1e-11)
    g = Hq // Hkv
    tkg = tk.grad[0].numpy().transpose(1, 0, 2).reshape(L, Hkv, g, d).sum(2)
    tvg = tv.grad[0].numpy().transpose(1, 0, 2).reshape(L, Hkv, g, d).sum(2)
    np.testing.assert_allclose(dk, tkg, atol=1e-11)
    np.testing.assert_allclose(dv, tvg, atol=1e-11)
    scores = torch.einsum("hid,hjd->hij", tq[0].detach(), tk[0].detach()) * scale + mask
    np.testing.assert_allclose(lse, torch.logsumexp(scores, -1).numpy(), atol=1e-12)


# ------------------------------------------------------- sampled-row forms

def test_sampled_rows_equal_full_oracle():
    lens = [70, 33, 101]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, Hq, Hkv, d = cu[-1], 4, 2, 16
    q, k, v, do = rnd(60, T, Hq, d), rnd(61, T, Hkv, d), rnd(62, T, Hkv, d), rnd(63, T, Hq, d)
    slopes = I.alibi_slopes(Hq).astype(np.float64)
    dq, dk, dv, O, lse, _ = A.attention_backward(q, k, v, do, 0.25, True, cu, slopes)
    rows = [(0, 0), (69, 3), (70, 1), (102, 2), (T - 1, 0), (150, 3)]
    O_r, lse_r = A.forward_rows(q, k, v, 0.25, True, rows, cu, slopes)
    dq_r = A.backward_query_rows(q, k, v, do, 0.25, True, rows, cu, slopes)
    for n, (t, h) in enumerate(rows):
        np.testing.assert_allclose(O_r[n], O[t, h], atol=1e-13)
        assert abs(lse_r[n] - lse[h, t]) < 1e-13
        np.testing.assert_allclose(dq_r[n], dq[t, h], atol=1e-13)
    krows = [(0, 0), (69, 1), (70, 0), (T - 1, 1), (120, 1)]
    dk_r, dv_r = A.backward_key_rows(q, k, v, do, 0.25, True, krows, cu, slopes)
    for n, (t, g) in enumerate(krows):
        np.testing.assert_allclose(dk_r[n], dk[t, g], atol=1e-12)
        np.testing.assert_allclose(dv_r[n], dv[t, g], atol=1e-12)


# ----------------------------------------------------- whole-head row blocks

@pytest.mark.parametrize("causal,slope,window", [(False, None, None), (True, None, None),
                                                 (True, 0.37, None), (True, None, 5),
                                                 (False, 0.2, None)])
@pytest.mark.parametrize("chunk", [1, 3, 7, 40])
def test_chunked_head_forms_equal_the_whole_matrices(causal, slope, window, chunk):
    """The row-block forms used for whole heads of long sequences give the
    whole-matrix oracle's O, LSE, D and gradients (to 1e-12): a block that
    is dropped, mis-offset (the causal mask, the band and the ALiBi index
    use the block's first row) or overwritten instead of summed fails."""
    L, d = 29, 6
    q, k, v, do = rnd(90, L, d), rnd(91, L, d), rnd(92, L, d), rnd(93, L, d)
    O, lse, _ = A.head_forward(q, k, v, 0.45, causal, slope, window)
    Oc, lsec = A.head_forward_chunked(q, k, v, 0.45, causal, slope, window, chunk=chunk)
    np.testing.assert_allclose(Oc, O, atol=1e-12)
    np.testing.assert_allclose(lsec, lse, atol=1e-12)
    ref = A.head_backward(q, k, v, do, 0.45, causal, slope, window)
    got = A.head_backward_chunked(q, k, v, do, 0.45, causal, slope, window, chunk=chunk)
    for name, r, g in zip(("dQ", "dK", "dV", "O", "LSE", "D"), ref, got):
        np.testing.assert_allclose(g, r, atol=1e-12, err_msg=name)


def test_chunked_head_backward_matches_finite_differences():
    """Independently of the whole-matrix form: fp64 central differences of
    <dO, O> (O from the chunked forward) agree with the chunked gradients."""
    L, d, scale, slope = 7, 3, 0.8, 0.3
    q, k, v, do = rnd(94, L, d), rnd(95, L, d), rnd(96, L, d), rnd(97, L, d)
    dq, dk, dv, *_ = A.head_backward_chunked(q, k, v, do, scale, True, slope, chunk=3)

    def f(q_, k_, v_):
        return float((do * A.head_forward_chunked(q_, k_, v_, scale, True, slope, chunk=2)[0]).sum())

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            ap = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            am = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            num[idx] = (f(*ap) - f(*am)) / (2 * h)
        assert np.max(np.abs(num - g)) / np.max(np.abs(g)) <= 1e-6, name


# ------------------------------------------------------------ sliding window

@pytest.mark.parametrize("w", [0, 1, 5, 28])
def test_window_zero_query_gives_band_mean(w):
    """Q = 0: row i averages V over the band [max(0, i - w), i] and LSE_i is
    ln(band length)."""
    L, d = 29, 8
    v = rnd(70, L, d)
    O, lse, _ = A.head_forward(np.zeros((L, d)), rnd(71, L, d), v, 0.3, True, None, w)
    for i in range(L):
        lo = max(0, i - w)
        np.testing.assert_allclose(O[i], v[lo:i + 1].mean(0), rtol=0, atol=1e-13)
        assert abs(lse[i] - np.log(i - lo + 1)) < 1e-13


def test_window_zero_is_the_diagonal_and_wide_window_is_causal():
    L, d = 21, 8
    q, k, v = rnd(72, L, d), rnd(73, L, d), rnd(74, L, d)
    O, lse, _ = A.head_forward(q, k, v, 0.4, True, None, 0)
    np.testing.assert_allclose(O, v, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, 0.4 * (q * k).sum(1), rtol=0, atol=1e-14)
    O1, l1, _ = A.head_forward(q, k, v, 0.4, True, 0.2, L - 1)
    O2, l2, _ = A.head_forward(q, k, v, 0.4, True, 0.2)
    np.testing.assert_allclose(O1, O2, atol=0)
    np.testing.assert_allclose(l1, l2, atol=0)
    with pytest.raises(ValueError):
        A.head_forward(q, k, v, 0.4, False, None, 3)


def test_window_ignores_keys_outside_the_band():
    """Rows whose band excludes key j are unchanged when k_j and v_j change."""
    L, d, w, j = 40, 8, 6, 10
    q, k, v = rnd(75, L, d), rnd(76, L, d), rnd(77, L, d)
    O1, l1, _ = A.head_forward(q, k, v, 0.5, True, None, w)
    k2, v2 = k.copy(), v.copy()
    k2[j] += 3.0
    v2[j] -= 2.0
    O2, l2, _ = A.head_forward(q, k2, v2, 0.5, True, None, w)
    outside = [i for i in range(L) if not (i - w <= j <= i)]
    inside = [i for i in range(L) if i - w <= j <= i]
    np.testing.assert_allclose(O1[outside], O2[outside], atol=0)
    assert np.abs(O1[inside] - O2[inside]).max() > 1e-3


@pytest.mark.parametrize("w,bq,bk", [(3, 1, 1), (7, 3, 5), (16, 40, 7)])
def test_window_online_recurrence_equals_two_pass(w, bq, bk):
    L, d = 40, 8
    q, k, v = rnd(78, L, d, scale=2.0), rnd(79, L, d), rnd(80, L, d)
    O_ref, lse_ref, _ = A.head_forward(q, k, v, 0.4, True, 0.3, w)
    O, lse = A.online_softmax_forward(q, k, v, 0.4, True, 0.3, bq, bk, window=w)
    np.testing.assert_allclose(O, O_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_window_gradients_match_finite_differences():
    q, k, v, do, cu, slopes = _fd_case(True, True, 2, 1, [7, 4])
    scale, w = 0.6, 2

    def f(q_, k_, v_):
        O, _ = A.attention_forward(q_, k_, v_, scale, True, cu, slopes, window=w)
        return float((do * O).sum())

    dq, dk, dv, *_ = A.attention_backward(q, k, v, do, scale, True, cu, slopes, window=w)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            num[idx] = (f(*args_p) - f(*args_m)) / (2 * h)
        assert np.max(np.abs(num - g)) / np.max(np.abs(g)) <= 1e-6, name


def test_window_matches_torch_float64_sdpa():
    torch = pytest.importorskip("torch")
    L, H, d, w, scale = 33, 2, 16, 5, 0.25
    q, k, v, do = rnd(81, L, H, d), rnd(82, L, H, d), rnd(83, L, H, d), rnd(84, L, H, d)
    dq, dk, dv, O, lse, _ = A.attention_backward(q, k, v, do, scale, True, window=w)
    tq, tk, tv = (torch.tensor(x.transpose(1, 0, 2)[None], requires_grad=True) for x in (q, k, v))
    i = torch.arange(L)[:, None]
    j = torch.arange(L)[None, :]
    mask = torch.zeros(L, L, dtype=torch.float64).masked_fill((j > i) | (j < i - w), float("-inf"))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    out.backward(torch.tensor(do.transpose(1, 0, 2)[None]))
    np.testing.assert_allclose(O, out[0].detach().numpy().transpose(1, 0, 2), atol=1e-12)
    for a, t in ((dq, tq), (dk, tk), (dv, tv)):
        np.testing.assert_allclose(a, t.grad[0].numpy().transpose(1, 0, 2), atol=1e-11)


def test_window_sampled_rows_equal_full_oracle():
    lens = [70, 33, 101]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, Hq, Hkv, d, w = cu[-1], 4, 2, 16, 9
    q, k, v, do = rnd(85, T, Hq, d), rnd(86, T, Hkv, d), rnd(87, T, Hkv, d), rnd(88, T, Hq, d)
    slopes = I.alibi_slopes(Hq).astype(np.float64)
    dq, dk, dv, O, lse, _ = A.attention_backward(q, k, v, do, 0.25, True, cu, slopes, window=w)
    rows = [(0, 0), (69, 3), (70, 1), (102, 2), (T - 1, 0), (150, 3)]
    O_r, lse_r = A.forward_rows(q, k, v, 0.25, True, rows, cu, slopes, window=w)
    dq_r = A.backward_query_rows(q, k, v, do, 0.25, True, rows, cu, slopes, window=w)
    for n, (t, h) in enumerate(rows):
        np.testing.assert_allclose(O_r[n], O[t, h], atol=1e-13)
        assert abs(lse_r[n] - lse[h, t]) < 1e-13
        np.testing.assert_allclose(dq_r[n], dq[t, h], atol=1e-13)
    krows = [(0, 0), (69, 1), (70, 0), (T - 1, 1), (120, 1)]
    dk_r, dv_r = A.backward_key_rows(q, k, v, do, 0.25, True, krows, cu, slopes, window=w)
    for n, (t, g) in enumerate(krows):
        np.testing.assert_allclose(dk_r[n], dk[t, g], atol=1e-12)
        np.testing.assert_allclose(dv_r[n], dv[t, g], atol=1e-12)


# ------------------------------------------------------------------- decode

def _cache_case(seed, lens, S_max, Hq, Hkv, d, q_len):
    """Sequences of the given lengths laid out as a [B, S_max, Hkv, d] cache
    (slots past each length hold garbage), with the newest q_len tokens' queries."""
    B = len(lens)
    kc = rnd(seed, B, S_max, Hkv, d)
    vc = rnd(seed + 1, B, S_max, Hkv, d)
    qf = rnd(seed + 2, B, S_max, Hq, d)          # queries of every position
    q = np.concatenate([qf[b, L - q_len:L] for b, L in enumerate(lens)])
    return q, kc, vc, qf


@pytest.mark.parametrize("q_len,alibi,window,Hq,Hkv", [
    (1, False, None, 4, 2), (1, True, None, 8, 2), (3, False, None, 2, 2),
    (4, True, 5, 4, 1), (1, False, 0, 2, 1), (2, False, 40, 3, 3)])
def test_decode_is_the_last_rows_of_the_causal_forward(q_len, alibi, window, Hq, Hkv):
    """R10: decode equals the causal forward over each whole sequence, read at
    its newest q_len rows (the forward is pinned by the tests above)."""
    lens, S_max, d, scale = [37, 4, 60], 64, 8, 0.3
    q, kc, vc, qf = _cache_case(70, lens, S_max, Hq, Hkv, d, q_len)
    slopes = I.alibi_slopes(Hq).astype(np.float64) if alibi else None
    O, lse = A.decode_forward(q, kc, vc, np.array(lens), scale, q_len, slopes, window)
    for b, L in enumerate(lens):
        Of, lf = A.attention_forward(qf[b, :L], kc[b, :L], vc[b, :L], scale, True, None, slopes,
                                     window=window)
        np.testing.assert_allclose(O[b * q_len:(b + 1) * q_len], Of[L - q_len:], atol=1e-12)
        np.testing.assert_allclose(lse[:, b * q_len:(b + 1) * q_len], lf[:, L - q_len:], atol=1e-12)


@pytest.mark.parametrize("window", [None, 0, 3])
def test_decode_equal_keys_give_the_visible_mean(window):
    """With all keys zero every visible score is 0 (no bias): O is the mean of
    the visible values and LSE = log(count)."""
    lens, S_max, Hq, Hkv, d, q_len = [9, 2, 16], 16, 2, 1, 4, 2
    q, kc, vc, _ = _cache_case(80, lens, S_max, Hq, Hkv, d, q_len)
    kc[:] = 0.0
    O, lse = A.decode_forward(q, kc, vc, np.array(lens), 0.5, q_len, None, window)
    for b, L in enumerate(lens):
        for i in range(q_len):
            p = L - q_len + i
            lo = 0 if window is None else max(0, p - window)
            for h in range(Hq):
                np.testing.assert_allclose(O[b * q_len + i, h], vc[b, lo:p + 1, 0].mean(0), atol=1e-13)
                assert abs(lse[h, b * q_len + i] - math.log(p + 1 - lo)) < 1e-13


def test_decode_single_cached_token():
    """L = 1: the one key is the answer; LSE = scale q . k."""
    q, kc, vc, _ = _cache_case(90, [1, 1], 4, 2, 2, 8, 1)
    O, lse = A.decode_forward(q, kc, vc, np.array([1, 1]), 0.7, 1)
    for b in range(2):
        for h in range(2):
            np.testing.assert_allclose(O[b, h], vc[b, 0, h], atol=1e-14)
            assert abs(lse[h, b] - 0.7 * q[b, h] @ kc[b, 0, h]) < 1e-13


def test_decode_matches_torch_float64_sdpa():
    torch = pytest.importorskip("torch")
    lens, S_max, Hq, Hkv, d, q_len, scale = [50, 7], 64, 4, 2, 16, 3, 0.25
    q, kc, vc, _ = _cache_case(95, lens, S_max, Hq, Hkv, d, q_len)
    slopes = I.alibi_slopes(Hq).astype(np.float64)
    O, lse = A.decode_forward(q, kc, vc, np.array(lens), scale, q_len, slopes, 20)
    g = Hq // Hkv
    for b, L in enumerate(lens):
        tq = torch.tensor(q[b * q_len:(b + 1) * q_len].transpose(1, 0, 2)[None])
        tk = torch.tensor(np.repeat(kc[b, :L], g, 1).transpose(1, 0, 2)[None])
        tv = torch.tensor(np.repeat(vc[b, :L], g, 1).transpose(1, 0, 2)[None])
        i = torch.arange(L - q_len, L, dtype=torch.float64)[:, None]
        j = torch.arange(L, dtype=torch.float64)[None, :]
        mask = torch.tensor(slopes)[:, None, None] * (j - i)[None]
        mask = mask.masked_fill(((j > i) | (j < i - 20))[None], float("-inf"))
        out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask[None],
                                                               scale=scale)
        np.testing.assert_allclose(O[b * q_len:(b + 1) * q_len],
                                   out[0].numpy().transpose(1, 0, 2), atol=1e-12)
        scores = torch.einsum("hid,hjd->hij", tq[0], tk[0]) * scale + mask
        np.testing.assert_allclose(lse[:, b * q_len:(b + 1) * q_len],
                                   torch.logsumexp(scores, -1).numpy(), atol=1e-12)
