"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each mutant replaces one oracle function with a plausible wrong version (a
dropped term, a wrong sign or index, a missing scale, a transposed operand)
and the test asserts that at least one pin of ``test_oracle`` fails under it.
The mistakes are planted in the oracle on the CPU, never in the CUDA path.
"""
import numpy as np
import pytest

from oracle import attention_fp64 as A
import tests.test_oracle as P

_orig_scores = A.head_scores
_orig_backward = A.head_backward
_orig_softmax = A._softmax_rows


def scores_alibi_sign(q, k, scale, causal, slope=None, window=None):
    return _orig_scores(q, k, scale, causal, None if slope is None else -slope, window)


def scores_causal_off_by_one(q, k, scale, causal, slope=None, window=None):
    S = _orig_scores(q, k, scale, False, slope)
    if causal:
        L = S.shape[0]
        vis = np.arange(S.shape[1])[None, :] < np.arange(L)[:, None]
        vis[0, 0] = True
        S = np.where(vis, S, -np.inf)
    return S


def scores_scale_twice(q, k, scale, causal, slope=None, window=None):
    return _orig_scores(q, k, scale * scale, causal, slope, window) if scale != 1.0 else \
        _orig_scores(q, k, 0.5, causal, slope, window)


def scores_bias_scaled(q, k, scale, causal, slope=None, window=None):
    return _orig_scores(q, k, scale, causal, None if slope is None else slope * scale, window)


def softmax_log2(S):
    Pm, lse = _orig_softmax(S)
    return Pm, lse / np.log(2.0)


def _backward_mutant(kind):
    def f(q, k, v, do, scale, causal, slope=None, window=None):
        q, k, v, do = (np.asarray(x, np.float64) for x in (q, k, v, do))
        O, lse, Pm = A.head_forward(q, k, v, scale, causal, slope, window)
        dP = do @ v.T
        D = (Pm * dP).sum(1)
        if kind == "D_dropped":
            D = np.zeros_like(D)
        if kind == "D_rowsum_dP":
            D = dP.sum(1)
        dS = Pm * (dP - D[:, None])
        dV = Pm.T @ do
        if kind == "dV_untransposed":
            dV = Pm @ do
        dQ = scale * (dS @ k)
        if kind == "dQ_no_scale":
            dQ = dS @ k
        dK = scale * (dS.T @ q)
        if kind == "dK_untransposed":
            dK = scale * (dS @ q)
        if kind == "dK_sign":
            dK = -dK
        return dQ, dK, dV, O, lse, D
    return f


def scores_window_off_by_one(q, k, scale, causal, slope=None, window=None):
    return _orig_scores(q, k, scale, causal, slope, None if window is None else window - 1)


MUTANTS = {
    "window_off_by_one": ("head_scores", scores_window_off_by_one),
    "alibi_sign": ("head_scores", scores_alibi_sign),
    "causal_off_by_one": ("head_scores", scores_causal_off_by_one),
    "scale_twice": ("head_scores", scores_scale_twice),
    "bias_scaled": ("head_scores", scores_bias_scaled),
    "lse_log2": ("_softmax_rows", softmax_log2),
    "D_dropped": ("head_backward", _backward_mutant("D_dropped")),
    "D_rowsum_dP": ("head_backward", _backward_mutant("D_rowsum_dP")),
    "dV_untransposed": ("head_backward", _backward_mutant("dV_untransposed")),
    "dQ_no_scale": ("head_backward", _backward_mutant("dQ_no_scale")),
    "dK_untransposed": ("head_backward", _backward_mutant("dK_untransposed")),
    "dK_sign": ("head_backward", _backward_mutant("dK_sign")),
}

PINS = [
    lambda: P.test_probability_rows_sum_to_one(True, 0.37),
    lambda: P.test_zero_query_gives_mean_of_visible_values(True),
    P.test_causal_first_row_is_first_value,
    P.test_closed_form_two_keys,
    P.test_closed_form_scale_factor,
    lambda: P.test_online_recurrence_equals_two_pass(True, 0.5, 3, 7),
    lambda: P.test_gradients_match_finite_differences(True, True, 2, 2, [5]),
    lambda: P.test_gradients_match_finite_differences(True, False, 2, 1, [3, 5]),
    P.test_alibi_sign_and_index_by_row_shift,
    P.test_alibi_huge_slope_picks_diagonal,
    lambda: P.test_matches_torch_float64_sdpa_and_autograd(True, True, 4, 2),
    lambda: P.test_window_zero_query_gives_band_mean(5),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(A, attr, fn)
    caught = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError):   # a failed check or a shape error
            caught.append(pin)
    assert caught, f"no pin catches mutant {name}"


def test_gqa_mapping_mistake_is_caught(monkeypatch):
    """kv head h % Hkv instead of h // (Hq/Hkv): the GQA-vs-repeated-MHA pin fails."""
    orig_fwd = A.attention_forward

    def attention_backward_interleaved(q, k, v, do, scale, causal, cu_seqlens=None,
                                       alibi_slopes=None, heads=None, seqs=None):
        T, Hq, d = q.shape
        Hkv = k.shape[1]
        dQ = np.zeros(q.shape); dK = np.zeros(k.shape); dV = np.zeros(v.shape)
        O = np.zeros(q.shape); LSE = np.zeros((Hq, T)); D = np.zeros((Hq, T))
        for h in range(Hq):
            g = h % Hkv
            sl = None if alibi_slopes is None else float(alibi_slopes[h])
            dq, dk, dv, o, lse, dd = A.head_backward(q[:, h], k[:, g], v[:, g], do[:, h],
                                                     scale, causal, sl)
            dQ[:, h] = dq; dK[:, g] += dk; dV[:, g] += dv; O[:, h] = o; LSE[h] = lse; D[h] = dd
        return dQ, dK, dV, O, LSE, D

    monkeypatch.setattr(A, "attention_backward", attention_backward_interleaved)
    with pytest.raises(AssertionError):
        P.test_gqa_equals_mha_with_repeated_kv()
    assert orig_fwd is A.attention_forward


# ------------------------------------------------------------------- decode

_orig_decode = A.decode_forward


def _decode_mutant(kind):
    """decode_forward with one plausible mistake, written out in full."""
    def f(q, k_cache, v_cache, cache_seqlens, scale, q_len=1, alibi_slopes=None, window=None):
        B, S_max, Hkv, d = k_cache.shape
        Hq = q.shape[1]
        group = Hq // Hkv
        O = np.empty((B * q_len, Hq, v_cache.shape[3]))
        LSE = np.empty((Hq, B * q_len))
        for b in range(B):
            L = S_max if cache_seqlens is None else int(cache_seqlens[b])
            off = L - q_len + (1 if kind == "position_plus_one" else 0)
            pos = (off + np.arange(q_len))[:, None]
            j = np.arange(L)[None, :]
            vis = j <= pos
            if window is not None:
                vis &= j > pos - window if kind == "window_strict" else j >= pos - window
            rows = slice(b * q_len, (b + 1) * q_len)
            for h in range(Hq):
                g = h % Hkv if kind == "kv_head_interleaved" else h // group
                S = scale * (np.asarray(q[rows, h], np.float64) @ np.asarray(k_cache[b, :L, g], np.float64).T)
                if alibi_slopes is not None:
                    sgn = -1.0 if kind == "alibi_sign" else 1.0
                    S = S - sgn * float(alibi_slopes[h]) * (pos - j)
                P_, lse = A._softmax_rows(np.where(vis, S, -np.inf))
                O[rows, h] = P_ @ np.asarray(v_cache[b, :L, g], np.float64)
                LSE[h, rows] = lse
        return O, LSE
    return f


DECODE_PINS = [
    lambda: P.test_decode_is_the_last_rows_of_the_causal_forward(3, False, None, 2, 2),
    lambda: P.test_decode_is_the_last_rows_of_the_causal_forward(1, True, None, 8, 2),
    lambda: P.test_decode_is_the_last_rows_of_the_causal_forward(4, True, 5, 4, 1),
    lambda: P.test_decode_equal_keys_give_the_visible_mean(3),
    P.test_decode_matches_torch_float64_sdpa,
]


@pytest.mark.parametrize("kind", ["position_plus_one", "window_strict", "kv_head_interleaved",
                                  "alibi_sign"])
def test_planted_decode_mistake_is_caught(kind, monkeypatch):
    monkeypatch.setattr(A, "decode_forward", _decode_mutant(kind))
    caught = 0
    for pin in DECODE_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught += 1
    assert caught, f"no pin catches decode mutant {kind}"


def test_decode_mutant_harness_passes_unmutated(monkeypatch):
    """The written-out copy without a mistake passes every decode pin, so the
    failures above come from the planted mistakes."""
    monkeypatch.setattr(A, "decode_forward", _decode_mutant("none"))
    for pin in DECODE_PINS:
        pin()
