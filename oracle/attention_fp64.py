"""fp64 CPU oracle for exact scaled-dot-product attention, forward and backward.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import or run this module.  The
product (the CUDA library and its Python binding) never calls it, and it
shares no code with the product: it depends on NumPy alone.

Pages followed (cited by title and section):

* [FA1 note] "FlashAttention: Faster Attention Without Dropping a Single
  Interaction" (awesome.papernotes.org note on arXiv 2205.14135).
  - Key design 1: S = QK^T/sqrt(d), P = softmax(S), O = PV.
  - Key design 2: the mergeable (m, l, O) update and its table (FA2 stores
    L = m + log l).
  - Key design 3: D_i = dO_i . O_i and dS = P o (dP - D); dV = P^T dO,
    dQ = dS K, dK = dS^T Q.
  - Usage contract table: scale, causal flag, Q/KV lengths; ALiBi and MQA
    named among the mask/variant features.
* [Memory-wall page] "FlashAttention: The Algorithm That Beat the Memory
  Wall" (repo-explainer.com), "A Tile, a Register File, and a Trick Called
  Online Softmax" (per-step normalised recurrence) and "Varlen Is the Quiet
  Superpower" (packed sequences).

The plain definition is the oracle: for each (sequence, query head) it
materialises S and P in float64 and applies the formulas above directly.  The
method reaches that same result up to rounding order, so no step of the tiled
algorithm is emulated here, except in ``online_softmax_forward`` which exists
only so the tests can check the pages' recurrence against the definition.

Readings where the pages are silent or ambiguous (each also stated where used):

R1  A bias or mask is added after the 1/sqrt(d) scaling and is not scaled.
R2  The FA1 note's backward sketch forms raw scores with no scale; by the chain
    rule dQ and dK carry the factor ``scale`` and dV does not.
R3  "log" in L = m + log l is the natural logarithm.
R4  ALiBi: bias[i, j] = -slope_h * (i - j), i the query and j the key position
    local to the sequence; slopes are per query head.
R5  GQA/MQA: contiguous groups, kv head g = h // (Hq / Hkv); dK and dV of a kv
    head are sums over its query heads.
R6  Causal: key j visible to query i iff j <= i, positions local to the
    sequence; query and key lengths are equal per sequence.
R7  A row with no visible key (cannot occur under R6) gets O = 0, LSE = -inf.
R8  No dropout (the usage contract's example passes dropout_p = 0.0).
R9  Sliding window (named only, among the mask variants of the usage contract
    table): a causal band, key j visible to query i iff i - window <= j <= i;
    window None (or < 0) means no window; window requires causal.
R10 Decode over a KV cache (named only: flash_attn_with_kvcache and the
    small-query paths in [FA1 note] "Long context and inference remain
    unsolved"): sequence b holds L_b cached tokens, the new ones included; its
    q_len query rows are its newest tokens, at positions L_b - q_len + i, and
    attend under R6 (causal, positions local to the sequence), with R4's bias
    and R9's window.  Decode therefore equals the last q_len rows of the
    causal forward over the whole sequence.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "attention_forward", "attention_backward", "head_forward", "head_backward",
    "head_scores", "online_softmax_forward", "online_softmax_forward_normalised",
    "forward_rows", "backward_query_rows", "backward_key_rows", "head_row_stats",
    "decode_forward", "head_forward_chunked", "head_backward_chunked",
]


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def _window(window, causal):
    if window is None or window < 0:
        return None
    if not causal:
        raise ValueError("a sliding window needs causal=True (R9)")
    return int(window)


def head_scores(q, k, scale, causal, slope=None, window=None):
    """Scores of one (sequence, head): S = scale * q k^T + bias, masked.

    [FA1 note] Key design 1, S = QK^T / sqrt(d) with ``scale`` in place of
    1/sqrt(d) (usage contract: softmax_scale).  ALiBi bias per R4, added after
    scaling (R1).  Causal mask per R6, sliding window per R9: masked entries
    are -inf.
    """
    window = _window(window, causal)
    q = _f64(q)
    k = _f64(k)
    L = q.shape[0]
    S = scale * (q @ k.T)
    if slope is not None:
        i = np.arange(L, dtype=np.float64)[:, None]
        j = np.arange(k.shape[0], dtype=np.float64)[None, :]
        S = S - float(slope) * (i - j)
    if causal:
        vis = np.arange(k.shape[0])[None, :] <= np.arange(L)[:, None]
        if window is not None:
            vis &= np.arange(k.shape[0])[None, :] >= np.arange(L)[:, None] - window
        S = np.where(vis, S, -np.inf)
    return S


def _softmax_rows(S):
    """P = softmax(S) row-wise and LSE = m + log(l) (R3, R7)."""
    m = S.max(axis=1, initial=-np.inf) if S.shape[1] else np.full(S.shape[0], -np.inf)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    E = np.exp(S - m_safe[:, None])
    E[~finite] = 0.0
    l = E.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        P = np.where(l[:, None] > 0, E / np.where(l > 0, l, 1.0)[:, None], 0.0)
        lse = np.where(l > 0, m_safe + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return P, lse


def head_forward(q, k, v, scale, causal, slope=None, window=None):
    """O and LSE of one (sequence, head), materialising S and P.

    [FA1 note] Key design 1: P = softmax(S), O = P V.  Key design 2's table:
    L = m + log l is saved per row for the backward (R3).
    Returns (O, LSE, P).
    """
    S = head_scores(q, k, scale, causal, slope, window)
    P, lse = _softmax_rows(S)
    O = P @ _f64(v)
    return O, lse, P


def head_backward(q, k, v, do, scale, causal, slope=None, window=None):
    """dQ, dK, dV of one (sequence, head) from the materialised P.

    [FA1 note] Key design 3: dV = P^T dO; dP = dO V^T; D_i = rowsum(P o dP)
    (equal to dO_i . O_i); dS = P o (dP - D); dQ = dS K, dK = dS^T Q with the
    chain-rule factor ``scale`` (R2).  The bias has no gradient.
    Returns (dQ, dK, dV, O, LSE, D).
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    do = _f64(do)
    O, lse, P = head_forward(q, k, v, scale, causal, slope, window)
    dV = P.T @ do
    dP = do @ v.T
    D = (P * dP).sum(axis=1)
    dS = P * (dP - D[:, None])
    dQ = scale * (dS @ k)
    dK = scale * (dS.T @ q)
    return dQ, dK, dV, O, lse, D


def _layout(q, k, cu_seqlens):
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    if cu_seqlens is None:
        cu = np.array([0, T], dtype=np.int64)
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
    return T, Hq, Hkv, d, cu


def _slope(alibi_slopes, h):
    return None if alibi_slopes is None else float(alibi_slopes[h])


def attention_forward(q, k, v, scale, causal, cu_seqlens=None, alibi_slopes=None,
                      heads=None, seqs=None, window=None):
    """O [T, Hq, d] and LSE [Hq, T] of packed multi-head attention.

    Sequences are the segments [cu[b], cu[b+1]) of the token axis ([Memory-wall
    page] Varlen); kv head of query head h per R5.  ``heads`` / ``seqs``
    restrict the work to whole heads / sequences (other entries stay NaN).
    """
    T, Hq, Hkv, d, cu = _layout(q, k, cu_seqlens)
    group = Hq // Hkv
    O = np.full((T, Hq, v.shape[2]), np.nan)
    LSE = np.full((Hq, T), np.nan)
    for b in (range(len(cu) - 1) if seqs is None else seqs):
        s, e = int(cu[b]), int(cu[b + 1])
        for h in (range(Hq) if heads is None else heads):
            g = h // group
            o, lse, _ = head_forward(q[s:e, h], k[s:e, g], v[s:e, g], scale, causal,
                                     _slope(alibi_slopes, h), window)
            O[s:e, h] = o
            LSE[h, s:e] = lse
    return O, LSE


def attention_backward(q, k, v, do, scale, causal, cu_seqlens=None, alibi_slopes=None,
                       heads=None, seqs=None, window=None):
    """dQ, dK, dV (plus O, LSE, D) of packed multi-head attention.

    dK and dV of kv head g sum the contributions of its query heads (R5).
    ``heads`` selects query heads; a kv head's dK/dV is complete only when all
    of its group's query heads are selected.
    """
    T, Hq, Hkv, d, cu = _layout(q, k, cu_seqlens)
    group = Hq // Hkv
    dQ = np.full(q.shape, np.nan)
    dK = np.zeros(k.shape)
    dV = np.zeros(v.shape)
    O = np.full((T, Hq, v.shape[2]), np.nan)
    LSE = np.full((Hq, T), np.nan)
    D = np.full((Hq, T), np.nan)
    for b in (range(len(cu) - 1) if seqs is None else seqs):
        s, e = int(cu[b]), int(cu[b + 1])
        for h in (range(Hq) if heads is None else heads):
            g = h // group
            dq, dk, dv, o, lse, dd = head_backward(
                q[s:e, h], k[s:e, g], v[s:e, g], do[s:e, h], scale, causal,
                _slope(alibi_slopes, h), window)
            dQ[s:e, h] = dq
            dK[s:e, g] += dk
            dV[s:e, g] += dv
            O[s:e, h] = o
            LSE[h, s:e] = lse
            D[h, s:e] = dd
    return dQ, dK, dV, O, LSE, D


# --------------------------------------------------------------------------
# The pages' recurrences, written out so that the tests can check them
# against the definition above (exactness, FA1 Theorem 1).
# --------------------------------------------------------------------------

def online_softmax_forward(q, k, v, scale, causal, slope=None, block_q=1, block_k=1, window=None):
    """Forward by the mergeable (m, l, O) state, FA1 loop order.

    [FA1 note] Key design 1: K/V blocks in the outer loop, Q blocks in the
    inner loop, state kept per query row.  Key design 2: for a new score tile
    with row max m~ and local sum l~ of P~ = exp(S - m~):
        m' = max(m, m~),  l' = e^(m - m') l + e^(m~ - m') l~,
        O' = (e^(m - m') l O + e^(m~ - m') P~ V) / l'.
    Returns (O, LSE) with LSE = m + log l (FA2, Key design 2's table).
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    Lq, Lk = q.shape[0], k.shape[0]
    O = np.zeros((Lq, v.shape[1]))
    m = np.full(Lq, -np.inf)
    l = np.zeros(Lq)
    S_all = head_scores(q, k, scale, causal, slope, window)   # tiles are read from here
    for ks in range(0, Lk, block_k):
        ke = min(ks + block_k, Lk)
        for qs in range(0, Lq, block_q):
            qe = min(qs + block_q, Lq)
            S = S_all[qs:qe, ks:ke]
            m_t = S.max(axis=1)
            ok = np.isfinite(m_t)
            if not ok.any():
                continue
            P_t = np.zeros_like(S)
            P_t[ok] = np.exp(S[ok] - m_t[ok, None])
            l_t = P_t.sum(axis=1)
            # rows that see no key of this tile merge nothing and keep their state
            rows = np.arange(qs, qe)[ok]
            m_old, l_old, O_old = m[rows], l[rows], O[rows]
            m_t, l_t, PV_t = m_t[ok], l_t[ok], (P_t @ v[ks:ke])[ok]
            m_new = np.maximum(m_old, m_t)
            a_old = np.where(np.isfinite(m_old), np.exp(m_old - m_new), 0.0)
            a_new = np.exp(m_t - m_new)
            l_new = a_old * l_old + a_new * l_t
            O[rows] = ((a_old * l_old)[:, None] * O_old + a_new[:, None] * PV_t) / l_new[:, None]
            m[rows] = m_new
            l[rows] = l_new
    lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return O, lse


def online_softmax_forward_normalised(q, k, v, scale, causal, slope=None, block_k=1):
    """Forward by the per-step normalised recurrence, one query tile.

    [Memory-wall page] online-softmax sketch: per K/V tile, m_new = max(m,
    max S); P = exp(S - m_new); l_new = e^(m - m_new) l + sum P;
    O = (e^(m - m_new) l / l_new) O + (P V) / l_new.  The sketch calls l
    "running_lse"; it is the running exponential sum (read as such).
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    Lq, Lk = q.shape[0], k.shape[0]
    S_all = head_scores(q, k, scale, causal, slope)
    O = np.zeros((Lq, v.shape[1]))
    m = np.full(Lq, -np.inf)
    l = np.zeros(Lq)
    for ks in range(0, Lk, block_k):
        S = S_all[:, ks:ks + block_k]
        m_new = np.maximum(m, S.max(axis=1))
        live = np.isfinite(m_new)
        P = np.zeros_like(S)
        P[live] = np.exp(S[live] - m_new[live, None])
        alpha = np.where(np.isfinite(m), np.exp(m - np.where(live, m_new, 0.0)), 0.0)
        l_new = alpha * l + P.sum(axis=1)
        safe = np.where(l_new > 0, l_new, 1.0)
        O = np.where(live[:, None],
                     (alpha * l / safe)[:, None] * O + (P @ v[ks:ks + block_k]) / safe[:, None],
                     O)
        m, l = np.where(live, m_new, m), np.where(live, l_new, l)
    lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return O, lse


# --------------------------------------------------------------------------
# Row-sampled forms for workloads too large to materialise whole: each output
# row is computed from its own definition, one at a time.
# --------------------------------------------------------------------------

def _seq_of(cu, t):
    b = int(np.searchsorted(cu, t, side="right") - 1)
    return b, int(cu[b]), int(cu[b + 1])


def forward_rows(q, k, v, scale, causal, rows, cu_seqlens=None, alibi_slopes=None, window=None):
    """O and LSE at sampled (token t, query head h) rows.

    Row i of Key design 1's definition needs only q_i and the sequence's keys:
    S_i = scale q_i k^T + bias_i (masked), P_i = softmax(S_i), O_i = P_i V.
    Returns (O [n, d], LSE [n]).
    """
    T, Hq, Hkv, d, cu = _layout(q, k, cu_seqlens)
    group = Hq // Hkv
    outO, outL = [], []
    for t, h in rows:
        b, s, e = _seq_of(cu, t)
        g = h // group
        i = t - s
        kk = _f64(k[s:e, g])
        srow = scale * (kk @ _f64(q[t, h]))
        if alibi_slopes is not None:
            srow = srow - float(alibi_slopes[h]) * (i - np.arange(e - s, dtype=np.float64))
        if causal:
            vis = np.arange(e - s) <= i
            if _window(window, causal) is not None:
                vis &= np.arange(e - s) >= i - window
            srow = np.where(vis, srow, -np.inf)
        P, lse = _softmax_rows(srow[None, :])
        outO.append((P @ _f64(v[s:e, g]))[0])
        outL.append(lse[0])
    return np.array(outO), np.array(outL)


def head_row_stats(q, k, v, do, scale, causal, s, e, h, g, slope=None, chunk=1024, window=None):
    """LSE_i and D_i = dO_i . O_i of every query row of one (sequence, head).

    Computed in row chunks (each chunk materialises its rows of S), so whole
    long heads fit in memory.  D is None when ``do`` is None.
    """
    L = e - s
    kk = _f64(k[s:e, g])
    vv = _f64(v[s:e, g])
    lse = np.empty(L)
    D = None if do is None else np.empty(L)
    for r0 in range(0, L, chunk):
        r1 = min(r0 + chunk, L)
        S = scale * (_f64(q[s + r0:s + r1, h]) @ kk.T)
        i = np.arange(r0, r1, dtype=np.float64)[:, None]
        j = np.arange(L, dtype=np.float64)[None, :]
        if slope is not None:
            S = S - slope * (i - j)
        if causal:
            vis = j <= i
            if _window(window, causal) is not None:
                vis &= j >= i - window
            S = np.where(vis, S, -np.inf)
        P, lse[r0:r1] = _softmax_rows(S)
        if D is not None:
            D[r0:r1] = (_f64(do[s + r0:s + r1, h]) * (P @ vv)).sum(axis=1)
    return lse, D


def backward_query_rows(q, k, v, do, scale, causal, rows, cu_seqlens=None,
                        alibi_slopes=None, window=None):
    """dQ at sampled (token t, query head h) rows.

    Row i of Key design 3: P_i from its scores, dP_i = dO_i V^T,
    D_i = dO_i . O_i, dS_i = P_i o (dP_i - D_i), dQ_i = scale dS_i K (R2).
    """
    T, Hq, Hkv, d, cu = _layout(q, k, cu_seqlens)
    group = Hq // Hkv
    out = []
    for t, h in rows:
        b, s, e = _seq_of(cu, t)
        g = h // group
        i = t - s
        kk = _f64(k[s:e, g])
        vv = _f64(v[s:e, g])
        srow = scale * (kk @ _f64(q[t, h]))
        if alibi_slopes is not None:
            srow = srow - float(alibi_slopes[h]) * (i - np.arange(e - s, dtype=np.float64))
        if causal:
            vis = np.arange(e - s) <= i
            if _window(window, causal) is not None:
                vis &= np.arange(e - s) >= i - window
            srow = np.where(vis, srow, -np.inf)
        P, _ = _softmax_rows(srow[None, :])
        P = P[0]
        o = P @ vv
        dOi = _f64(do[t, h])
        dP = vv @ dOi
        D = dOi @ o
        dS = P * (dP - D)
        out.append(scale * (dS @ kk))
    return np.array(out)


def backward_key_rows(q, k, v, do, scale, causal, rows, cu_seqlens=None,
                      alibi_slopes=None, stats_cache=None, window=None):
    """dK and dV at sampled (token t, kv head g) rows.

    Column j of Key design 3's formulas: dV_j = sum_i P_ij dO_i and
    dK_j = scale sum_i dS_ij q_i, summed over the query heads of g's group
    (R5), with P_ij = exp(S_ij - LSE_i) and dS_ij = P_ij (dP_ij - D_i).  LSE_i
    and D_i of every row come from ``head_row_stats``.
    Returns (dK [n, d], dV [n, d]).
    """
    T, Hq, Hkv, d, cu = _layout(q, k, cu_seqlens)
    group = Hq // Hkv
    if stats_cache is None:
        stats_cache = {}
    outK, outV = [], []
    for t, g in rows:
        b, s, e = _seq_of(cu, t)
        j = t - s
        dk = np.zeros(d)
        dv = np.zeros(v.shape[2])
        for h in range(g * group, (g + 1) * group):
            slope = _slope(alibi_slopes, h)
            if (b, h) not in stats_cache:
                stats_cache[(b, h)] = head_row_stats(q, k, v, do, scale, causal,
                                                     s, e, h, g, slope, window=window)
            lse, D = stats_cache[(b, h)]
            qq = _f64(q[s:e, h])
            dd = _f64(do[s:e, h])
            i = np.arange(e - s, dtype=np.float64)
            scol = scale * (qq @ _f64(k[t, g]))
            if slope is not None:
                scol = scol - slope * (i - j)
            if causal:
                vis = i >= j
                if _window(window, causal) is not None:
                    vis &= i <= j + window
                scol = np.where(vis, scol, -np.inf)
            Pcol = np.where(np.isfinite(scol), np.exp(scol - lse), 0.0)
            dPcol = dd @ _f64(v[t, g])
            dScol = Pcol * (dPcol - D)
            dv += Pcol @ dd
            dk += scale * (dScol @ qq)
        outK.append(dk)
        outV.append(dv)
    return np.array(outK), np.array(outV)


# --------------------------------------------------------------------------
# Whole heads of long sequences, by blocks of query rows.  Rows of S and P
# are independent of each other, so each block of rows is Key design 1 / 3
# applied to those rows; the sums over rows that make dK and dV are added
# block by block.  Only the memory held at once changes, not the arithmetic
# of any entry.
# --------------------------------------------------------------------------

def _score_rows(q_rows, k, scale, causal, r0, slope=None, window=None):
    """Rows r0 .. r0 + len(q_rows) - 1 of ``head_scores`` (same definition:
    scale q k^T, R4's bias -slope (i - j), R6's causal mask and R9's band)."""
    window = _window(window, causal)
    S = scale * (_f64(q_rows) @ _f64(k).T)
    i = np.arange(r0, r0 + S.shape[0], dtype=np.float64)[:, None]
    j = np.arange(S.shape[1], dtype=np.float64)[None, :]
    if slope is not None:
        S = S - float(slope) * (i - j)
    if causal:
        vis = j <= i
        if window is not None:
            vis &= j >= i - window
        S = np.where(vis, S, -np.inf)
    return S


def head_forward_chunked(q, k, v, scale, causal, slope=None, window=None, chunk=1024):
    """O and LSE of one (sequence, head), ``chunk`` query rows at a time.

    [FA1 note] Key design 1 for each block of rows: S rows, P = softmax(S)
    row-wise, O = P V, and L = m + log l (Key design 2's table, R3)."""
    L = q.shape[0]
    vv = _f64(v)
    O = np.empty((L, vv.shape[1]))
    lse = np.empty(L)
    for r0 in range(0, L, chunk):
        r1 = min(r0 + chunk, L)
        P, lse[r0:r1] = _softmax_rows(_score_rows(q[r0:r1], k, scale, causal, r0, slope, window))
        O[r0:r1] = P @ vv
    return O, lse


def head_backward_chunked(q, k, v, do, scale, causal, slope=None, window=None, chunk=1024):
    """dQ, dK, dV, O, LSE and D of one (sequence, head), ``chunk`` query rows
    at a time.

    [FA1 note] Key design 3 for each block of rows: P from the rows' scores,
    dP = dO V^T, D = rowsum(P o dP), dS = P o (dP - D), dQ = scale dS K (R2)
    for those rows; dV = P^T dO and dK = scale dS^T Q summed over the blocks.
    Same results as ``head_backward`` without holding the whole L x L
    matrices.  Returns (dQ, dK, dV, O, LSE, D)."""
    L = q.shape[0]
    qq, kk, vv, dd = _f64(q), _f64(k), _f64(v), _f64(do)
    dQ = np.empty(qq.shape)
    dK = np.zeros(kk.shape)
    dV = np.zeros(vv.shape)
    O = np.empty((L, vv.shape[1]))
    lse = np.empty(L)
    D = np.empty(L)
    for r0 in range(0, L, chunk):
        r1 = min(r0 + chunk, L)
        P, lse[r0:r1] = _softmax_rows(_score_rows(qq[r0:r1], kk, scale, causal, r0, slope, window))
        O[r0:r1] = P @ vv
        dP = dd[r0:r1] @ vv.T
        D[r0:r1] = (P * dP).sum(axis=1)
        dS = P * (dP - D[r0:r1, None])
        dQ[r0:r1] = scale * (dS @ kk)
        dK += scale * (dS.T @ qq[r0:r1])
        dV += P.T @ dd[r0:r1]
    return dQ, dK, dV, O, lse, D


# --------------------------------------------------------------------------
# Decode: the newest tokens of each sequence against its KV cache (R10).
# --------------------------------------------------------------------------

def decode_forward(q, k_cache, v_cache, cache_seqlens, scale, q_len=1, alibi_slopes=None,
                   window=None):
    """O and LSE of the q_len newest tokens of every sequence (R10).

    q: [B * q_len, Hq, d], rows b * q_len .. b * q_len + q_len - 1 belonging to
    sequence b; k_cache, v_cache: [B, S_max, Hkv, d]; cache_seqlens: [B] (None:
    every sequence holds S_max tokens).  Row i of sequence b is the query at
    position p_i = L_b - q_len + i; keys j < L_b of its cache; S = scale q k^T
    plus R4's bias -slope (p_i - j), masked where j > p_i or (R9)
    j < p_i - window; P = softmax(S) ([FA1 note] Key design 1); O = P V.
    Returns O [B * q_len, Hq, d] and LSE [Hq, B * q_len].
    """
    B, S_max, Hkv, d = k_cache.shape
    Hq = q.shape[1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    group = Hq // Hkv
    window = _window(window, True)
    O = np.empty((B * q_len, Hq, v_cache.shape[3]))
    LSE = np.empty((Hq, B * q_len))
    for b in range(B):
        L = S_max if cache_seqlens is None else int(cache_seqlens[b])
        if not q_len <= L <= S_max:
            raise ValueError("a cache must hold its q_len new tokens and at most S_max")
        pos = (L - q_len + np.arange(q_len))[:, None]
        j = np.arange(L)[None, :]
        vis = j <= pos
        if window is not None:
            vis &= j >= pos - window
        rows = slice(b * q_len, (b + 1) * q_len)
        for h in range(Hq):
            g = h // group
            S = scale * (_f64(q[rows, h]) @ _f64(k_cache[b, :L, g]).T)
            if alibi_slopes is not None:
                S = S - float(alibi_slopes[h]) * (pos - j)
            P, lse = _softmax_rows(np.where(vis, S, -np.inf))
            O[rows, h] = P @ _f64(v_cache[b, :L, g])
            LSE[h, rows] = lse
    return O, LSE
