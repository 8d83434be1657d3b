"""Parity at the four bf16 workloads' full sizes, through the same C-ABI
calls and launch configuration the benchmark times (GPU).

Three kinds of check, all against the fp64 oracle:

* the GPT-2-medium shape (B=8, H=16, N=1024, d=64) whole: every element of
  O, LSE, dQ, dK and dV;
* whole heads of the long workloads, every row: one query head of the
  long-context workload, one query head across all 64 sequences of the
  packed batch, and one kv head's whole group of 8 query heads (so its dK
  and dV are complete) of the GQA + ALiBi workload.  The oracle computes
  them by blocks of query rows (``head_backward_chunked``);
* sampled rows of every head: O, LSE and dQ of sampled (token, head) rows
  (``forward_rows``, ``backward_query_rows``) and dK / dV of sampled key rows
  (``backward_key_rows``), at sequence starts and ends, 64/128/256-row tile
  edges and random positions.

Tolerances as in the other parity tests (O stored as fp32): O 1e-2, LSE 1e-3,
each gradient 2e-2 x the largest |value| of that gradient among the rows the
oracle computed.
"""
import numpy as np
import pytest

from oracle import attention_fp64 as A
from exact_io_aware_36_gb300 import fa
from exact_io_aware_36_gb300 import inputs as I
from tests import gpu_util as G

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL_O, TOL_LSE, TOL_GRAD = 1e-2, 1e-3, 2e-2


def run_on_gpu(x):
    """fa_fwd and fa_bwd through the binding; returns torch tensors on the
    GPU: O (fp32), LSE, dQ, dK, dV."""
    t = G.torch()
    w = x.workload
    q, k, v, do = (G.to_dev(x, n) for n in ("q", "k", "v", "do"))
    cu = t.from_numpy(x.cu_seqlens).cuda() if w.varlen else None
    slopes = t.from_numpy(x.alibi_slopes).cuda() if x.alibi_slopes is not None else None
    kw = dict(causal=w.causal, scale=x.scale, cu_seqlens=cu, max_seqlen=w.N if w.varlen else None,
              batch=None if w.varlen else w.B, alibi_slopes=slopes, window=w.window, check=True)
    o, lse = fa.attention_forward(q, k, v, out_dtype=t.float32, **kw)
    dq, dk, dv = fa.attention_backward(q, k, v, o, do, lse, **kw)
    t.cuda.synchronize()
    del q, k, v, do
    return o, lse, dq, dk, dv


def f64(t_):
    return G.as_f64(t_)


def sample_rows(x, n_random, rng, heads):
    cu = x.cu_seqlens
    rows = []
    for b in range(len(cu) - 1):
        s, e = int(cu[b]), int(cu[b + 1])
        for off in (0, 63, 64, 127, 128, 255, 256, e - s - 1):
            if 0 <= off < e - s:
                rows.append(s + off)
        if len(rows) >= n_random:
            break
    rows = sorted(set(rows))[:n_random] + [int(t) for t in rng.integers(0, x.T, size=n_random)]
    return [(t, int(rng.integers(0, heads))) for t in rows]


def check_sampled(x, outs):
    w = x.workload
    o, lse, dq, dk, dv = outs
    rng = np.random.Generator(np.random.PCG64(1234))
    qrows = sample_rows(x, 24, rng, w.Hq)
    O_r, lse_r = A.forward_rows(x.q, x.k, x.v, x.scale, w.causal, qrows, x.cu_seqlens,
                                x.alibi_slopes)
    dq_r = A.backward_query_rows(x.q, x.k, x.v, x.do, x.scale, w.causal, qrows, x.cu_seqlens,
                                 x.alibi_slopes)
    tq = [t for t, _ in qrows]
    hq = [h for _, h in qrows]
    O_g = f64(o[tq, hq])
    lse_g = f64(lse[hq, tq])
    dq_g = f64(dq[tq, hq])
    # key rows from two (sequence, kv head) slices: the oracle computes the
    # row statistics of each query head of those slices once
    cu = x.cu_seqlens
    krows = []
    for b in (0, len(cu) - 2):
        s, e = int(cu[b]), int(cu[b + 1])
        g = int(rng.integers(0, w.Hkv))
        for off in (0, 1, 127, 128, (e - s) // 2, e - s - 1):
            if 0 <= off < e - s:
                krows.append((s + off, g))
    dk_r, dv_r = A.backward_key_rows(x.q, x.k, x.v, x.do, x.scale, w.causal, krows, x.cu_seqlens,
                                     x.alibi_slopes, {})
    tk = [t for t, _ in krows]
    gk = [g for _, g in krows]
    errs = {"O": np.abs(O_g - O_r).max(), "LSE": np.abs(lse_g - lse_r).max(),
            "dQ": np.abs(dq_g - dq_r).max() / np.abs(dq_r).max(),
            "dK": np.abs(f64(dk[tk, gk]) - dk_r).max() / np.abs(dk_r).max(),
            "dV": np.abs(f64(dv[tk, gk]) - dv_r).max() / np.abs(dv_r).max()}
    return errs


def check_whole_heads(x, outs, seqs, kv_head):
    """Every row of the query heads of kv head ``kv_head`` (all of its group)
    in the sequences ``seqs``: O, LSE, dQ of each head; dK and dV of the kv
    head, summed over the group."""
    w = x.workload
    o, lse, dq, dk, dv = outs
    group = w.Hq // w.Hkv
    cu = x.cu_seqlens
    worst = {"O": 0.0, "LSE": 0.0}
    gerr = {"dQ": [0.0, 0.0], "dK": [0.0, 0.0], "dV": [0.0, 0.0]}   # max |err|, max |ref|
    for b in seqs:
        s, e = int(cu[b]), int(cu[b + 1])
        if e == s:
            continue
        dK_r = np.zeros((e - s, w.d))
        dV_r = np.zeros((e - s, w.d))
        for h in range(kv_head * group, (kv_head + 1) * group):
            slope = None if x.alibi_slopes is None else float(x.alibi_slopes[h])
            dq_r, dk_h, dv_h, O_r, lse_r, _ = A.head_backward_chunked(
                x.q[s:e, h], x.k[s:e, kv_head], x.v[s:e, kv_head], x.do[s:e, h], x.scale,
                w.causal, slope, w.window)
            dK_r += dk_h
            dV_r += dv_h
            worst["O"] = max(worst["O"], np.abs(f64(o[s:e, h]) - O_r).max())
            worst["LSE"] = max(worst["LSE"], np.abs(f64(lse[h, s:e]) - lse_r).max())
            ge = gerr["dQ"]
            ge[0] = max(ge[0], np.abs(f64(dq[s:e, h]) - dq_r).max())
            ge[1] = max(ge[1], np.abs(dq_r).max())
        for name, got, ref in (("dK", dk, dK_r), ("dV", dv, dV_r)):
            ge = gerr[name]
            ge[0] = max(ge[0], np.abs(f64(got[s:e, kv_head]) - ref).max())
            ge[1] = max(ge[1], np.abs(ref).max())
    errs = dict(worst)
    for name, (err, ref) in gerr.items():
        errs[name] = err / ref
    return errs


def assert_within(errs, what):
    print(what, {k_: float(v_) for k_, v_ in errs.items()})
    assert errs["O"] <= TOL_O and errs["LSE"] <= TOL_LSE, (what, errs)
    assert errs["dQ"] <= TOL_GRAD and errs["dK"] <= TOL_GRAD and errs["dV"] <= TOL_GRAD, (what, errs)


def test_gpt2m_shape_whole():
    """B=8, H=16, N=1024, d=64: every element of every output."""
    x = I.make_inputs(I.workload("c2_gpt2m"), seed=0)
    o, lse, dq, dk, dv = (f64(t_) for t_ in run_on_gpu(x))
    w = x.workload
    dq_r, dk_r, dv_r, O_r, lse_r, _ = A.attention_backward(x.q, x.k, x.v, x.do, x.scale, w.causal,
                                                           x.cu_seqlens, x.alibi_slopes)
    errs = {"O": np.abs(o - O_r).max(), "LSE": np.abs(lse - lse_r).max()}
    for name, g, r in (("dQ", dq, dq_r), ("dK", dk, dk_r), ("dV", dv, dv_r)):
        errs[name] = np.abs(g - r).max() / np.abs(r).max()
    assert_within(errs, "c2_gpt2m whole")


# workload -> (sequences, kv head) whose every row is checked
WHOLE_HEADS = {
    "c3_long": ([0], 31),              # one head of the 16384-token sequence
    "c4_varlen": (list(range(64)), 7), # one head across all 64 packed sequences
    "c5_gqa_alibi": ([1], 3),          # kv head 3 and its 8 query heads, sequence 1
}


@pytest.mark.parametrize("name", ["c2_gpt2m", "c3_long", "c4_varlen", "c5_gqa_alibi"])
def test_full_size(name):
    x = I.make_inputs(I.workload(name), seed=0)
    outs = run_on_gpu(x)
    for t_ in outs:
        assert bool(G.torch().isfinite(t_).all())
    assert_within(check_sampled(x, outs), name + " sampled rows")
    if name in WHOLE_HEADS:
        seqs, g = WHOLE_HEADS[name]
        assert_within(check_whole_heads(x, outs, seqs, g), name + " whole heads")
