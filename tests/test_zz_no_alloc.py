"""fa_bwd_static_scratch: the backward for callers that cannot allocate.

Plugins or custom-op hooks that get no workspace, runtimes that forbid
device allocation after start-up, and code that must not call cudaMalloc on
its hot path use this entry point instead of fa_bwd; it keeps its scratch in
a fixed array inside the library.  These tests call it through the C ABI and
compare it with fa_bwd (given a workspace allocated here) on two calls in a
row, with different problem sizes, larger first, so the second call runs
over whatever the first left in the shared array:

* deterministic backward: dq, dk and dv must equal fa_bwd's bit for bit
  (same kernels, same inputs, no atomics), so any stale scratch shows;
* default backward: dk and dv bit for bit (they never touch the scratch's
  accumulator), dq within 2e-2 x max |dq| (its fp32 reduce order varies);
* one case against the fp64 oracle at the backward tolerances.

Host-side checks (no GPU): argument errors get fa_bwd's status codes, an
empty packed batch succeeds, and only then is the size limit applied.

This file is named to be collected last, so a run that stops at the first
failure has run every other test before it.
"""
import numpy as np
import pytest

from exact_io_aware_36_gb300 import build, fa
from exact_io_aware_36_gb300 import inputs as I

TOL_GRAD = 2e-2


@pytest.fixture(scope="module")
def lib():
    build.build()
    return fa.load()


def _static(**kw):
    A = 0x10000      # fake, aligned device address: never dereferenced here
    a = dict(B=1, Hq=32, Hkv=32, N=16384, d=128, causal=1, window=-1, cu=None, T=0, det=0,
             dtype=fa.FA_BF16, q=A)
    a.update(kw)
    return fa.fa_bwd_static_scratch(a["q"], A, A, A, A, A, A, A, A, a["B"], a["Hq"], a["Hkv"],
                                    a["N"], a["d"], 0.088, a["causal"], a["window"], a["cu"],
                                    a["T"], None, a["dtype"], fa.FA_FP32, a["det"], None)


def test_refuses_problems_larger_than_the_scratch(lib):
    """A problem whose workspace exceeds the fixed array is refused with
    FA_ERR_WORKSPACE before any CUDA call (runs without a GPU)."""
    B, Hq, N, d = 1, 32, 16384, 128
    assert fa.fa_bwd_workspace_size(B, Hq, N, d, 0) > fa.FA_BWD_STATIC_SCRATCH_BYTES
    assert _static() == 5
    assert _static(det=1) == 5


def test_argument_errors_come_before_the_size_limit(lib):
    """Arguments fa_bwd rejects get fa_bwd's status, not FA_ERR_WORKSPACE,
    and an empty packed batch (no tokens, however large B * N) succeeds
    without touching the GPU (runs without a GPU)."""
    assert _static(Hkv=5) == 2                     # Hq % Hkv != 0: FA_ERR_SHAPE
    assert _static(d=96) == 3                      # FA_ERR_UNSUPPORTED
    assert _static(dtype=fa.FA_FP32) == 3
    assert _static(det=2) == 3
    assert _static(window=8, causal=0) == 3
    assert _static(q=None) == 1                    # FA_ERR_NULL
    assert _static(q=0x10008) == 4                 # FA_ERR_ALIGN
    assert _static(B=64, N=1 << 20, cu=0x20000, T=0) == 0   # empty packed batch: FA_OK
    assert _static(B=0) == 0


def _inputs(w, seed):
    import torch
    x = I.make_inputs(w, seed=seed)
    dev = lambda n: torch.from_numpy(x.bits[n].view(np.int16)).view(torch.bfloat16).cuda()
    return x, dev("q"), dev("k"), dev("v"), dev("do")


def _run_pair(w, seed, deterministic):
    """fa_fwd, then fa_bwd (caller workspace) and fa_bwd_static_scratch on the
    same inputs; returns the inputs and both gradient triples (torch, on the
    GPU)."""
    import torch
    x, q, k, v, do = _inputs(w, seed)
    cu = torch.from_numpy(x.cu_seqlens).cuda() if w.varlen else None
    slopes = torch.from_numpy(x.alibi_slopes).cuda() if w.alibi else None
    T = x.T
    o = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty((w.Hq, T), dtype=torch.float32, device="cuda")
    sp = torch.cuda.current_stream().cuda_stream
    P = lambda t: None if t is None else t.data_ptr()
    common = (w.B, w.Hq, w.Hkv, w.N, w.d, float(x.scale), int(w.causal), w.window_arg, P(cu), T,
              P(slopes))
    assert fa.fa_fwd(P(q), P(k), P(v), P(o), P(lse), *common, fa.FA_BF16, fa.FA_FP32, sp) == 0
    ref = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    ws_bytes = fa.fa_bwd_workspace_size(w.B, w.Hq, w.N, w.d, T)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    assert fa.fa_bwd(P(q), P(k), P(v), P(o), P(do), P(lse), *(P(t) for t in ref), *common,
                     fa.FA_BF16, fa.FA_FP32, deterministic, P(ws), ws_bytes, sp) == 0
    got = [torch.full_like(q, float("nan")), torch.full_like(k, float("nan")),
           torch.full_like(v, float("nan"))]
    assert fa.fa_bwd_static_scratch(P(q), P(k), P(v), P(o), P(do), P(lse), *(P(t) for t in got),
                                    *common, fa.FA_BF16, fa.FA_FP32, deterministic, sp) == 0
    assert fa.fa_check_device_error(sp) == 0
    return x, ref, got


CASES = [
    # larger first, so the second call reuses a scratch holding stale data
    I.small_case("bf16", causal=True, B=2, Hq=4, Hkv=2, N=520, d=128, alibi=True),
    I.small_case("bf16", causal=True, Hq=2, Hkv=1, d=64, seqlens=(17, 300, 1)),
]


@pytest.mark.gpu
def test_deterministic_matches_fa_bwd_bit_for_bit(lib):
    import torch
    for n, w in enumerate(CASES):
        _, ref, got = _run_pair(w, seed=40 + n, deterministic=1)
        for name, r, g in zip(("dQ", "dK", "dV"), ref, got):
            assert torch.equal(r.view(torch.int16), g.view(torch.int16)), (n, name)


@pytest.mark.gpu
def test_matches_fa_bwd_on_two_calls_in_a_row(lib):
    import torch
    for n, w in enumerate(CASES):
        _, ref, got = _run_pair(w, seed=50 + n, deterministic=0)
        for name, r, g in zip(("dK", "dV"), ref[1:], got[1:]):
            assert torch.equal(r.view(torch.int16), g.view(torch.int16)), (n, name)
        r, g = ref[0].double().cpu().numpy(), got[0].double().cpu().numpy()
        assert np.isfinite(g).all(), n
        err = np.abs(g - r).max() / max(np.abs(r).max(), 1e-30)
        assert err <= TOL_GRAD, (n, "dQ", err)


@pytest.mark.gpu
def test_matches_the_oracle(lib):
    from oracle import attention_fp64 as A
    w = CASES[0]
    x, _, got = _run_pair(w, seed=60, deterministic=0)
    refs = A.attention_backward(x.q, x.k, x.v, x.do, x.scale, w.causal, x.cu_seqlens,
                                x.alibi_slopes)[:3]
    for name, r, g in zip(("dQ", "dK", "dV"), refs, got):
        g = g.double().cpu().numpy()
        err = np.abs(g - r).max() / np.abs(r).max()
        assert err <= TOL_GRAD, (name, err)
