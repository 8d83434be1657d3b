"""The persistent dK/dV kernel's scheduling (GPU).

One CTA per SM takes (key tile, kv head, sequence) items from a counter in
the workspace, and every ring and barrier continues across the items a CTA
takes.  These cases stress what per-tile launches never saw:
- many more items than SMs, so each CTA crosses many item boundaries,
  including items of a single step;
- many short packed sequences, whose key tiles past a sequence's end hold
  no work and are skipped;
- repeated launches of the dK/dV stage alone on one workspace: the kernel's
  last CTA must put the counter back to zero, so the second launch
  recomputes every item.
Tolerances as in the other parity tests (O stored fp32).
"""
import numpy as np
import pytest

from oracle import attention_fp64 as A
from exact_io_aware_36_gb300 import fa
from exact_io_aware_36_gb300 import inputs as I
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

TOL_GRAD = 2e-2


def _check(x, res):
    w = x.workload
    _, _, dq, dk, dv = res
    dq_r, dk_r, dv_r, *_ = A.attention_backward(x.q, x.k, x.v, x.do, x.scale, w.causal,
                                                x.cu_seqlens, x.alibi_slopes, window=w.window)
    for name, a, r in (("dQ", dq, dq_r), ("dK", dk, dk_r), ("dV", dv, dv_r)):
        err = np.abs(a - r).max() / max(np.abs(r).max(), 1e-3)
        assert err <= TOL_GRAD, (name, err)


@pytest.mark.parametrize("deterministic", [False, True])
def test_many_items_per_cta(deterministic):
    # 16 key tiles x 32 heads = 512 items, about 3.4 per SM; causal, so the
    # items run from 32 steps down to 2
    w = I.small_case("bf16", causal=True, B=1, Hq=32, Hkv=32, N=2048, d=64)
    x = I.make_inputs(w, seed=71)
    _check(x, G.backward(x, deterministic=deterministic))


def test_many_short_packed_sequences():
    # 120 sequences of 1..200 tokens with max_seqlen 512: most (sequence, key
    # tile) items lie past their sequence's end and must be skipped
    g = np.random.Generator(np.random.PCG64(5))
    lens = tuple(int(v) for v in g.integers(1, 201, 120))
    w = I.small_case("bf16", causal=True, Hq=4, Hkv=2, d=128, seqlens=lens + (512,))
    x = I.make_inputs(w, seed=72)
    _check(x, G.backward(x))


@pytest.mark.parametrize("deterministic", [0, 1])
def test_repeated_dkdv_stage_recomputes_every_item(deterministic):
    t = G.torch()
    w = I.small_case("bf16", causal=True, B=2, Hq=8, Hkv=4, N=1200, d=128)
    x = I.make_inputs(w, seed=73)
    q, k, v, do = (G.to_dev(x, n) for n in ("q", "k", "v", "do"))
    o, lse = fa.attention_forward(q, k, v, causal=True, scale=x.scale, batch=w.B,
                                  out_dtype=t.float32, check=True)
    T, H, Hkv, d = w.B * w.N, w.Hq, w.Hkv, w.d
    dq, dk, dv = t.empty_like(q), t.empty_like(k), t.empty_like(v)
    wsb = fa.fa_bwd_workspace_size(w.B, H, w.N, d, 0)
    ws = t.empty(wsb, dtype=t.uint8, device="cuda")
    p = lambda a: a.data_ptr()
    stream = t.cuda.current_stream().cuda_stream

    def stage(s):
        st = fa.fa_bwd_stage(s, p(q), p(k), p(v), p(o), p(do), p(lse), p(dq), p(dk), p(dv), w.B, H,
                             Hkv, w.N, d, x.scale, True, -1, None, 0, None, fa.FA_BF16, fa.FA_FP32,
                             deterministic, p(ws), wsb, stream)
        assert st == 0, fa.fa_status_string(st)

    stage(0)
    stage(1)
    t.cuda.synchronize()
    dk1, dv1 = dk.clone(), dv.clone()
    dk.zero_()
    dv.zero_()
    stage(1)                       # no preprocess in between
    t.cuda.synchronize()
    assert fa.fa_check_device_error(None) == 0
    assert t.equal(dk, dk1) and t.equal(dv, dv1)
    _, _, _, dk_r, dv_r = G.backward(x, deterministic=bool(deterministic), base_workspace=True)
    assert np.array_equal(G.as_f64(dk), dk_r) and np.array_equal(G.as_f64(dv), dv_r)


def test_dkdv_stage_with_a_negative_counter_reports_and_recovers():
    # A workspace whose item counter was never zeroed (here: -1000) must not
    # turn into negative item indices: the stage does no work, sets
    # FA_ERR_WORKSPACE, and puts the counter back to zero, so the next launch
    # computes every item.
    t = G.torch()
    w = I.small_case("bf16", causal=True, B=1, Hq=4, Hkv=2, N=700, d=128)
    x = I.make_inputs(w, seed=74)
    q, k, v, do = (G.to_dev(x, n) for n in ("q", "k", "v", "do"))
    o, lse = fa.attention_forward(q, k, v, causal=True, scale=x.scale, batch=w.B,
                                  out_dtype=t.float32, check=True)
    T, H, Hkv, d = w.B * w.N, w.Hq, w.Hkv, w.d
    dq, dk, dv = t.empty_like(q), t.empty_like(k), t.empty_like(v)
    wsb = fa.fa_bwd_workspace_size(w.B, H, w.N, d, 0)
    ws = t.empty(wsb, dtype=t.uint8, device="cuda")
    r256 = lambda n: (n + 255) // 256 * 256
    ctr = ws[r256(H * T * 4) + r256(H * T * d * 4):].view(t.int32)
    p = lambda a: a.data_ptr()
    stream = t.cuda.current_stream().cuda_stream

    def stage(s):
        st = fa.fa_bwd_stage(s, p(q), p(k), p(v), p(o), p(do), p(lse), p(dq), p(dk), p(dv), w.B, H,
                             Hkv, w.N, d, x.scale, True, -1, None, 0, None, fa.FA_BF16, fa.FA_FP32,
                             0, p(ws), wsb, stream)
        assert st == 0, fa.fa_status_string(st)

    stage(0)
    ctr[0] = -1000
    ctr[1] = 0
    stage(1)
    t.cuda.synchronize()
    assert fa.STATUS[fa.fa_check_device_error(None)] == "FA_ERR_WORKSPACE"
    assert int(ctr[0]) == 0 and int(ctr[1]) == 0
    stage(1)
    stage(2)
    t.cuda.synchronize()
    assert fa.fa_check_device_error(None) == 0
    _, _, dq_r, dk_r, dv_r = G.backward(x, base_workspace=True)
    assert np.array_equal(G.as_f64(dk), dk_r) and np.array_equal(G.as_f64(dv), dv_r)
    err = np.abs(G.as_f64(dq) - dq_r).max() / max(np.abs(dq_r).max(), 1e-3)
    assert err <= 1e-2, err
