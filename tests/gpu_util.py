"""Helpers of the GPU parity tests: move seeded inputs to the device, call
the library through its binding, and guard output buffers with canary bands
(extra head and tail regions filled with a NaN pattern that must survive the
call, a bounds check of every store)."""
import numpy as np

from exact_io_aware_36_gb300 import fa
from exact_io_aware_36_gb300 import inputs as I

GUARD = 4096   # elements of canary before and after each output


def torch():
    import torch as t
    return t


def to_dev(x: I.Inputs, name: str):
    t = torch()
    arr = getattr(x, name)
    if arr is None:
        return None
    if x.workload.dtype == "bf16":
        return t.from_numpy(np.ascontiguousarray(x.bits[name]).view(np.int16)).view(t.bfloat16).cuda()
    return t.from_numpy(np.ascontiguousarray(arr)).cuda()


def guarded_empty(shape, dtype):
    """A device tensor of `shape` inside a larger buffer with NaN canaries."""
    t = torch()
    n = int(np.prod(shape))
    buf = t.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
    if dtype == t.bfloat16:
        buf.view(t.int16).fill_(0x7FC1)
    else:
        buf.view(t.int32).fill_(0x7FC00001)
    return buf, buf[GUARD:GUARD + n].view(*shape)


def assert_guards(buf):
    t = torch()
    raw = buf.view(t.int16) if buf.dtype == t.bfloat16 else buf.view(t.int32)
    pat = 0x7FC1 if buf.dtype == t.bfloat16 else 0x7FC00001
    head, tail = raw[:GUARD], raw[-GUARD:]
    assert bool((head == pat).all()), "store before the output buffer"
    assert bool((tail == pat).all()), "store after the output buffer"


def as_f64(t_):
    t = torch()
    return t_.detach().to(t.float64).cpu().numpy()


def forward(x: I.Inputs, guard=True, check=True, out_dtype=None):
    """Run fa_fwd on inputs `x`; returns (O, LSE) as float64 numpy arrays.
    O is stored as fp32 unless `out_dtype` says otherwise."""
    t = torch()
    w = x.workload
    q, k, v = to_dev(x, "q"), to_dev(x, "k"), to_dev(x, "v")
    cu = t.from_numpy(x.cu_seqlens).cuda() if w.varlen else None
    slopes = t.from_numpy(x.alibi_slopes).cuda() if x.alibi_slopes is not None else None
    obuf, o = guarded_empty(q.shape, out_dtype or t.float32)
    lbuf, lse = guarded_empty((w.Hq, x.T), t.float32)
    fa.attention_forward(q, k, v, causal=w.causal, scale=x.scale, cu_seqlens=cu,
                         max_seqlen=w.N if w.varlen else None, batch=None if w.varlen else w.B,
                         alibi_slopes=slopes, window=w.window, out=o, lse=lse, check=check)
    t.cuda.synchronize()
    if guard:
        assert_guards(obuf)
        assert_guards(lbuf)
    return as_f64(o), as_f64(lse)


def backward(x: I.Inputs, guard=True, check=True, out_dtype=None, deterministic=False,
             base_workspace=False):
    """Run fa_fwd then fa_bwd; returns float64 numpy (O, LSE, dQ, dK, dV).
    O is stored as fp32 unless `out_dtype` says otherwise.  The workspace is
    the binding's default (fa_bwd_workspace_size_gqa bytes), or exactly
    fa_bwd_workspace_size bytes with `base_workspace` (grouped-query dK/dV
    work then is not split)."""
    t = torch()
    w = x.workload
    q, k, v, do = (to_dev(x, n) for n in ("q", "k", "v", "do"))
    cu = t.from_numpy(x.cu_seqlens).cuda() if w.varlen else None
    slopes = t.from_numpy(x.alibi_slopes).cuda() if x.alibi_slopes is not None else None
    kw = dict(causal=w.causal, scale=x.scale, cu_seqlens=cu, max_seqlen=w.N if w.varlen else None,
              batch=None if w.varlen else w.B, alibi_slopes=slopes, window=w.window, check=check)
    o, lse = fa.attention_forward(q, k, v, out_dtype=out_dtype or t.float32, **kw)
    bufs = [guarded_empty(q.shape, q.dtype), guarded_empty(k.shape, k.dtype),
            guarded_empty(v.shape, v.dtype)]
    ws = None
    if base_workspace:
        ws = t.empty(max(fa.fa_bwd_workspace_size(w.B if not w.varlen else len(x.cu_seqlens) - 1,
                                                  w.Hq, w.N, w.d, x.T), 1),
                     dtype=t.uint8, device="cuda")
    dq, dk, dv = fa.attention_backward(q, k, v, o, do, lse, dq=bufs[0][1], dk=bufs[1][1],
                                       dv=bufs[2][1], deterministic=deterministic, workspace=ws,
                                       **kw)
    t.cuda.synchronize()
    if guard:
        for b, _ in bufs:
            assert_guards(b)
    return as_f64(o), as_f64(lse), as_f64(dq), as_f64(dk), as_f64(dv)


def bits_to_dev(bits: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(t.bfloat16).cuda()


def decode(x: I.DecodeInputs, guard=True, check=True, out_dtype=None, with_seqlens=True):
    """Run fa_decode on inputs `x`; returns (O, LSE) as float64 numpy arrays.
    O is stored as fp32 unless `out_dtype` says otherwise."""
    t = torch()
    w = x.workload
    q, kc, vc = bits_to_dev(x.q_bits), bits_to_dev(x.k_bits), bits_to_dev(x.v_bits)
    cs = t.from_numpy(x.seqlens.astype(np.int32)).cuda() if with_seqlens else None
    slopes = t.from_numpy(x.alibi_slopes).cuda() if x.alibi_slopes is not None else None
    obuf, o = guarded_empty(q.shape, out_dtype or t.float32)
    lbuf, lse = guarded_empty((w.Hq, q.shape[0]), t.float32)
    fa.attention_decode(q, kc, vc, cache_seqlens=cs, q_len=w.q_len, scale=x.scale,
                        alibi_slopes=slopes, window=w.window, out=o, lse=lse, check=check)
    t.cuda.synchronize()
    if guard:
        assert_guards(obuf)
        assert_guards(lbuf)
    return as_f64(o), as_f64(lse)
