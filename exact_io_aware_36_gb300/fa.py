"""Thin ctypes binding of libfa (include/fa.h).

Only argument marshalling happens here: torch tensors become device pointers
and the current CUDA stream becomes a ``cudaStream_t``.  Every step of the
attention computation runs in the library's CUDA kernels.  There is no other
implementation behind these functions: if the library is missing or fails
to load, the calls raise.

Raw entry points with the C names (``fa_fwd``, ``fa_bwd``,
``fa_bwd_workspace_size``, ``fa_check_device_error``, ``fa_status_string``)
take integer pointers; ``attention_forward`` / ``attention_backward`` take
torch tensors and allocate the outputs with torch.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libfa.so")

FA_BF16, FA_FP32 = 0, 1
STATUS = {
    0: "FA_OK", 1: "FA_ERR_NULL", 2: "FA_ERR_SHAPE", 3: "FA_ERR_UNSUPPORTED", 4: "FA_ERR_ALIGN",
    5: "FA_ERR_WORKSPACE", 6: "FA_ERR_CUDA", 7: "FA_ERR_DEVICE_TIMEOUT", 8: "FA_ERR_CU_SEQLENS",
}
EXPORTS = ("fa_fwd", "fa_bwd", "fa_bwd_stage", "fa_bwd_workspace_size", "fa_check_device_error",
           "fa_status_string", "fa_version", "fa_bwd_static_scratch", "fa_selftest_wait_timeout",
           "fa_decode", "fa_decode_workspace_size", "fa_fp8_layout_get", "fa_fp8_quantize",
           "fa_fwd_fp8", "fa_host_cache_stats", "fa_bwd_workspace_size_gqa", "fa_bwd_dkdv_split")
FA_BWD_PREPROCESS, FA_BWD_DKDV, FA_BWD_DQ_CONVERT = 0, 1, 2


class FAError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        name = STATUS.get(status, str(status))
        msg = f"{what}: {name}" if what else name
        try:
            msg += f" ({fa_status_string(status)})"
        except Exception:
            pass
        super().__init__(msg)


_lib = None


class FP8Layout(ctypes.Structure):
    """fa_fp8_layout: byte offsets of the FP8 codes and scales in one buffer."""
    _fields_ = [("q8", ctypes.c_size_t), ("k8", ctypes.c_size_t), ("v8t", ctypes.c_size_t),
                ("q_scale", ctypes.c_size_t), ("k_scale", ctypes.c_size_t),
                ("v_scale", ctypes.c_size_t), ("v_scale_max", ctypes.c_size_t),
                ("total", ctypes.c_size_t), ("nblk", ctypes.c_int)]


def load(path: Optional[str] = None):
    """Load libfa (once) and declare the C signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise FAError(6, f"libfa not built ({p} missing); run exact_io_aware_36_gb300.build")
    lib = ctypes.CDLL(p)
    vp, i, f, ll, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong, ctypes.c_size_t
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, ll, vp, i, i, vp]
    lib.fa_fwd.restype = i
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, ll, vp,
                           i, i, i, vp, sz, vp]
    lib.fa_bwd.restype = i
    lib.fa_bwd_stage.argtypes = [i] + lib.fa_bwd.argtypes
    lib.fa_bwd_stage.restype = i
    lib.fa_bwd_workspace_size.argtypes = [i, i, i, i, ll]
    lib.fa_bwd_workspace_size.restype = sz
    lib.fa_bwd_workspace_size_gqa.argtypes = [i, i, i, i, i, ll]
    lib.fa_bwd_workspace_size_gqa.restype = sz
    lib.fa_decode_workspace_size.argtypes = [i, i, i, i, i, i]
    lib.fa_decode_workspace_size.restype = sz
    lib.fa_decode.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, i, vp, sz, vp]
    lib.fa_decode.restype = i
    lib.fa_fp8_layout_get.argtypes = [i, i, i, i, i, ll, ctypes.POINTER(FP8Layout)]
    lib.fa_fp8_layout_get.restype = i
    lib.fa_fp8_quantize.argtypes = [vp, vp, vp, vp, i, i, i, i, i, vp, ll, vp, sz, vp]
    lib.fa_fp8_quantize.restype = i
    lib.fa_fwd_fp8.argtypes = [vp, sz, vp, vp, i, i, i, i, i, f, i, i, vp, ll, vp, i, vp]
    lib.fa_fwd_fp8.restype = i
    lib.fa_check_device_error.argtypes = [vp]
    lib.fa_check_device_error.restype = i
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_version.argtypes = []
    lib.fa_version.restype = i
    if path is None:
        _lib = lib
    return lib


# ------------------------------------------------------------ raw C entry points

def fa_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, causal, window, cu_seqlens, total_tokens,
           alibi_slopes, dtype, o_dtype, stream) -> int:
    return load().fa_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, int(causal), int(window),
                         cu_seqlens, total_tokens, alibi_slopes, dtype, o_dtype, stream)


def fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, causal, window, cu_seqlens,
           total_tokens, alibi_slopes, dtype, o_dtype, deterministic, workspace, workspace_bytes,
           stream) -> int:
    return load().fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, int(causal),
                         int(window), cu_seqlens, total_tokens, alibi_slopes, dtype, o_dtype,
                         int(deterministic), workspace, workspace_bytes, stream)


def fa_bwd_stage(stage, q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, causal, window,
                 cu_seqlens, total_tokens, alibi_slopes, dtype, o_dtype, deterministic, workspace,
                 workspace_bytes, stream) -> int:
    return load().fa_bwd_stage(stage, q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale,
                               int(causal), int(window), cu_seqlens, total_tokens, alibi_slopes,
                               dtype, o_dtype, int(deterministic), workspace, workspace_bytes,
                               stream)


FA_BWD_STATIC_SCRATCH_BYTES = 64 << 20


def fa_bwd_static_scratch(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, causal,
                          window, cu_seqlens, total_tokens, alibi_slopes, dtype, o_dtype,
                          deterministic, stream) -> int:
    """fa_bwd without a workspace argument, for callers that cannot allocate
    device memory: the scratch lives in a fixed array of
    FA_BWD_STATIC_SCRATCH_BYTES inside the library (see include/fa.h)."""
    lib = load()
    fn = lib.fa_bwd_static_scratch
    if fn.restype is not ctypes.c_int or not fn.argtypes:
        fn.argtypes = lib.fa_bwd.argtypes[:23] + [ctypes.c_void_p]
        fn.restype = ctypes.c_int
    return fn(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, int(causal), int(window),
              cu_seqlens, total_tokens, alibi_slopes, dtype, o_dtype, int(deterministic), stream)


def fa_decode_workspace_size(B, Hq, Hkv, S_max, q_len, d) -> int:
    return load().fa_decode_workspace_size(B, Hq, Hkv, S_max, q_len, d)


def fa_decode(q, k_cache, v_cache, cache_seqlens, o, lse, B, Hq, Hkv, S_max, q_len, d, scale,
              window, alibi_slopes, o_dtype, workspace, workspace_bytes, stream) -> int:
    return load().fa_decode(q, k_cache, v_cache, cache_seqlens, o, lse, B, Hq, Hkv, S_max, q_len,
                            d, scale, int(window), alibi_slopes, o_dtype, workspace,
                            workspace_bytes, stream)


def fa_fp8_layout_get(B, Hq, Hkv, N, d, total_tokens):
    """(status, FP8Layout)."""
    lay = FP8Layout()
    st = load().fa_fp8_layout_get(B, Hq, Hkv, N, d, total_tokens, ctypes.byref(lay))
    return st, lay


def fa_fp8_quantize(q, k, v, signs, B, Hq, Hkv, N, d, cu_seqlens, total_tokens, fp8_buf,
                    fp8_bytes, stream) -> int:
    return load().fa_fp8_quantize(q, k, v, signs, B, Hq, Hkv, N, d, cu_seqlens, total_tokens,
                                  fp8_buf, fp8_bytes, stream)


def fa_fwd_fp8(fp8_buf, fp8_bytes, o, lse, B, Hq, Hkv, N, d, scale, causal, window, cu_seqlens,
               total_tokens, alibi_slopes, o_dtype, stream) -> int:
    return load().fa_fwd_fp8(fp8_buf, fp8_bytes, o, lse, B, Hq, Hkv, N, d, scale, int(causal),
                             int(window), cu_seqlens, total_tokens, alibi_slopes, o_dtype, stream)


def fa_bwd_workspace_size(B, Hq, N, d, total_tokens) -> int:
    return load().fa_bwd_workspace_size(B, Hq, N, d, total_tokens)


def fa_bwd_workspace_size_gqa(B, Hq, Hkv, N, d, total_tokens) -> int:
    return load().fa_bwd_workspace_size_gqa(B, Hq, Hkv, N, d, total_tokens)


def fa_bwd_dkdv_split(B, Hq, Hkv, N, d, causal, window, cu_seqlens, workspace_bytes) -> int:
    lib = load()
    fn = lib.fa_bwd_dkdv_split
    fn.argtypes = [ctypes.c_int] * 7 + [ctypes.c_void_p, ctypes.c_size_t]
    fn.restype = ctypes.c_int
    return fn(B, Hq, Hkv, N, d, int(causal), int(window), cu_seqlens, workspace_bytes)


def fa_selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    """Launch one block whose bounded wait can never complete (see fa.h)."""
    lib = load()
    fn = lib.fa_selftest_wait_timeout
    fn.argtypes = [ctypes.c_ulonglong, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn(limit_ns, stream)


def fa_host_cache_stats():
    """(descriptors encoded, descriptors reused, shared-memory limits set)."""
    lib = load()
    fn = lib.fa_host_cache_stats
    u = ctypes.c_ulonglong
    fn.argtypes = [ctypes.POINTER(u)] * 3
    fn.restype = None
    a, b, c = u(), u(), u()
    fn(ctypes.byref(a), ctypes.byref(b), ctypes.byref(c))
    return a.value, b.value, c.value


def fa_check_device_error(stream=None) -> int:
    return load().fa_check_device_error(stream)


def fa_status_string(status: int) -> str:
    return load().fa_status_string(status).decode()


# ------------------------------------------------------------ torch wrappers

def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(status: int, what: str):
    if status != 0:
        raise FAError(status, what)


def _sizes(q, k, cu_seqlens, max_seqlen, batch):
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    if cu_seqlens is not None:
        B = cu_seqlens.numel() - 1
        if max_seqlen is None:
            raise ValueError("max_seqlen is required with cu_seqlens")
        N = int(max_seqlen)
    else:
        B = int(batch) if batch is not None else 1
        N = T // B if B else 0
    return T, B, Hq, Hkv, N, d


def _dtype_code(dt):
    import torch
    return FA_BF16 if dt == torch.bfloat16 else FA_FP32 if dt == torch.float32 else -1


def attention_forward(q, k, v, *, causal: bool, scale: Optional[float] = None, cu_seqlens=None,
                      max_seqlen: Optional[int] = None, batch: Optional[int] = None,
                      alibi_slopes=None, window: Optional[int] = None, out=None, lse=None,
                      out_dtype=None, stream=None, check: bool = False):
    """O, LSE = attention(q, k, v) through ``fa_fwd``.

    q: [T, Hq, d], k/v: [T, Hkv, d] (bf16 or fp32, contiguous, on the GPU).
    Dense batches pass ``batch`` (T = batch * N); packed batches pass int32
    ``cu_seqlens`` [B+1] and ``max_seqlen``.  Returns (o [T, Hq, d] of
    ``out_dtype`` (default: ``out``'s dtype, else q's), lse float32 [Hq, T]).
    ``window`` w (causal only): query i sees keys i - w .. i; None: no window.
    """
    import torch
    T, B, Hq, Hkv, N, d = _sizes(q, k, cu_seqlens, max_seqlen, batch)
    dtype = _dtype_code(q.dtype)
    if dtype < 0:
        raise TypeError(f"unsupported dtype {q.dtype}")
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype or q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    st = fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, N, d, float(scale),
                causal, -1 if window is None else window, _ptr(cu_seqlens), T,
                _ptr(alibi_slopes), dtype, _dtype_code(out.dtype), _stream(stream))
    _check(st, "fa_fwd")
    if check:
        _check(fa_check_device_error(_stream(stream)), "fa_fwd (device)")
    return out, lse


def attention_backward(q, k, v, o, dO, lse, *, causal: bool, scale: Optional[float] = None,
                       cu_seqlens=None, max_seqlen: Optional[int] = None,
                       batch: Optional[int] = None, alibi_slopes=None,
                       window: Optional[int] = None, deterministic: bool = False,
                       workspace=None, dq=None, dk=None, dv=None, stream=None,
                       check: bool = False):
    """dQ, dK, dV through ``fa_bwd`` (bf16).  ``workspace`` (uint8 device
    tensor of at least ``fa_bwd_workspace_size`` bytes; the default is
    ``fa_bwd_workspace_size_gqa``'s size, which lets grouped-query problems
    split their dK/dV work) is allocated when not given.  ``window`` as in attention_forward; ``deterministic`` selects
    the backward whose results do not vary from run to run."""
    import torch
    T, B, Hq, Hkv, N, d = _sizes(q, k, cu_seqlens, max_seqlen, batch)
    if q.dtype != torch.bfloat16:
        raise TypeError("fa_bwd takes bf16 tensors")
    if scale is None:
        scale = d ** -0.5
    need = fa_bwd_workspace_size_gqa(B, Hq, Hkv, N, d, T)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    st = fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk),
                _ptr(dv), B, Hq, Hkv, N, d, float(scale), causal,
                -1 if window is None else window, _ptr(cu_seqlens), T, _ptr(alibi_slopes),
                FA_BF16, _dtype_code(o.dtype), deterministic, _ptr(workspace),
                workspace.numel(), _stream(stream))
    _check(st, "fa_bwd")
    if check:
        _check(fa_check_device_error(_stream(stream)), "fa_bwd (device)")
    return dq, dk, dv


def attention_decode(q, k_cache, v_cache, *, cache_seqlens=None, q_len: int = 1,
                     scale: Optional[float] = None, alibi_slopes=None,
                     window: Optional[int] = None, out=None, lse=None, out_dtype=None,
                     workspace=None, stream=None, check: bool = False):
    """O, LSE of the q_len newest tokens of each sequence through ``fa_decode``.

    q: bf16 [B * q_len, Hq, d]; k_cache, v_cache: bf16 [B, S_max, Hkv, d];
    cache_seqlens: int32 [B] on the GPU (None: every cache holds S_max).
    Returns (o [B * q_len, Hq, d] of ``out_dtype`` (default fp32), lse
    float32 [Hq, B * q_len]).
    """
    import torch
    B, S_max, Hkv, d = k_cache.shape
    Hq = q.shape[1]
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype or torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((Hq, q.shape[0]), dtype=torch.float32, device=q.device)
    need = fa_decode_workspace_size(B, Hq, Hkv, S_max, q_len, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = fa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cache_seqlens), _ptr(out), _ptr(lse),
                   B, Hq, Hkv, S_max, q_len, d, float(scale), -1 if window is None else window,
                   _ptr(alibi_slopes), _dtype_code(out.dtype), _ptr(workspace), workspace.numel(),
                   _stream(stream))
    _check(st, "fa_decode")
    if check:
        _check(fa_check_device_error(_stream(stream)), "fa_decode (device)")
    return out, lse


def attention_forward_fp8(q, k, v, signs, *, causal: bool, scale: Optional[float] = None,
                          cu_seqlens=None, max_seqlen: Optional[int] = None,
                          batch: Optional[int] = None, alibi_slopes=None,
                          window: Optional[int] = None, out=None, lse=None, out_dtype=None,
                          fp8_buf=None, stream=None, check: bool = False):
    """O, LSE through ``fa_fp8_quantize`` and ``fa_fwd_fp8`` (d = 128).

    q: bf16 [T, Hq, 128], k/v: bf16 [T, Hkv, 128]; signs: float32 [128] of
    +-1 on the GPU.  Returns (o, lse, fp8_buf, layout): the buffer holds the
    codes and scales at the layout's offsets.
    """
    import torch
    T, B, Hq, Hkv, N, d = _sizes(q, k, cu_seqlens, max_seqlen, batch)
    if scale is None:
        scale = d ** -0.5
    st, lay = fa_fp8_layout_get(B, Hq, Hkv, N, d, T if cu_seqlens is not None else 0)
    _check(st, "fa_fp8_layout_get")
    if fp8_buf is None:
        fp8_buf = torch.empty(max(lay.total, 1), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype or torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    sp = _stream(stream)
    _check(fa_fp8_quantize(_ptr(q), _ptr(k), _ptr(v), _ptr(signs), B, Hq, Hkv, N, d,
                           _ptr(cu_seqlens), T, _ptr(fp8_buf), fp8_buf.numel(), sp), "fa_fp8_quantize")
    _check(fa_fwd_fp8(_ptr(fp8_buf), fp8_buf.numel(), _ptr(out), _ptr(lse), B, Hq, Hkv, N, d,
                      float(scale), causal, -1 if window is None else window, _ptr(cu_seqlens), T,
                      _ptr(alibi_slopes), _dtype_code(out.dtype), sp), "fa_fwd_fp8")
    if check:
        _check(fa_check_device_error(sp), "fa_fwd_fp8 (device)")
    return out, lse, fp8_buf, lay
