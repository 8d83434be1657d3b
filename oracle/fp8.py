"""Oracle of the FP8 forward: incoherent processing, per-block e4m3
quantization, and attention on the quantized values (CPU).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import or run this module.  It
shares no code with the product and depends on NumPy alone (plus this
package's fp64 attention).

Pages followed (cited by title and section):

* [FA1 note] "FlashAttention: Faster Attention Without Dropping a Single
  Interaction": FA3 adaptation (the FP8 path quantizes per block and applies
  the same random orthogonal Hadamard transform M to Q and K, so that
  (QM)(KM)^T = QK^T before quantization) and "Numerical exactness, low
  precision, and reproducibility" (block scales with the incoherent
  transform lower the RMSE against fp64 from 2.4e-2 with one scale per tensor
  to 9.1e-3; the FP8 path is not exact).

Readings (the pages name the steps but fix none of their details):

Q1  M = D H: D = diag(s) with s a random vector of +-1 (an input: the random
    numbers are drawn by the caller) and H the d x d Sylvester Hadamard
    matrix without normalisation, so M M^T = d I and
    (QM)(KM)^T = d QK^T; attention therefore uses S = scale (Q'K'^T) / d.
    The transform is computed in float32 by the iterative butterfly
    (strides 1, 2, 4, ..., d/2; (a, b) -> (a + b, a - b)) after the sign
    flip, because float32 is where the kernel takes it and float32 then
    decides the e4m3 codes (both sides must take that decision alike).
Q2  Blocks are 128 consecutive rows of one head within one sequence (the
    last block of a sequence may be shorter); one scale per block:
    scale = amax / 448 in float32 (448 is e4m3's largest finite value), 1 for
    an all-zero block.  The values are scaled by the block's reciprocal,
    inv = 448 / amax (one float32 division per block, 1 for an all-zero
    block): code = e4m3(x * inv), the product in float32.  (The pages fix no
    detail of the scaling; a multiply by one reciprocal per block is the
    usual way to apply a block scale.)
Q3  e4m3 is the OCP E4M3 format without infinities (bias 7, 3 mantissa bits,
    largest finite 448, smallest subnormal 2^-9); rounding is to nearest,
    ties to even, and values beyond 448 saturate to 448 (the kernel's
    cvt.rn.satfinite).  As in any IEEE-style rounding the sign is kept: a
    negative value that rounds to zero, and -0 itself, give -0 (code 0x80).
Q4  V is quantized per block the same way but not transformed (the pages
    apply M to Q and K only).
Q5  The attention on the quantized values is the exact operator of the FA1
    note (Key design 1) applied to the dequantized Q', K' (with the 1/d of
    Q1) and V; the kernel's further rounding (P to e4m3 inside the tiles,
    fp32 accumulation) is bounded by the tests, not emulated here.
"""
from __future__ import annotations

import numpy as np

from oracle import attention_fp64 as A

E4M3_MAX = 448.0
E4M3_MIN_SUB = 2.0 ** -9
BLOCK = 128

__all__ = ["e4m3_round", "e4m3_bits", "fwht_f32", "quantize_blocks", "quantize_inputs",
           "attention_forward_fp8", "per_tensor_quantized_forward", "rmse"]


def e4m3_round(x):
    """Nearest e4m3 value (ties to even), saturated at +-448 (Q3).  float32 in,
    float32 out; computed exactly in float64."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, E = np.frexp(a)                # a = m 2^E, m in [0.5, 1): floor(log2 a) = E - 1
    e = np.maximum(E.astype(np.float64) - 1.0, -6.0)
    q = np.exp2(e - 3.0)              # quantum: 2^(e - 3) for normals, 2^-9 below 2^-6
    r = np.rint(a / q) * q            # np.rint: round half to even (a / q is exact)
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, x).astype(np.float32)   # the sign survives, zeros too (Q3)


def e4m3_bits(x):
    """uint8 e4m3 codes of values already on the e4m3 grid."""
    x = np.asarray(x, dtype=np.float64)
    s = (np.signbit(x)).astype(np.uint8) << 7
    a = np.abs(x)
    out = np.zeros(x.shape, dtype=np.uint8)
    sub = a < 2.0 ** -6
    out[sub] = np.rint(a[sub] / E4M3_MIN_SUB).astype(np.uint8)
    nz = ~sub
    if nz.any():
        _, E = np.frexp(a[nz])
        e = E.astype(np.float64) - 1.0
        m = np.rint((a[nz] / np.exp2(e) - 1.0) * 8.0)
        out[nz] = ((e + 7).astype(np.uint8) << 3) | m.astype(np.uint8)
    return out | s


def fwht_f32(x):
    """Unnormalised Walsh-Hadamard transform along the last axis in float32,
    by the butterfly of Q1 (Sylvester ordering)."""
    y = np.array(x, dtype=np.float32, copy=True)
    d = y.shape[-1]
    h = 1
    while h < d:
        y = y.reshape(y.shape[:-1] + (d // (2 * h), 2, h))
        a = y[..., 0, :].copy()
        b = y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        y = y.reshape(y.shape[:-3] + (d,))
        h *= 2
    return y


def quantize_blocks(x, cu_seqlens, N):
    """Per-block e4m3 quantization of x [T, H, d] (float32) (Q2, Q3).

    Returns (codes [T, H, d] float32 e4m3 values, scales [H, B * nblk]
    float32) with nblk = ceil(N / 128); block i of sequence b has index
    b * nblk + i (unused entries stay 1)."""
    x = np.asarray(x, dtype=np.float32)
    T, H, d = x.shape
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    B = len(cu) - 1
    nblk = (N + BLOCK - 1) // BLOCK
    codes = np.zeros_like(x)
    scales = np.ones((H, B * nblk), dtype=np.float32)
    for b in range(B):
        s, e = int(cu[b]), int(cu[b + 1])
        for i, r0 in enumerate(range(s, e, BLOCK)):
            r1 = min(r0 + BLOCK, e)
            blk = x[r0:r1]                                      # [rows, H, d]
            amax = np.abs(blk).max(axis=(0, 2)).astype(np.float32)
            pos = amax > 0
            safe = np.where(pos, amax, np.float32(1.0)).astype(np.float32)
            sc = np.where(pos, safe / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
            inv = np.where(pos, np.float32(E4M3_MAX) / safe, np.float32(1.0)).astype(np.float32)
            codes[r0:r1] = e4m3_round((blk * inv[None, :, None]).astype(np.float32))
            scales[:, b * nblk + i] = sc
    return codes, scales


def quantize_inputs(q, k, v, signs, cu_seqlens, N):
    """Incoherent processing and block quantization of Q, K, V (Q1-Q4).
    Returns a dict of codes (float32 e4m3 values) and scales."""
    s = np.asarray(signs, dtype=np.float32)
    qt = fwht_f32(np.asarray(q, dtype=np.float32) * s)
    kt = fwht_f32(np.asarray(k, dtype=np.float32) * s)
    q8, qs = quantize_blocks(qt, cu_seqlens, N)
    k8, ks = quantize_blocks(kt, cu_seqlens, N)
    v8, vs = quantize_blocks(v, cu_seqlens, N)
    return {"q8": q8, "q_scale": qs, "k8": k8, "k_scale": ks, "v8": v8, "v_scale": vs,
            "q_t": qt, "k_t": kt}


def _dequant(codes, scales, cu_seqlens, N):
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    nblk = (N + BLOCK - 1) // BLOCK
    out = np.asarray(codes, dtype=np.float64).copy()
    for b in range(len(cu) - 1):
        s, e = int(cu[b]), int(cu[b + 1])
        for i, r0 in enumerate(range(s, e, BLOCK)):
            out[r0:min(r0 + BLOCK, e)] *= scales[:, b * nblk + i][None, :, None].astype(np.float64)
    return out


def attention_forward_fp8(qz, cu_seqlens, N, scale, causal, alibi_slopes=None, window=None):
    """O and LSE of attention on the dequantized inputs (Q5): Q' and K' carry
    the transform, so the scores use scale / d (Q1)."""
    q = _dequant(qz["q8"], qz["q_scale"], cu_seqlens, N)
    k = _dequant(qz["k8"], qz["k_scale"], cu_seqlens, N)
    v = _dequant(qz["v8"], qz["v_scale"], cu_seqlens, N)
    d = q.shape[2]
    return A.attention_forward(q, k, v, scale / d, causal, cu_seqlens, alibi_slopes, window=window)


def per_tensor_quantized_forward(q, k, v, cu_seqlens, scale, causal):
    """The pages' baseline: one scale per tensor, no transform; attention on
    the dequantized values."""
    def one(x):
        x = np.asarray(x, dtype=np.float32)
        sc = np.float32(np.abs(x).max()) / np.float32(E4M3_MAX)
        return e4m3_round((x / sc).astype(np.float32)).astype(np.float64) * float(sc)
    return A.attention_forward(one(q), one(k), one(v), scale, causal, cu_seqlens)


def rmse(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.sqrt(np.mean((a - b) ** 2)))
