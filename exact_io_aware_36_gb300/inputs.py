"""Seeded synthetic workloads for exact attention.

This module only draws random numbers, rounds them to the storage type and
packs sequences.  It holds none of the attention arithmetic, so both the CUDA
path and the fp64 oracle can take their inputs from here without sharing any
of the method.

Shapes follow the token-major layout of the FlashAttention user API
("FlashAttention: Faster Attention Without Dropping a Single Interaction",
Usage contract: ``flash_attn_func(q, k, v, dropout_p, softmax_scale, causal)``
with scale, causal flag and Q/KV lengths):

* ``q``, ``do``: ``[T, Hq, d]``; ``k``, ``v``: ``[T, Hkv, d]``; ``T`` the total
  token count (``B * N`` dense, ``cu_seqlens[B]`` packed).
* ``cu_seqlens``: int32 ``[B + 1]`` prefix sums of the sequence lengths, the
  packed ("varlen") layout of "FlashAttention: The Algorithm That Beat the
  Memory Wall", section "Varlen Is the Quiet Superpower".
* ``alibi_slopes``: fp32 ``[Hq]``, slope of query head ``h`` (1-indexed)
  ``2**(-8 h / Hq)``.

Draw recipe (one fresh ``numpy.random.Generator(PCG64(seed))`` per workload):
sequence lengths first (packed workloads only, ``integers(lo, hi + 1)``),
then ``q, k, v, do`` as ``standard_normal(dtype=float32)`` in that order;
``qk_gain`` multiplies q and k after the draw; bf16 workloads round every
tensor to bf16 with round-to-nearest-even.  The fp32 arrays returned for bf16
workloads hold exactly the bf16 values, so an fp64 upcast sees the same
numbers the GPU sees.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "EXTRA_WORKLOADS", "workload", "make_inputs", "small_case",
    "bf16_round", "bf16_bits", "bf16_from_bits", "alibi_slopes",
    "attended_pairs", "DecodeWorkload", "DECODE_WORKLOADS", "DecodeInputs",
    "make_decode_inputs", "decode_bytes", "hadamard_signs", "add_score_structure",
]


@dataclass(frozen=True)
class Workload:
    """One synthetic attention problem.

    ``N`` is the sequence length of dense workloads and the maximum length of
    packed ones.  ``seqlen_range`` makes the workload packed: ``B`` lengths are
    drawn uniformly from the closed range.
    """
    name: str
    dtype: str                 # "bf16" or "fp32": storage / MMA operand type
    causal: bool
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    backward: bool = True
    alibi: bool = False
    qk_gain: float = 1.0
    seqlen_range: Optional[tuple] = None
    seqlens: Optional[tuple] = None   # explicit packed lengths (tests)
    note: str = ""
    window: Optional[int] = None      # causal band: query i sees keys i-window .. i

    @property
    def window_arg(self) -> int:
        """The C ABI's window argument (-1: none)."""
        return -1 if self.window is None else int(self.window)

    @property
    def varlen(self) -> bool:
        return self.seqlen_range is not None or self.seqlens is not None

    @property
    def scale(self) -> float:
        return float(1.0 / np.sqrt(self.d))


# The five workloads the build is measured and checked on.
WORKLOADS = {
    "c1_fp32_fwd": Workload(
        "c1_fp32_fwd", "fp32", causal=False, B=1, Hq=1, Hkv=1, N=128, d=64,
        backward=False, note="fp32 forward only, non-causal, B=1 H=1 N=128 d=64"),
    "c2_gpt2m": Workload(
        "c2_gpt2m", "bf16", causal=True, B=8, Hq=16, Hkv=16, N=1024, d=64,
        note="GPT-2-medium attention shape, causal, B=8 H=16 N=1024 d=64"),
    "c3_long": Workload(
        "c3_long", "bf16", causal=True, B=1, Hq=32, Hkv=32, N=16384, d=128,
        qk_gain=0.5, note="long-context causal, B=1 H=32 N=16384 d=128, q,k x0.5"),
    "c4_varlen": Workload(
        "c4_varlen", "bf16", causal=True, B=64, Hq=32, Hkv=32, N=4096, d=128,
        seqlen_range=(128, 4096),
        note="64 packed sequences, lengths U[128,4096], causal, H=32 d=128"),
    "c5_gqa_alibi": Workload(
        "c5_gqa_alibi", "bf16", causal=True, B=2, Hq=32, Hkv=4, N=8192, d=128,
        alibi=True, note="GQA 32/4 with ALiBi, causal, B=2 N=8192 d=128"),
}

# Further workloads for the rows beyond the five above: each is checked and
# measured the same way but is not one of the five.
EXTRA_WORKLOADS = {
    "b4_n4096": Workload(
        "b4_n4096", "bf16", causal=True, B=4, Hq=32, Hkv=32, N=4096, d=128,
        note="causal, B=4 H=32 N=4096 d=128 (dense batch of the persistent forward's size)"),
    "swa_32k": Workload(
        "swa_32k", "bf16", causal=True, B=1, Hq=32, Hkv=8, N=32768, d=128, window=4095,
        note="sliding window 4096 keys (causal band), GQA 32/8, B=1 N=32768 d=128"),
}


def workload(name: str) -> Workload:
    return WORKLOADS[name] if name in WORKLOADS else EXTRA_WORKLOADS[name]


def small_case(dtype="bf16", causal=True, B=1, Hq=2, Hkv=2, N=128, d=64,
               alibi=False, seqlens=None, qk_gain=1.0, backward=True,
               name="small", window=None) -> Workload:
    """A small workload for parity tests (explicit packed lengths allowed)."""
    if seqlens is not None:
        seqlens = tuple(int(x) for x in seqlens)
        B = len(seqlens)
        N = max(seqlens) if seqlens else 0
    return Workload(name, dtype, causal, B, Hq, Hkv, N, d, backward=backward,
                    alibi=alibi, qk_gain=qk_gain, seqlens=seqlens, window=window)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of float32 ``x`` with round-to-nearest-even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    out = ((u + rounding) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_from_bits(b: np.ndarray) -> np.ndarray:
    """float32 values of bf16 bit patterns (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_round(x: np.ndarray) -> np.ndarray:
    return bf16_from_bits(bf16_bits(x))


def alibi_slopes(Hq: int) -> np.ndarray:
    """ALiBi slope of each query head: 2**(-8 h / Hq) for h = 1..Hq."""
    h = np.arange(1, Hq + 1, dtype=np.float64)
    return np.exp2(-8.0 * h / Hq).astype(np.float32)


def _seqlens(w: Workload, rng: np.random.Generator) -> np.ndarray:
    if w.seqlens is not None:
        return np.asarray(w.seqlens, dtype=np.int64)
    if w.seqlen_range is not None:
        lo, hi = w.seqlen_range
        return rng.integers(lo, hi + 1, size=w.B).astype(np.int64)
    return np.full(w.B, w.N, dtype=np.int64)


def attended_pairs(w: Workload, seqlens=None) -> int:
    """Number of (query, key) pairs the workload attends, over heads and sequences.

    Causal: L(L+1)/2 per sequence and query head; otherwise L*L.  With a
    window w, query i attends min(i, w) + 1 keys: the band's area is
    (w+1)(w+2)/2 + (L-w-1)(w+1) once L > w + 1.
    """
    if seqlens is None:
        seqlens = make_seqlens(w)
    L = np.asarray(seqlens, dtype=np.int64)
    per = L * (L + 1) // 2 if w.causal else L * L
    if w.causal and w.window is not None and w.window >= 0:
        b = np.int64(w.window) + 1
        per = np.where(L > b, b * (b + 1) // 2 + (L - b) * b, per)
    return int(per.sum()) * w.Hq


def make_seqlens(w: Workload, seed: int = 0) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    return _seqlens(w, rng)


@dataclass
class Inputs:
    workload: Workload
    seed: int
    seqlens: np.ndarray
    cu_seqlens: np.ndarray          # int32 [B+1]
    q: np.ndarray                   # float32 [T, Hq, d] (bf16-exact for bf16)
    k: np.ndarray                   # float32 [T, Hkv, d]
    v: np.ndarray
    do: Optional[np.ndarray]        # float32 [T, Hq, d]
    alibi_slopes: Optional[np.ndarray]
    scale: float
    bits: dict = field(default_factory=dict)   # bf16 bit patterns (uint16)

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])


def make_inputs(w: Workload, seed: int = 0, with_do: Optional[bool] = None) -> Inputs:
    """Draw the inputs of workload ``w`` following the recipe in the module doc."""
    rng = np.random.Generator(np.random.PCG64(seed))
    L = _seqlens(w, rng)
    cu = np.zeros(len(L) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(L)
    T = int(cu[-1])
    if with_do is None:
        with_do = w.backward

    def draw(H):
        x = rng.standard_normal(size=(T, H, w.d), dtype=np.float32)
        return x

    q = draw(w.Hq)
    k = draw(w.Hkv)
    v = draw(w.Hkv)
    do = draw(w.Hq) if with_do else None
    if w.qk_gain != 1.0:
        q *= np.float32(w.qk_gain)
        k *= np.float32(w.qk_gain)
    bits = {}
    if w.dtype == "bf16":
        for name, x in (("q", q), ("k", k), ("v", v), ("do", do)):
            if x is None:
                continue
            b = bf16_bits(x)
            bits[name] = b
            x[...] = bf16_from_bits(b)
    slopes = alibi_slopes(w.Hq) if w.alibi else None
    return Inputs(w, seed, L, cu.astype(np.int32), q, k, v, do, slopes, w.scale, bits)


# Dominant keys of the "late_dominant" structure: offsets within each
# sequence (the second, fourth and sixth 128-key tiles) and the score each
# adds, as a multiple of the structure's strength.
_DOMINANT_AT = ((128 + 37, 1.0), (384 + 5, 2.0), (640 + 90, 3.0))


def add_score_structure(x: Inputs, kind: str, strength: float, seed: int = 0) -> Inputs:
    """Overlay a peaked or drifting score pattern on drawn inputs, in place.

    The softmax regimes these produce are the ones where the running maximum
    of a row changes by many nats between key tiles.  One direction u_g per
    kv head is drawn (``standard_normal``, rescaled to |u_g|^2 = d) from a
    fresh PCG64(seed) generator; every query row of a head of g's group gets
    + u_g, and keys get + c u_g, which adds c * scale * d to their scores
    against every query row (c is chosen so that this is ``strength`` nats
    times the pattern's profile):

    * ``"late_dominant"``: the keys at offsets 165, 389 and 730 of each
      sequence (second, fourth and sixth 128-key tile, where the sequence is
      long enough) get 1, 2 and 3 x strength: rows past them see their
      maximum jump up at those tiles.
    * ``"rising"``: key j of a sequence of length L gets strength * j / L.
    * ``"falling"``: key j gets strength * (1 - j / L).

    q and k are then rounded to the storage type again (bf16 workloads keep
    their bit patterns in ``x.bits``).  Nothing of the attention arithmetic
    is computed here: the pattern is an input.
    """
    w = x.workload
    rng = np.random.Generator(np.random.PCG64(seed))
    u = rng.standard_normal(size=(w.Hkv, w.d)).astype(np.float64)
    u *= np.sqrt(w.d) / np.linalg.norm(u, axis=1, keepdims=True)
    group = w.Hq // w.Hkv
    unit = 1.0 / (x.scale * w.d)          # key coefficient that adds one nat
    q = x.q.astype(np.float64)
    k = x.k.astype(np.float64)
    q += np.repeat(u, group, axis=0)[None, :, :]
    cu = x.cu_seqlens.astype(np.int64)
    for b in range(len(cu) - 1):
        s, e = int(cu[b]), int(cu[b + 1])
        L = e - s
        if L == 0:
            continue
        if kind == "late_dominant":
            prof = np.zeros(L)
            for off, mult in _DOMINANT_AT:
                if off < L:
                    prof[off] = mult
        elif kind == "rising":
            prof = np.arange(L) / L
        elif kind == "falling":
            prof = 1.0 - np.arange(L) / L
        else:
            raise ValueError(f"unknown structure {kind!r}")
        k[s:e] += (strength * unit * prof)[:, None, None] * u[None, :, :]
    for name, arr in (("q", q), ("k", k)):
        f32 = arr.astype(np.float32)
        if w.dtype == "bf16":
            x.bits[name] = bf16_bits(f32)
            f32 = bf16_from_bits(x.bits[name])
        getattr(x, name)[...] = f32
    return x


def with_seqlens(w: Workload, seqlens) -> Workload:
    return replace(w, seqlens=tuple(int(x) for x in seqlens), B=len(seqlens),
                   N=int(max(seqlens)), seqlen_range=None)


# --------------------------------------------------------------------------
# Decode over a KV cache: the q_len newest tokens of B sequences against
# their caches [B, S_max, Hkv, d] of cache_seqlens[b] tokens.
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class DecodeWorkload:
    """One synthetic decode step.  Cache lengths are drawn uniformly from
    ``len_range`` (closed), or given as ``lens``; ``S_max`` is the cache
    capacity per sequence."""
    name: str
    B: int
    Hq: int
    Hkv: int
    S_max: int
    d: int
    q_len: int = 1
    len_range: Optional[tuple] = None
    lens: Optional[tuple] = None
    alibi: bool = False
    window: Optional[int] = None
    note: str = ""

    @property
    def scale(self) -> float:
        return float(1.0 / np.sqrt(self.d))

    @property
    def window_arg(self) -> int:
        return -1 if self.window is None else int(self.window)


DECODE_WORKLOADS = {
    "decode_gqa": DecodeWorkload(
        "decode_gqa", B=16, Hq=32, Hkv=8, S_max=32768, d=128, q_len=1, len_range=(1024, 32768),
        note="decode step: 16 sequences, caches U[1024, 32768] tokens, GQA 32/8, d=128, bf16"),
}


@dataclass
class DecodeInputs:
    workload: DecodeWorkload
    seed: int
    seqlens: np.ndarray             # int32 [B]
    q: np.ndarray                   # float32 [B * q_len, Hq, d], bf16-exact
    q_bits: np.ndarray              # uint16, same shape
    k_bits: np.ndarray              # uint16 [B, S_max, Hkv, d]
    v_bits: np.ndarray
    alibi_slopes: Optional[np.ndarray]
    scale: float

    def cache(self, name: str, seqs=None) -> np.ndarray:
        """float32 copy of the k or v cache (bf16-exact), of the sequences
        ``seqs`` (all when None)."""
        bits = self.k_bits if name == "k" else self.v_bits
        return bf16_from_bits(bits if seqs is None else bits[list(seqs)])


def make_decode_inputs(w: DecodeWorkload, seed: int = 0) -> DecodeInputs:
    """Draw a decode step: lengths first (when drawn), then q, then the k and v
    caches one sequence at a time, all ``standard_normal(float32)`` rounded to
    bf16.  Cache slots at or past a sequence's length hold drawn values that
    attention never reads."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if w.lens is not None:
        lens = np.asarray(w.lens, dtype=np.int64)
    elif w.len_range is not None:
        lo, hi = w.len_range
        lens = rng.integers(lo, hi + 1, size=w.B).astype(np.int64)
    else:
        lens = np.full(w.B, w.S_max, dtype=np.int64)
    q = rng.standard_normal(size=(w.B * w.q_len, w.Hq, w.d), dtype=np.float32)
    q_bits = bf16_bits(q)
    q = bf16_from_bits(q_bits)
    caches = []
    for _ in ("k", "v"):
        bits = np.empty((w.B, w.S_max, w.Hkv, w.d), dtype=np.uint16)
        for b in range(w.B):
            bits[b] = bf16_bits(rng.standard_normal(size=(w.S_max, w.Hkv, w.d), dtype=np.float32))
        caches.append(bits)
    slopes = alibi_slopes(w.Hq) if w.alibi else None
    return DecodeInputs(w, seed, lens.astype(np.int32), q, q_bits, caches[0], caches[1], slopes,
                        w.scale)


def decode_bytes(w: DecodeWorkload, seqlens) -> int:
    """HBM bytes one decode step must move: every cached key and value read
    once (bf16), q read (bf16), O written (fp32) and LSE written."""
    L = np.asarray(seqlens, dtype=np.int64)
    kv = int(L.sum()) * w.Hkv * w.d * 2 * 2
    rows = w.B * w.q_len * w.Hq
    return kv + rows * w.d * 2 + rows * w.d * 4 + rows * 4


def hadamard_signs(d: int, seed: int = 0) -> np.ndarray:
    """The random diagonal of the FP8 path's transform: float32 [d] of +-1,
    from its own PCG64(seed) generator (one uniform draw per entry)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.where(rng.random(d) < 0.5, -1.0, 1.0).astype(np.float32)
