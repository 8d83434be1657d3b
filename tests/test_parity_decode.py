"""Decode over a KV cache: the CUDA path against the fp64 oracle (GPU).

The q_len newest tokens of each sequence attend to its cache (reading R10 of
the oracle).  Tolerances as for the forward: O max abs error <= 1e-2 (O stored
fp32; the kernel keeps P in fp32, so the error is far below that), LSE <= 1e-3.
Cases cover GQA groups of 1-16 rows per kv head, q_len 1-4, cache lengths at
and around the 64-key tiles and the chunk edges (small batches use 64-key
chunks, so a cache is merged from many partial states), ALiBi, windows, bf16
output, and caches given without lengths.
"""
import numpy as np
import pytest

from oracle import attention_fp64 as A
from exact_io_aware_36_gb300 import inputs as I
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE = 1e-2, 1e-3


def _oracle(x, seqs=None):
    w = x.workload
    seqs = list(range(w.B)) if seqs is None else list(seqs)
    rows = np.concatenate([np.arange(b * w.q_len, (b + 1) * w.q_len) for b in seqs])
    return A.decode_forward(x.q[rows], x.cache("k", seqs), x.cache("v", seqs), x.seqlens[seqs],
                            x.scale, w.q_len, x.alibi_slopes, w.window), rows


def _check(x, O, lse, seqs=None, o_rel=0.0):
    (O_r, lse_r), rows = _oracle(x, seqs)
    e_o = np.abs(O[rows] - O_r) - o_rel * np.abs(O_r)
    assert e_o.max() <= TOL_O, float(np.abs(O[rows] - O_r).max())
    assert np.abs(lse[:, rows] - lse_r).max() <= TOL_LSE


@pytest.mark.parametrize("B,Hq,Hkv,S_max,d,q_len,lens", [
    (1, 1, 1, 64, 64, 1, (1,)),
    (2, 4, 1, 300, 128, 1, (300, 65)),
    (3, 8, 1, 1000, 128, 1, (64, 129, 1000)),
    (2, 16, 2, 513, 64, 1, (513, 200)),
    (1, 16, 1, 4096, 128, 1, (4096,)),
    (2, 4, 2, 777, 128, 2, (2, 777)),
    (4, 8, 2, 1030, 64, 4, (1030, 4, 127, 500)),
    (2, 2, 2, 256, 128, 3, (128, 131)),
    (5, 6, 3, 2000, 128, 1, (1999, 1, 64, 1500, 63)),
])
def test_decode_small(B, Hq, Hkv, S_max, d, q_len, lens):
    w = I.DecodeWorkload("t", B=B, Hq=Hq, Hkv=Hkv, S_max=S_max, d=d, q_len=q_len, lens=lens)
    x = I.make_decode_inputs(w, seed=S_max + q_len)
    _check(x, *G.decode(x))


@pytest.mark.parametrize("alibi,window,q_len", [(True, None, 1), (True, None, 3), (False, 0, 1),
                                                (False, 5, 2), (True, 100, 1), (False, 700, 4),
                                                (True, 2500, 2)])
def test_decode_alibi_window(alibi, window, q_len):
    w = I.DecodeWorkload("t", B=3, Hq=8, Hkv=2, S_max=2100, d=128, q_len=q_len,
                         lens=(2100, 333, 1024), alibi=alibi, window=window)
    x = I.make_decode_inputs(w, seed=5)
    _check(x, *G.decode(x))


def test_decode_bf16_output_and_full_caches():
    t = pytest.importorskip("torch")
    w = I.DecodeWorkload("t", B=2, Hq=8, Hkv=8, S_max=700, d=64, q_len=1)
    x = I.make_decode_inputs(w, seed=8)
    O, lse = G.decode(x, out_dtype=t.bfloat16, with_seqlens=False)   # every cache holds S_max
    _check(x, O, lse, o_rel=2.0 ** -8)


def test_decode_larger_chunks():
    """A batch large enough that the chunks grow past 64 keys (B * Hkv = 512
    caches of 1024: 256-key chunks)."""
    w = I.DecodeWorkload("t", B=64, Hq=16, Hkv=8, S_max=1024, d=128, q_len=1, len_range=(1, 1024))
    x = I.make_decode_inputs(w, seed=9)
    O, lse = G.decode(x)
    _check(x, O, lse, seqs=[0, 1, 2, 31, 63] + [int(b) for b in np.argsort(x.seqlens)[:3]])


def test_decode_matches_the_forward_kernel_last_rows():
    """fa_decode equals the last q_len rows of fa_fwd over the whole sequence
    (both through the library; same tolerance to each other as to the oracle)."""
    L, Hq, Hkv, d, q_len = 900, 8, 2, 128, 2
    fw = I.small_case("bf16", causal=True, B=1, Hq=Hq, Hkv=Hkv, N=L, d=d)
    xf = I.make_inputs(fw, seed=12)
    O_f, lse_f = G.forward(xf)
    w = I.DecodeWorkload("t", B=1, Hq=Hq, Hkv=Hkv, S_max=L, d=d, q_len=q_len, lens=(L,))
    x = I.make_decode_inputs(w, seed=0)
    x.q_bits = np.ascontiguousarray(xf.bits["q"][L - q_len:])
    x.q = xf.q[L - q_len:]
    x.k_bits = np.ascontiguousarray(xf.bits["k"][None])
    x.v_bits = np.ascontiguousarray(xf.bits["v"][None])
    O, lse = G.decode(x)
    assert np.abs(O - O_f[L - q_len:]).max() <= TOL_O
    assert np.abs(lse - lse_f[:, L - q_len:]).max() <= TOL_LSE
    _check(x, O, lse)


def test_decode_bad_lengths_reported():
    t = pytest.importorskip("torch")
    from exact_io_aware_36_gb300 import fa
    w = I.DecodeWorkload("t", B=2, Hq=4, Hkv=2, S_max=128, d=64, q_len=2, lens=(100, 128))
    x = I.make_decode_inputs(w, seed=1)
    q, kc, vc = G.bits_to_dev(x.q_bits), G.bits_to_dev(x.k_bits), G.bits_to_dev(x.v_bits)
    for bad in ((1, 128), (100, 129)):                 # shorter than q_len; longer than S_max
        cs = t.tensor(bad, dtype=t.int32, device="cuda")
        fa.attention_decode(q, kc, vc, cache_seqlens=cs, q_len=2)
        assert fa.fa_check_device_error(None) == 8
    G.decode(x)                                         # the context is still usable


@pytest.mark.slow
def test_decode_full_size_sampled():
    """The decode workload at full size, run as the benchmark runs it; every
    row of four sequences (the shortest, the longest and two others) checked
    against the oracle."""
    w = I.DECODE_WORKLOADS["decode_gqa"]
    x = I.make_decode_inputs(w, seed=0)
    O, lse = G.decode(x, guard=False)
    assert np.isfinite(O).all() and np.isfinite(lse).all()
    order = np.argsort(x.seqlens)
    _check(x, O, lse, seqs=sorted({int(order[0]), int(order[-1]), 3, 10}))
