"""The forward's build-time option of a correction warpgroup (GPU).

Built with FA_FWD_CORRECTION_WARPS=1, the persistent forward runs a fourth
warpgroup that rescales O rows in TMEM when a softmax warp raises its
reference max and writes each item's epilogue (O / l, LSE), so the softmax
warps only compute P ("FlashAttention: Faster Attention Without Dropping a
Single Interaction", FA3 adaptation: producer, consumer and correction
roles).  It is slower than the default build on every workload measured
(the default keeps both jobs in the softmax warps), so it is not the default;
this file keeps it correct: it builds that variant of the library and
checks it against the fp64 oracle on the cases that reach its paths (many
items per CTA, ragged tails, packed batches, and rows whose max jumps by
far more than the rescale threshold, which send rescale requests).
"""
import numpy as np
import pytest

from oracle import attention_fp64 as A
from exact_io_aware_36_gb300 import build, fa
from exact_io_aware_36_gb300 import inputs as I
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    return fa.load(build.build_variant("corr", ["FA_FWD_CORRECTION_WARPS=1"]))


CASES = [
    # kind, B, Hq, Hkv, N, d, causal, alibi, seqlens
    (None, 2, 8, 2, 1000, 128, True, False, None),
    (None, 1, 4, 4, 300, 64, False, True, None),
    (None, 1, 4, 2, 0, 128, True, False, (5, 300, 1, 600, 129)),
    ("late_dominant", 1, 4, 2, 1024, 128, True, False, None),
    ("rising", 1, 4, 2, 1024, 64, True, False, None),
    ("falling", 1, 4, 2, 1024, 128, True, True, None),
]


@pytest.mark.parametrize("kind,B,Hq,Hkv,N,d,causal,alibi,seqlens", CASES)
def test_correction_warpgroup_variant(lib, kind, B, Hq, Hkv, N, d, causal, alibi, seqlens):
    t = G.torch()
    w = I.small_case("bf16", causal=causal, B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, alibi=alibi,
                     seqlens=seqlens)
    x = I.make_inputs(w, seed=31)
    if kind is not None:
        I.add_score_structure(x, kind, {"late_dominant": 30.0, "rising": 200.0, "falling": 200.0}[kind],
                              seed=32)
    q, k, v = G.to_dev(x, "q"), G.to_dev(x, "k"), G.to_dev(x, "v")
    cu = t.from_numpy(x.cu_seqlens).cuda() if w.varlen else None
    sl = t.from_numpy(x.alibi_slopes).cuda() if w.alibi else None
    obuf, o = G.guarded_empty(q.shape, t.float32)
    lbuf, lse = G.guarded_empty((w.Hq, x.T), t.float32)
    P = lambda a: None if a is None else a.data_ptr()
    sp = t.cuda.current_stream().cuda_stream
    st = lib.fa_fwd(P(q), P(k), P(v), P(o), P(lse), w.B, w.Hq, w.Hkv, w.N, w.d, x.scale,
                    int(causal), -1, P(cu), x.T, P(sl), fa.FA_BF16, fa.FA_FP32, sp)
    assert st == 0
    assert lib.fa_check_device_error(sp) == 0
    G.assert_guards(obuf)
    G.assert_guards(lbuf)
    O_r, lse_r = A.attention_forward(x.q, x.k, x.v, x.scale, causal, x.cu_seqlens, x.alibi_slopes)
    assert np.abs(G.as_f64(o) - O_r).max() <= 1e-2
    assert np.abs(G.as_f64(lse) - lse_r).max() <= 1e-3
