"""The seeded input recipe (CPU only)."""
import numpy as np
import pytest

from exact_io_aware_36_gb300 import inputs as I


def test_varlen_total_tokens_seed0():
    w = I.workload("c4_varlen")
    L = I.make_seqlens(w, 0)
    assert len(L) == 64 and L.min() >= 128 and L.max() <= 4096
    assert int(L.sum()) == 137663


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.random.Generator(np.random.PCG64(1)).standard_normal(100000).astype(np.float32)
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 3.0e38]
    ours = I.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_inputs_are_bf16_exact_and_seeded():
    w = I.small_case("bf16", B=2, Hq=4, Hkv=2, N=33, d=64)
    a = I.make_inputs(w, seed=5)
    b = I.make_inputs(w, seed=5)
    for n in ("q", "k", "v", "do"):
        np.testing.assert_array_equal(getattr(a, n), getattr(b, n))
        x = getattr(a, n)
        np.testing.assert_array_equal(I.bf16_round(x), x)
        np.testing.assert_array_equal(I.bf16_from_bits(a.bits[n]).reshape(x.shape), x)
    assert a.q.shape == (66, 4, 64) and a.k.shape == (66, 2, 64)
    assert list(a.cu_seqlens) == [0, 33, 66]


def test_attended_pairs():
    assert I.attended_pairs(I.workload("c3_long")) == 32 * 16384 * 16385 // 2
    assert I.attended_pairs(I.workload("c1_fp32_fwd")) == 128 * 128


def test_attended_pairs_counts_the_band():
    """Band area against a brute-force count of visible (i, j) pairs."""
    for L, wnd in ((1, 0), (5, 0), (300, 40), (129, 128), (129, 127), (64, 1000)):
        w = I.small_case("bf16", causal=True, B=1, Hq=3, Hkv=1, N=L, d=64, window=wnd)
        brute = sum(1 for i in range(L) for j in range(L) if i - wnd <= j <= i)
        assert I.attended_pairs(w) == 3 * brute
    w = I.small_case("bf16", causal=True, Hq=2, Hkv=2, d=64, seqlens=(7, 0, 50), window=3)
    brute = sum(1 for L in (7, 0, 50) for i in range(L) for j in range(L) if i - 3 <= j <= i)
    assert I.attended_pairs(w) == 2 * brute
