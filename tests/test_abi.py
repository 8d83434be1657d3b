"""The C ABI loads and validates its arguments on the host (CPU only).

No test here launches a kernel: every call below is rejected (or is empty)
before the library touches the GPU.
"""
import ctypes
import os
import re

import pytest

from exact_io_aware_36_gb300 import build, fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return fa.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_abi():
    assert declared_functions() == sorted(fa.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(9):
        assert fa.fa_status_string(code)
    assert "unknown" in fa.fa_status_string(99)
    assert lib.fa_version() >= 10000


A = 0x10000   # a fake, 256-byte aligned device address (never dereferenced)


def fwd(**kw):
    a = dict(q=A, k=A, v=A, o=A, lse=A, B=1, Hq=2, Hkv=2, N=128, d=64, scale=0.125, causal=1,
             window=-1, cu=None, T=0, alibi=None, dtype=fa.FA_BF16, odt=fa.FA_BF16, stream=None)
    a.update(kw)
    return fa.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["N"],
                     a["d"], a["scale"], a["causal"], a["window"], a["cu"], a["T"], a["alibi"],
                     a["dtype"], a["odt"], a["stream"])


def bwd(**kw):
    a = dict(B=1, Hq=2, Hkv=2, N=128, d=64, scale=0.125, causal=1, window=-1, cu=None, T=0,
             alibi=None, dtype=fa.FA_BF16, odt=fa.FA_FP32, det=0, ws=A, wsb=1 << 40, stream=None,
             ptr=A)
    a.update(kw)
    p = a["ptr"]
    return fa.fa_bwd(p, p, p, p, p, p, p, p, p, a["B"], a["Hq"], a["Hkv"], a["N"], a["d"],
                     a["scale"], a["causal"], a["window"], a["cu"], a["T"], a["alibi"], a["dtype"],
                     a["odt"], a["det"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(lse=None), 1), (dict(o=None), 1),
    (dict(Hq=3, Hkv=2), 2), (dict(B=-1), 2), (dict(N=-5), 2), (dict(Hkv=0), 2),
    (dict(T=999), 2),                      # dense batch with T != B*N
    (dict(d=96), 3), (dict(d=256, dtype=fa.FA_FP32, odt=fa.FA_FP32), 3), (dict(dtype=7), 3),
    (dict(scale=0.0), 3), (dict(scale=float("nan")), 3), (dict(scale=-1.0), 3),
    (dict(q=A + 8), 4), (dict(v=A + 2), 4),
    (dict(dtype=fa.FA_FP32, q=A + 2, odt=fa.FA_FP32), 4),
    (dict(dtype=fa.FA_FP32, odt=fa.FA_BF16), 3), (dict(odt=5), 3),
    (dict(B=0), 0), (dict(N=0), 0),        # empty: nothing to launch
    (dict(window=4, causal=0), 3),         # a sliding window is a causal band
    (dict(window=0, causal=0), 3),
    (dict(window=4, B=0), 0), (dict(window=-7, causal=0, B=0), 0),
])
def test_fwd_rejects_before_launch(lib, kw, code):
    assert fwd(**kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(ptr=None), 1), (dict(Hq=4, Hkv=3), 2), (dict(odt=9), 3), (dict(d=32), 3), (dict(dtype=fa.FA_FP32), 3),
    (dict(ptr=A + 4), 4), (dict(ws=None), 5), (dict(wsb=1024), 5), (dict(ws=A + 16), 4),
    (dict(B=0), 0),
    (dict(window=3, causal=0), 3), (dict(det=2), 3), (dict(det=-1), 3),
    (dict(window=3, B=0), 0),
])
def test_bwd_rejects_before_launch(lib, kw, code):
    assert bwd(**kw) == code


def test_bwd_stage_rejects_unknown_stage(lib):
    p = A
    args = (p, p, p, p, p, p, p, p, p, 1, 2, 2, 128, 64, 0.125, 1, -1, None, 0, None, fa.FA_BF16,
            fa.FA_FP32, 0, A, 1 << 40, None)
    assert fa.fa_bwd_stage(3, *args) == 3
    assert fa.fa_bwd_stage(-1, *args) == 3
    bad = list(args)
    bad[0] = None
    assert fa.fa_bwd_stage(0, *bad) == 1


def test_workspace_size(lib):
    T, Hq, d = 1000, 3, 64
    n = fa.fa_bwd_workspace_size(1, Hq, T, d, 0)
    r = lambda x: (x + 255) // 256 * 256
    assert n == r(Hq * T * 4) + r(Hq * T * d * 4) + 256     # D, dQ accumulator, work counter
    assert fa.fa_bwd_workspace_size(2, Hq, 4096, d, T) == n   # packed: T given
    assert fa.fa_bwd_workspace_size(-1, Hq, T, d, 0) == 0


def dec(**kw):
    a = dict(q=A, k=A, v=A, cs=None, o=A, lse=A, B=2, Hq=8, Hkv=2, S=4096, ql=1, d=128,
             scale=0.088, window=-1, alibi=None, odt=fa.FA_FP32, ws=A, wsb=1 << 40, stream=None)
    a.update(kw)
    return fa.fa_decode(a["q"], a["k"], a["v"], a["cs"], a["o"], a["lse"], a["B"], a["Hq"],
                        a["Hkv"], a["S"], a["ql"], a["d"], a["scale"], a["window"], a["alibi"],
                        a["odt"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(lse=None), 1),
    (dict(Hq=6, Hkv=4), 2), (dict(B=-1), 2), (dict(ql=0), 2), (dict(S=-1), 2),
    (dict(ql=5000), 2),                          # more new tokens than the cache holds
    (dict(d=96), 3), (dict(Hq=32, Hkv=1), 3),    # 32 rows per kv head > 16
    (dict(Hq=8, Hkv=2, ql=5), 3), (dict(scale=0.0), 3), (dict(odt=4), 3),
    (dict(q=A + 8), 4), (dict(o=A + 4), 4), (dict(ws=A + 16), 4),
    (dict(ws=None), 5), (dict(wsb=1000), 5),
    (dict(B=0), 0),
])
def test_decode_rejects_before_launch(lib, kw, code):
    assert dec(**kw) == code


def test_decode_workspace_size(lib):
    from exact_io_aware_36_gb300 import inputs as I  # noqa: F401  (import check only)
    n = fa.fa_decode_workspace_size(16, 32, 8, 32768, 1, 128)
    # 16 x 8 (sequence, kv head) pairs, chunks of 2048 keys -> 16 chunks; R = 4 rows
    units = 16 * 8 * 16
    assert n == units * 4 * 128 * 4 + ((units * 4 * 3 * 4 + 255) // 256) * 256
    assert fa.fa_decode_workspace_size(1, 3, 2, 64, 1, 64) == 0      # Hq % Hkv != 0
    assert fa.fa_decode_workspace_size(1, 32, 1, 64, 1, 64) == 0     # 32 rows


def test_gqa_workspace_size(lib):
    """The grouped-query workspace adds two per-part sums of dK and dV
    (float32 [2][2][T, Hkv, d], 256-byte aligned) when Hq / Hkv is even,
    and equals the base size otherwise."""
    base = fa.fa_bwd_workspace_size(2, 32, 8192, 128, 0)
    assert fa.fa_bwd_workspace_size_gqa(2, 32, 4, 8192, 128, 0) == base + 2 * 2 * 16384 * 4 * 128 * 4
    assert fa.fa_bwd_workspace_size_gqa(2, 32, 16, 8192, 128, 0) == base + 2 * 2 * 16384 * 16 * 128 * 4
    assert fa.fa_bwd_workspace_size_gqa(2, 32, 32, 8192, 128, 0) == base
    assert fa.fa_bwd_workspace_size_gqa(1, 6, 2, 100, 64, 0) == fa.fa_bwd_workspace_size(1, 6, 100, 64, 0)
    assert fa.fa_bwd_workspace_size_gqa(1, 6, 4, 100, 64, 0) == 0        # Hq % Hkv != 0
    assert fa.fa_bwd_workspace_size_gqa(3, 8, 1, 0, 64, 1000) == \
        fa.fa_bwd_workspace_size(3, 8, 0, 64, 1000) + ((2 * 2 * 1000 * 1 * 64 * 4 + 255) // 256) * 256
