"""Host-side set-up is done once per shape: the per-shape cache of TMA
descriptors and the once-per-(device, kernel) shared-memory limit.

A launch needs descriptors for its tensors (address, sizes, strides, box);
repeated calls on the same buffers, as in a training or serving loop, must
reuse them instead of encoding them through the driver again.
"""
import numpy as np
import pytest

from exact_io_aware_36_gb300 import build, fa
from exact_io_aware_36_gb300 import inputs as I


@pytest.fixture(scope="module")
def lib():
    build.build()
    return fa.load()


def test_stats_are_exported_and_start_at_zero_without_a_gpu(lib):
    """No call above launched anything here (CPU: every call is rejected or
    empty before the set-up), so nothing was encoded or set."""
    enc, reused, attrs = fa.fa_host_cache_stats()
    assert enc >= 0 and reused >= 0 and attrs >= 0
    import torch
    if not torch.cuda.is_available():
        assert (enc, reused, attrs) == (0, 0, 0)


@pytest.mark.gpu
def test_repeated_calls_encode_nothing(lib):
    import torch
    w = I.small_case("bf16", causal=True, B=2, Hq=4, Hkv=2, N=300, d=128, alibi=True)
    x = I.make_inputs(w, seed=3)
    dev = lambda n: torch.from_numpy(x.bits[n].view(np.int16)).view(torch.bfloat16).cuda()
    q, k, v, do = dev("q"), dev("k"), dev("v"), dev("do")
    slopes = torch.from_numpy(x.alibi_slopes).cuda()
    kw = dict(causal=True, scale=x.scale, batch=w.B, alibi_slopes=slopes)
    o = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty((w.Hq, x.T), dtype=torch.float32, device="cuda")
    ws = torch.empty(fa.fa_bwd_workspace_size(w.B, w.Hq, w.N, w.d, 0), dtype=torch.uint8,
                     device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def call():
        fa.attention_forward(q, k, v, out=o, lse=lse, **kw)
        fa.attention_backward(q, k, v, o, do, lse, workspace=ws, dq=dq, dk=dk, dv=dv, **kw)

    call()                                 # first call: encodes what it needs
    torch.cuda.synchronize()
    first = [t.clone() for t in (o, lse, dq, dk, dv)]
    e0, r0, a0 = fa.fa_host_cache_stats()
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    e1, r1, a1 = fa.fa_host_cache_stats()
    assert e1 == e0, "a repeated call encoded descriptors again"
    assert a1 == a0, "a repeated call set a shared-memory limit again"
    # forward: q, k, v; dK/dV kernel: q, dO, k, v; three calls
    assert r1 - r0 >= 3 * 7
    assert fa.fa_check_device_error() == 0
    # the reused descriptors address the same tensors: same results (dK, dV
    # and the forward bit for bit; dq's fp32 reduction order may vary)
    for a, b in zip(first[:2] + first[3:], (o, lse, dk, dv)):
        assert torch.equal(a, b)
