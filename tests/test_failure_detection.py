"""Failure detection on the device without a GPU fault (GPU).

A pipeline wait that can never complete returns an error status within its
limit instead of hanging; malformed cu_seqlens are reported by the kernels;
in both cases the context stays usable.  Nothing here faults, traps or hangs
a GPU: the stall is a barrier nothing arrives on, bounded by %globaltimer.
"""
import time

import numpy as np
import pytest

from exact_io_aware_36_gb300 import build, fa
from exact_io_aware_36_gb300 import inputs as I
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    build.build()
    import torch as t
    t.cuda.init()
    return t


def _small_forward_ok(torch):
    w = I.small_case("bf16", causal=True, B=1, Hq=2, Hkv=2, N=200, d=64)
    x = I.make_inputs(w, seed=4)
    O, lse = G.forward(x)      # checks the device status after the call
    assert np.isfinite(O).all()


def test_stalled_wait_returns_timeout_status(torch):
    assert fa.fa_check_device_error(None) == 0
    t0 = time.time()
    assert fa.fa_selftest_wait_timeout(50_000_000, None) == 0       # 50 ms limit
    assert fa.fa_check_device_error(None) == 7                        # FA_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 10.0
    assert fa.fa_check_device_error(None) == 0                        # read clears it
    _small_forward_ok(torch)


def test_selftest_rejects_bad_limits(torch):
    assert fa.fa_selftest_wait_timeout(0, None) == 3
    assert fa.fa_selftest_wait_timeout(20_000_000_000, None) == 3


def test_malformed_cu_seqlens_reported(torch):
    w = I.small_case("bf16", causal=True, Hq=2, Hkv=2, d=64, seqlens=(64, 64, 64))
    x = I.make_inputs(w, seed=1)
    q, k, v = G.to_dev(x, "q"), G.to_dev(x, "k"), G.to_dev(x, "v")
    bad = torch.tensor([0, 100, 50, 192], dtype=torch.int32, device="cuda")   # not monotone
    o = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty((2, x.T), dtype=torch.float32, device="cuda")
    st = fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 3, 2, 2,
                   64, 64, x.scale, 1, -1, bad.data_ptr(), x.T, None, fa.FA_BF16, fa.FA_FP32, None)
    assert st == 0                                                   # detected on the device
    assert fa.fa_check_device_error(None) == 8                       # FA_ERR_CU_SEQLENS
    too_long = torch.tensor([0, 64, 192, 192], dtype=torch.int32, device="cuda")   # 128 > N=64
    st = fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 3, 2, 2,
                   64, 64, x.scale, 1, -1, too_long.data_ptr(), x.T, None, fa.FA_BF16, fa.FA_FP32,
                   None)
    assert st == 0
    assert fa.fa_check_device_error(None) == 8
    _small_forward_ok(torch)
