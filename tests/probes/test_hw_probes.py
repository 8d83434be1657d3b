"""Hardware probes behind the kernels' design choices (GPU).

Each probe is a small CUDA program in this folder, compiled with nvcc for
sm_103a and run on the GPU; the test checks that it ran cleanly (no CUDA
error, no timed-out wait) and prints the rates it measured:

* mma_rate.cu     sustained tcgen05.mma rate by shape (M 128; N 64, 128, 256;
                  operands from shared memory or A from TMEM).
* mma_mix.cu      the backward dK/dV kernel's five products per 64-query step,
                  alone and together.
* reduce_rate.cu  L2 throughput of cp.reduce.async.bulk .add.f32 into an
                  accumulator larger than L2 and into one that fits.
* alu_rate.cu     per-SM rates of the forward softmax's per-score
                  instructions (ex2, cvt to bf16x2, prmt, packed add) and of
                  its whole per-pair body with either bf16 packing.

All operands are zero and every wait is bounded; nothing here faults or hangs.
"""
import os
import re
import shutil
import subprocess

import pytest

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))


def _build_and_run(name, tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / name)
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"),
                    os.path.join(HERE, name + ".cu"), "-o", exe], check=True, capture_output=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=120).stdout
    print(out)
    errs = re.findall(r"err=(\d+)", out)
    assert errs and all(e == "0" for e in errs), out
    assert all(s == "0" for s in re.findall(r"status=(\d+)", out)), out
    return out


@pytest.mark.parametrize("name", ["mma_rate", "mma_mix", "reduce_rate", "alu_rate"])
def test_probe(name, tmp_path):
    out = _build_and_run(name, tmp_path)
    rates = [float(a or b) for a, b in re.findall(r"([\d.]+) T[BF]|rate=([\d.]+)", out)]
    assert rates and min(rates) > 0
