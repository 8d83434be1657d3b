"""The benchmark's host-side pieces (CPU): the oracle samples behind the
`cpu_baseline` objects and the reference arm's line.

Each runs on a small workload here; on the GPU machine the same functions run
on the bench workload.  Only the shape of what they report is checked: the
oracle's values are pinned by the oracle tests.
"""
import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from exact_io_aware_36_gb300 import inputs as I  # noqa: E402


def _check_baseline(cb):
    assert cb["kind"] == "oracle" and cb["unit"] == "TFLOP/s"
    assert cb["value"] > 0 and cb["cores"] >= 1
    assert "sequence 0" in cb["sample"]


def test_bf16_oracle_sample():
    w = I.small_case("bf16", causal=True, B=2, Hq=4, Hkv=2, N=96, d=64, alibi=True)
    x = I.make_inputs(w, seed=1)
    fl, dt, what = bench.oracle_sample(w, x)
    # one causal head of 96 tokens, forward and backward: 14 d per pair
    assert fl == 14.0 * 64 * 96 * 97 / 2
    assert dt > 0 and "1 of 8" in what
    _check_baseline(bench.cpu_baseline(w, x))


def test_fp8_oracle_sample():
    w = I.small_case("bf16", causal=True, B=2, Hq=4, Hkv=2, N=200, d=128, alibi=True)
    x = I.make_inputs(w, seed=2, with_do=False)
    cb = bench.oracle_fp8_baseline(w, x, I.hadamard_signs(w.d, seed=0))
    _check_baseline(cb)
    assert "L=200" in cb["sample"]


def test_reference_arm_line_for_the_fp32_workload():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "c1_fp32_fwd", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.FWD_FP32_METRIC
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert np.isfinite(line["value"]) and line["value"] > 0


def test_secondary_roofs_algorithmic_bytes(monkeypatch):
    # c3: the forward reads q, k, v (bf16) and writes O (fp32) and LSE:
    # 403 MB + 270 MB; dK/dV reads q, k, v, dO, LSE, D and the fp32 dQ
    # accumulator and writes dK, dV and the accumulator: 810 MB + 537 MB.
    import types
    import torch
    monkeypatch.setattr(torch.cuda, "get_device_properties",
                        lambda dev: types.SimpleNamespace(multi_processor_count=152))
    monkeypatch.setattr(bench, "max_sm_mhz", lambda dev: 2070.0)
    w = I.workload("c3_long")
    T = w.B * w.N
    fl = bench.flops_per_step(w, [w.N] * w.B)
    out = bench.secondary_roofs(w, T, fl, {"fwd": 1.0, "bwd_dkdv": 2.0}, "cpu", 6796.9)
    assert out["fwd"]["alg_bytes"] == 402_653_184 + 270_532_608
    assert out["bwd_dkdv"]["alg_bytes"] == 809_500_672 + 536_870_912
    # one exp2 per attended pair; peak 152 x 30.3 x 2.07 GHz
    assert abs(out["fwd"]["exp2_per_s"] / (fl["pairs"] / 1e-3) - 1) < 1e-3
    assert abs(out["fwd"]["exp2_peak_per_s"] / (152 * 30.3 * 2070e6) - 1) < 1e-3
    det = bench.secondary_roofs(w, T, fl, {"fwd": 1.0, "bwd_dkdv": 2.0}, "cpu", 6796.9, det=True)
    assert det["bwd_dkdv"]["alg_bytes"] == out["bwd_dkdv"]["alg_bytes"] - 2 * 4 * T * w.Hq * w.d
