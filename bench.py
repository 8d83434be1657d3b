#!/usr/bin/env python
"""Benchmark: causal bf16 attention forward + backward TFLOP/s on one GB300.

One step is one pass of the whole hot path over one batch: the forward
kernel (O, LSE), then the three backward kernels (D and dQ-accumulator
reset; dK, dV and dQ accumulation; dQ convert).  The default workload is the
long-context configuration B=1, H=32, N=16384, d=128, causal, bf16 (q, k
scaled by 0.5), the one the throughput target is stated on.  Inputs are
seeded synthetic data (no dataset), resident in HBM before the timed region.
At the default workload they total 537 MB, larger than the 129 MB L2, so the
steps run back to back; a workload whose inputs fit L2 gets a 512 MB write
between steps (outside each step's events) and its time is the sum of the
steps' own event intervals.

FLOPs are algorithmic: 4*d per attended pair forward, 10*d backward (five
MMAs, with the recomputation of S counted), so 14*d*pairs per step; causal
pairs are L(L+1)/2 per sequence and head.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun each rank runs its own replica (the path shards into
independent problems; there is no data-path collective): "scaling": "weak".
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_io_aware_36_gb300 import inputs as I  # noqa: E402

METRIC = "causal bf16 attention fwd+bwd TFLOP/s on 1 GB300; % of dense BF16 tensor peak"
FWD_FP32_METRIC = "fp32 attention forward TFLOP/s on 1 GB300 (latency-bound size)"
UNIT = "TFLOP/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_dram_traffic.json")
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="c3_long",
                    choices=sorted(I.WORKLOADS) + sorted(I.EXTRA_WORKLOADS) +
                    sorted(I.DECODE_WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--fp8", action="store_true",
                    help="time the FP8 forward (quantize + e4m3 attention) on the workload")
    ap.add_argument("--deterministic", action="store_true",
                    help="time the deterministic backward (dQ by its own kernel, no atomics)")
    ap.add_argument("--record-traffic", metavar="NCU_CSV",
                    help="do not run: store the DRAM bytes per launch from an ncu --csv log of "
                         "this workload / mode in profiles/ncu_dram_traffic.json and exit")
    return ap.parse_args()


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The job's time is the slowest rank's: all-reduce MAX over the ranks
    (the only collective; replicas exchange no data)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank_step: float, ms_per_step: float, world: int) -> float:
    """Whole-job TFLOP/s: every rank runs the same replica (weak scaling)."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def flops_per_step(w: I.Workload, seqlens) -> dict:
    pairs = I.attended_pairs(w, seqlens)
    return {"pairs": pairs, "fwd": 4.0 * w.d * pairs, "bwd": 10.0 * w.d * pairs,
            "total": (14.0 if w.backward else 4.0) * w.d * pairs}


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), float(pk.get("hbm_gbs", 0.0)), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, 6800.0, "fallback"


def max_sm_mhz(dev) -> float:
    try:
        out = subprocess.run(["nvidia-smi", "-i", str(smi_index(dev.index or 0)),
                              "--query-gpu=clocks.max.sm", "--format=csv,noheader,nounits"],
                             capture_output=True, text=True, timeout=10).stdout
        return float(out.strip().splitlines()[0])
    except Exception:
        return 2070.0


def fp32_fma_peak_tflops(dev) -> float:
    """fp32 FMA peak of the CUDA cores: SMs x 128 lanes x 2 flops x the
    device's maximum SM clock."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    return round(sms * 128 * 2 * max_sm_mhz(dev) * 1e6 / 1e12, 2)


# ex2.approx.ftz.f32 issued per SM per clock on GB300: 8 independent chains of
# dependent ex2.approx per thread, 4 x 152 blocks of 512 threads, timed with
# CUDA events at the 2070 MHz maximum clock (a stand-alone microbenchmark)
EX2_PER_SM_CLK = 30.3


def secondary_roofs(w, T, fl, kern_ms, dev, hbm_gbs, det=False):
    """The exp2 (MUFU) and HBM roofs of the forward and dK/dV kernels beside
    their tensor roof: one exp2 per attended pair in each, and the bytes each
    must move at least (inputs read once, outputs written once; dK/dV also
    reads and writes the fp32 dQ accumulator once, except in the
    deterministic backward, which has none)."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ex2_peak = sms * EX2_PER_SM_CLK * max_sm_mhz(dev) * 1e6          # exp2 per second
    qb, kvb = T * w.Hq * w.d, T * w.Hkv * w.d                        # elements
    alg = {"fwd": 2 * qb + 2 * 2 * kvb + 4 * qb + 4 * w.Hq * T,        # q, k, v in; O fp32, LSE out
           "bwd_dkdv": (2 * qb + 2 * 2 * kvb + 2 * qb + 2 * 4 * w.Hq * T  # q, k, v, dO, LSE, D in
                        + 2 * 2 * kvb + (0 if det else 2 * 4 * qb))}   # dK, dV out; dQacc in and out
    out = {}
    for n in ("fwd", "bwd_dkdv"):
        if n not in kern_ms or (n == "bwd_dkdv" and not w.backward):
            continue
        sec = kern_ms[n] * 1e-3
        ex2_rate = fl["pairs"] / sec
        gbs = alg[n] / sec / 1e9
        out[n] = {"exp2_per_s": float(f"{ex2_rate:.4g}"), "exp2_peak_per_s": float(f"{ex2_peak:.4g}"),
                  "exp2_frac": round(ex2_rate / ex2_peak, 4),
                  "alg_bytes": int(alg[n]), "hbm_gbs": round(gbs, 1),
                  "hbm_frac": round(gbs / hbm_gbs, 4) if hbm_gbs else None}
    return out


def source_hash(name: str) -> str:
    src = os.path.join(ROOT, "exact_io_aware_36_gb300", "csrc", name)
    return hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]


L2_BYTES = 129e6


def input_mb(w, T):
    """The step's inputs in MB: q, k, v, dO in bf16 and O in fp32."""
    return T * w.d * (2 * (2 * w.Hq + 2 * w.Hkv) + 4 * w.Hq) / 1e6


def l2_note(w, T):
    """How the timing treats L2."""
    mb = input_mb(w, T)
    if mb * 1e6 > L2_BYTES:
        return f"inputs exceed L2 ({mb:.0f} MB); no flush between steps"
    return f"inputs fit L2 ({mb:.0f} MB); 512 MB written between steps, outside the step events"


def ncu_traffic(workload: str, kernel: str):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from the
    committed ncu summary, or None when there is none or when any source the
    kernel is built from has changed since the counters were taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)[workload][kernel]
        if any(source_hash(n) != h for n, h in rec["sources_sha256_16"].items()):
            return None
        return rec["bytes_per_launch"]
    except Exception:
        return None


# ncu kernel-name fragment -> (per-kernel key, the source files it is built from).
# The decode call (split + combine) launches two kernels; their figures are
# summed per call, a call being counted by the launches of its last kernel
# (CALL_LAST).
_COMMON_SOURCES = ["fa_ptx.cuh", "fa_internal.h", "fa_host_util.cu"]
KERNEL_SOURCES = [
    ("fwd_bf16_block_kernel", "fwd", "fa_fwd_bf16_block.cu"),
    ("fwd_bf16_kernel", "fwd", "fa_fwd_bf16.cu"),
    ("bwd_preprocess_kernel", "bwd_preprocess", "fa_bwd_bf16.cu"),
    ("bwd_dkdv_kernel", "bwd_dkdv", "fa_bwd_bf16.cu"),
    ("bwd_convert_kernel", "bwd_dq_convert", "fa_bwd_bf16.cu"),
    ("bwd_dq_kernel", "bwd_dq", "fa_bwd_dq_bf16.cu"),
    ("fwd_fp8_kernel", "fwd_fp8", "fa_fwd_fp8.cu"),
    ("quant_", "fp8_quantize", "fa_fp8_quant.cu"),
    ("decode_", "decode", "fa_decode_bf16.cu"),
]
CALL_LAST = {"decode": "combine"}
_BYTE_UNITS = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12}
_TIME_UNITS = {"ns": 1, "us": 1e3, "usecond": 1e3, "ms": 1e6, "msecond": 1e6, "nsecond": 1}


def traffic_key(args) -> str:
    return args.workload + (" fp8" if args.fp8 else "") + (" deterministic" if args.deterministic else "")


def record_traffic(csv_path: str, key: str) -> dict:
    """Per-kernel DRAM bytes per launch from an `ncu --csv` metrics log.

    Launches of one kernel are averaged; the decode call's split and combine
    kernels are summed per call.  Each
    entry carries a hash of every source the kernel is built from, so that
    ncu_traffic() drops it once the kernel changes."""
    import csv
    rows = [r for r in csv.reader(open(csv_path)) if r]
    hdr = next(i for i, r in enumerate(rows) if "Metric Name" in r)
    h = rows[hdr]
    col = {n: h.index(n) for n in ("ID", "Kernel Name", "Metric Name", "Metric Unit", "Metric Value")}
    launches = {}
    for r in rows[hdr + 1:]:
        if len(r) != len(h):
            continue
        name = r[col["Kernel Name"]]
        match = next((k for k in KERNEL_SOURCES if k[0] in name), None)
        if match is None:
            continue
        lid = r[col["ID"]]
        rec = launches.setdefault(lid, {"kernel": match[1], "source": match[2], "name": name})
        unit, metric = r[col["Metric Unit"]], r[col["Metric Name"]]
        try:
            val = float(r[col["Metric Value"]].replace(",", ""))
        except ValueError:           # a metric this kernel does not report ("n/a")
            continue
        if metric in ("dram__bytes_read.sum", "dram__bytes_write.sum", "lts__t_bytes.sum"):
            val *= _BYTE_UNITS.get(unit, 1)
        elif metric == "gpu__time_duration.sum":
            val *= _TIME_UNITS.get(unit, 1)
        rec[metric] = val
    per = {}
    for rec in launches.values():
        per.setdefault(rec["kernel"], []).append(rec)
    out = {}
    for kern, recs in per.items():
        last = CALL_LAST.get(kern)
        calls = len(recs) if last is None else max(1, sum(last in r["name"] for r in recs))
        tot = lambda m: sum(r.get(m, 0.0) for r in recs) / calls
        rd, wr = tot("dram__bytes_read.sum"), tot("dram__bytes_write.sum")
        srcs = [recs[0]["source"]] + _COMMON_SOURCES
        out[kern] = {"sources_sha256_16": {n: source_hash(n) for n in srcs},
                     "dram_bytes_read": int(rd), "dram_bytes_write": int(wr),
                     "bytes_per_launch": int(rd + wr),
                     "gpu_time_ns_under_ncu": int(tot("gpu__time_duration.sum")),
                     "launches_averaged": calls}
        if any("lts__t_bytes.sum" in r for r in recs):
            out[kern]["lts_bytes"] = int(tot("lts__t_bytes.sum"))
    try:
        with open(TRAFFIC_FILE) as f:
            table = json.load(f)
    except Exception:
        table = {}
    table[key] = out
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(table, f, indent=1)
        f.write("\n")
    return out


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        reasons = sorted({self.NAMES[i] for *_, fl in rows for i, v in enumerate(fl)
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "reasons": reasons,
                "samples": len(rows)}


def smi_index(local: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    parts = [p for p in vis.split(",") if p.strip()]
    if local < len(parts) and parts[local].strip().isdigit():
        return int(parts[local])
    return local


# ------------------------------------------------------------------ decode

DECODE_METRIC = "decode attention over a KV cache: HBM bytes moved per second"


def oracle_decode_sample(w, x):
    """All query rows of one sequence (sequence 0) of a decode step through the
    oracle as it stands; returns (bytes that step moves for it, seconds, what)."""
    from oracle import attention_fp64 as A
    t0 = time.perf_counter()
    A.decode_forward(x.q[:w.q_len], x.cache("k", [0]), x.cache("v", [0]), x.seqlens[:1], x.scale,
                     w.q_len, x.alibi_slopes, w.window)
    dt = time.perf_counter() - t0
    nbytes = I.decode_bytes(dataclasses.replace(w, B=1), x.seqlens[:1])
    return nbytes, dt, f"sequence 0 of {w.B} (cache of {int(x.seqlens[0])} tokens), all {w.Hq} heads"


def run_decode(args, world, rank, local):
    """One step = one fa_decode call (split + combine kernels) over the whole
    batch; `value` = the HBM bytes the step must move (every cached key and
    value once, q, O, LSE) per second."""
    import torch
    from exact_io_aware_36_gb300 import fa

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = I.DECODE_WORKLOADS[args.workload]
    x = I.make_decode_inputs(w, seed=0)
    nbytes = I.decode_bytes(w, x.seqlens)

    def todev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    q, kc, vc = todev(x.q_bits), todev(x.k_bits), todev(x.v_bits)
    cs = torch.from_numpy(x.seqlens.astype(np.int32)).to(dev)
    slopes = torch.from_numpy(x.alibi_slopes).to(dev) if w.alibi else None
    o = torch.empty(q.shape, dtype=torch.float32, device=dev)
    lse = torch.empty((w.Hq, q.shape[0]), dtype=torch.float32, device=dev)
    ws_bytes = fa.fa_decode_workspace_size(w.B, w.Hq, w.Hkv, w.S_max, w.q_len, w.d)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    P = lambda t: None if t is None else t.data_ptr()

    def step():
        st = fa.fa_decode(P(q), P(kc), P(vc), P(cs), P(o), P(lse), w.B, w.Hq, w.Hkv, w.S_max,
                          w.q_len, w.d, float(x.scale), w.window_arg, P(slopes), fa.FA_FP32,
                          P(ws), ws_bytes, sp)
        if st:
            raise fa.FAError(st, "fa_decode")

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize(dev)
    st = fa.fa_check_device_error(sp)
    if st:
        raise fa.FAError(st, "warm-up")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(smi_index(local))
    sampler.start()
    time.sleep(0.1)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    st = fa.fa_check_device_error(sp)
    if st:
        raise fa.FAError(st, "timed region")
    total_ms = max_over_ranks(start.elapsed_time(end), world, dev)
    ms_step = total_ms / args.steps
    gbs = world * nbytes / (ms_step * 1e-3) / 1e9
    call_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    _, hbm, src = load_peaks()
    ach = nbytes / (call_ms * 1e-3) / 1e9
    roof = {"kernel": "decode_split + decode_combine (one fa_decode call)", "bound": "hbm",
            "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s", "frac": round(ach / hbm, 4),
            "peak_source": f"{src} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
            "traffic": ncu_traffic(w.name, "decode")}
    e2e = None
    if not args.no_e2e:
        hq = torch.from_numpy(np.ascontiguousarray(x.q_bits).view(np.int16)).view(torch.bfloat16).pin_memory()
        hcs = torch.from_numpy(x.seqlens.astype(np.int32)).pin_memory()
        ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)

        def e2e_step():
            q.copy_(hq, non_blocking=True)
            cs.copy_(hcs, non_blocking=True)
            step()
            ho.copy_(o, non_blocking=True)
            hl.copy_(lse, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / args.steps
        e2e = {"value": round(world * nbytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
               "ms_per_step": round(ms, 4),
               "h2d_bytes_per_step": hq.numel() * 2 + hcs.numel() * 4,
               "d2h_bytes_per_step": ho.numel() * 4 + hl.numel() * 4,
               "path": "fa_decode through the C ABI; new tokens' q and cache lengths copied in, "
                       "O and LSE copied out (the cache stays resident)"}
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cb, dt, what = oracle_decode_sample(w, x)
        cpu = {"value": round(cb / dt / 1e9, 4), "unit": "GB/s", "cores": os.cpu_count(),
               "kind": "oracle", "sample": what, "seconds": round(dt, 2),
               "note": "NumPy float64; BLAS threads = all cores"}
    line = {
        "metric": DECODE_METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded PCG64, seed 0; no dataset)",
        "config": {"workload": w.name, "desc": w.note, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv,
                   "S_max": w.S_max, "d": w.d, "q_len": w.q_len,
                   "cache_tokens": int(x.seqlens.sum()), "bytes_per_step": nbytes,
                   "alibi": w.alibi, "window": w.window, "o_dtype": "fp32",
                   "pct_of_hbm_peak": round(100.0 * gbs / world / hbm, 2),
                   "l2": f"cache {nbytes / 1e9:.2f} GB read per step exceeds L2; no flush",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roof,
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- fp8

FP8_METRIC = "FP8 (e4m3) attention forward TFLOP/s on 1 GB300 (quantize + attention)"
FP8_OVER_BF16 = 2.0        # nominal dense fp8 / bf16 tensor rate (4.5 / 2.25 PFLOP/s)


def run_fp8(args, world, rank, local):
    """One step = fa_fp8_quantize (incoherent transform, per-block e4m3 codes)
    then fa_fwd_fp8 over the workload; FLOPs are the forward's 4 d per pair."""
    import torch
    from exact_io_aware_36_gb300 import fa

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = I.workload(args.workload)
    x = I.make_inputs(w, seed=0, with_do=False)
    fl = flops_per_step(w, x.seqlens)["fwd"]
    T = x.T

    def todev(name):
        return torch.from_numpy(x.bits[name].view("int16")).view(torch.bfloat16).to(dev)

    q, k, v = todev("q"), todev("k"), todev("v")
    signs = torch.from_numpy(I.hadamard_signs(w.d, seed=0)).to(dev)
    cu = torch.from_numpy(x.cu_seqlens).to(dev) if w.varlen else None
    slopes = torch.from_numpy(x.alibi_slopes).to(dev) if w.alibi else None
    o = torch.empty(q.shape, dtype=torch.float32, device=dev)
    lse = torch.empty((w.Hq, T), dtype=torch.float32, device=dev)
    st, lay = fa.fa_fp8_layout_get(w.B, w.Hq, w.Hkv, w.N, w.d, T if w.varlen else 0)
    if st:
        raise fa.FAError(st, "fa_fp8_layout_get")
    buf = torch.empty(lay.total, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    P = lambda t: None if t is None else t.data_ptr()

    ptrs0 = (P(q), P(k), P(v), P(o), P(lse))

    def step(evs=None, ptrs=ptrs0):
        pq, pk, pv, po, plse = ptrs
        if evs is not None:
            evs[0].record(stream)
        r = fa.fa_fp8_quantize(pq, pk, pv, P(signs), w.B, w.Hq, w.Hkv, w.N, w.d, P(cu), T,
                               P(buf), lay.total, sp)
        if r:
            raise fa.FAError(r, "fa_fp8_quantize")
        if evs is not None:
            evs[1].record(stream)
        r = fa.fa_fwd_fp8(P(buf), lay.total, po, plse, w.B, w.Hq, w.Hkv, w.N, w.d,
                          float(x.scale), int(w.causal), w.window_arg, P(cu), T, P(slopes),
                          fa.FA_FP32, sp)
        if r:
            raise fa.FAError(r, "fa_fwd_fp8")
        if evs is not None:
            evs[2].record(stream)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize(dev)
    if fa.fa_check_device_error(sp):
        raise fa.FAError(7, "warm-up")
    evsets = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(smi_index(local))
    sampler.start()
    time.sleep(0.1)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        step(evsets[i])
    end.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    st = fa.fa_check_device_error(sp)
    if st:
        raise fa.FAError(st, "timed region")
    ms_step = max_over_ranks(start.elapsed_time(end), world, dev) / args.steps
    value = job_throughput(fl, ms_step, world)
    q_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evsets)
    a_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evsets)
    bf16_peak, _, src = load_peaks()
    peak = bf16_peak * FP8_OVER_BF16
    ach = fl / (a_ms * 1e-3) / 1e12

    e2e = None
    if not args.no_e2e:
        # the quantized buffer is scratch of the compute stream: one suffices
        sets = [{"ins": [q, k, v], "outs": [o, lse], "ptrs": ptrs0}]
        q2, k2, v2, o2, lse2 = (torch.empty_like(t) for t in (q, k, v, o, lse))
        sets.append({"ins": [q2, k2, v2], "outs": [o2, lse2],
                     "ptrs": (P(q2), P(k2), P(v2), P(o2), P(lse2))})
        host = lambda n: torch.from_numpy(x.bits[n].view("int16")).view(torch.bfloat16)
        e2e = run_e2e(args, {"total": fl}, world, dev, stream, step,
                      [host("q"), host("k"), host("v")], sets, "fa_fp8_quantize + fa_fwd_fp8",
                      kernel_ms=ms_step)
    line = {
        "metric": FP8_METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic (seeded PCG64, seed 0; no dataset)",
        "config": {"workload": w.name, "desc": w.note, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv,
                   "N": w.N, "d": w.d, "causal": w.causal, "window": w.window, "alibi": w.alibi,
                   "varlen": w.varlen, "o_dtype": "fp32", "flops_per_step": fl,
                   "attention_only_tflops": round(ach, 1), "l2": l2_note(w, T),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "per_kernel": {"fp8_quantize": {"ms": round(q_ms, 4), "share": round(q_ms / (q_ms + a_ms), 4)},
                       "fwd_fp8": {"ms": round(a_ms, 4), "tflops": round(ach, 1),
                                   "share": round(a_ms / (q_ms + a_ms), 4)}},
        "roofline": {"kernel": "fwd_fp8", "bound": "tensor", "achieved": round(ach, 1),
                     "peak": round(peak, 1), "unit": "TFLOP/s", "frac": round(ach / peak, 4),
                     "peak_source": f"{src} bf16 burst x {FP8_OVER_BF16:g} (nominal e4m3 / bf16 ratio)",
                     "traffic": ncu_traffic(w.name + " fp8", "fwd_fp8")},
        "gpu_launches": 4 * args.steps,
        "clocks": clocks, "e2e": e2e,
        "cpu_baseline": (oracle_fp8_baseline(w, x, I.hadamard_signs(w.d, seed=0))
                         if rank == 0 and not args.no_cpu_baseline else None),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- ours

def run_ours(args, world, rank, local):
    import torch
    from exact_io_aware_36_gb300 import fa

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = I.workload(args.workload)
    x = I.make_inputs(w, seed=0)
    fl = flops_per_step(w, x.seqlens)
    T = x.T

    fp32 = w.dtype == "fp32"          # c1: fp32 operands, forward only
    in_dtype = fa.FA_FP32 if fp32 else fa.FA_BF16

    def host(name):
        if fp32:
            return torch.from_numpy(np.ascontiguousarray(getattr(x, name), dtype=np.float32))
        return torch.from_numpy(x.bits[name].view("int16")).view(torch.bfloat16)

    def todev(name):
        return host(name).to(dev)

    q, k, v = todev("q"), todev("k"), todev("v")
    do = todev("do") if w.backward else None
    o = torch.empty(q.shape, dtype=torch.float32, device=dev)
    lse = torch.empty((w.Hq, T), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    cu = torch.from_numpy(x.cu_seqlens).to(dev) if w.varlen else None
    slopes = torch.from_numpy(x.alibi_slopes).to(dev) if w.alibi else None
    ws_bytes = fa.fa_bwd_workspace_size_gqa(w.B, w.Hq, w.Hkv, w.N, w.d, T)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    P = lambda t: None if t is None else t.data_ptr()
    common = (w.B, w.Hq, w.Hkv, w.N, w.d, float(x.scale), int(w.causal), w.window_arg, P(cu), T,
              P(slopes))
    ptrs = (P(q), P(k), P(v), P(o), P(do), P(lse), P(dq), P(dk), P(dv))
    det = 1 if args.deterministic else 0
    # grouped-query problems split their dK/dV items when the workspace has
    # room for the per-part sums; stage 2 then also adds the parts up
    kv_split = fa.fa_bwd_dkdv_split(w.B, w.Hq, w.Hkv, w.N, w.d, w.causal, w.window_arg,
                                    P(cu), ws_bytes) if w.backward else 1
    names = ["fwd", "bwd_preprocess", "bwd_dkdv",
             ("bwd_dq" if det else "bwd_dq_convert") + ("+dkdv_convert" if kv_split > 1 else "")]

    def step(evs=None, ptrs=ptrs):
        if evs is not None:
            evs[0].record(stream)
        st = fa.fa_fwd(ptrs[0], ptrs[1], ptrs[2], ptrs[3], ptrs[5], *common, in_dtype,
                       fa.FA_FP32, sp)
        if st:
            raise fa.FAError(st, "fa_fwd")
        if not w.backward:
            if evs is not None:
                evs[1].record(stream)
            return
        for s in range(3):
            if evs is not None:
                evs[1 + s].record(stream)
            st = fa.fa_bwd_stage(s, *ptrs, *common, fa.FA_BF16, fa.FA_FP32, det, P(ws), ws_bytes,
                                 sp)
            if st:
                raise fa.FAError(st, "fa_bwd_stage")
        if evs is not None:
            evs[4].record(stream)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize(dev)
    st = fa.fa_check_device_error(sp)
    if st:
        raise fa.FAError(st, "warm-up")

    nev = 5 if w.backward else 2
    evsets = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]
    flush = None
    if input_mb(w, T) * 1e6 <= L2_BYTES:
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(smi_index(local))
    sampler.start()
    time.sleep(0.1)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        step(evsets[i])
    end.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    st = fa.fa_check_device_error(sp)
    if st:
        raise fa.FAError(st, "timed region")
    if flush is None:
        local_ms = start.elapsed_time(end)
    else:
        local_ms = sum(e[0].elapsed_time(e[-1]) for e in evsets)
    total_ms = max_over_ranks(local_ms, world, dev)
    ms_step = total_ms / args.steps
    value = job_throughput(fl["total"], ms_step, world)

    kern_ms = {}
    for j, name in enumerate(names[:nev - 1]):
        kern_ms[name] = statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evsets)
    # FLOPs each kernel's MMAs must do: the default dK/dV kernel runs all
    # five backward products (10 d per pair); in the deterministic backward it
    # runs four (S, dP, dV, dK: 8 d) and the dQ kernel three (S, dP, dQ: 6 d).
    if det:
        kern_flops = {"fwd": fl["fwd"], "bwd_dkdv": 8.0 * w.d * fl["pairs"],
                      "bwd_dq": 6.0 * w.d * fl["pairs"]}
    else:
        kern_flops = {"fwd": fl["fwd"], "bwd_dkdv": fl["bwd"]}
    dom = max(kern_ms, key=lambda n: kern_ms[n])
    peak, hbm, peak_src = load_peaks()
    if fp32:
        # fp32 FMAs on the CUDA cores: 128 lanes x 2 flops per SM per clock
        ach = kern_flops["fwd"] / (kern_ms["fwd"] * 1e-3) / 1e12
        alu = fp32_fma_peak_tflops(dev)
        roof = {"kernel": "fwd_fp32", "bound": "alu", "achieved": round(ach, 3), "peak": alu,
                "unit": "TFLOP/s", "frac": round(ach / alu, 5),
                "peak_source": "derived: SMs x 128 fp32 FMA lanes x 2 flops x max SM clock",
                "note": "latency-bound at this size (one launch of a few microseconds)",
                "traffic": None}
    elif dom in kern_flops:
        ach = kern_flops[dom] / (kern_ms[dom] * 1e-3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": round(ach, 1), "peak": peak,
                "unit": "TFLOP/s", "frac": round(ach / peak, 4),
                "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json bf16_tflops)",
                "traffic": ncu_traffic(w.name + (" deterministic" if det else ""), dom)}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": None, "peak": hbm, "unit": "GB/s",
                "frac": None, "traffic": ncu_traffic(w.name + (" deterministic" if det else ""), dom)}
    per_kernel = {n: {"ms": round(kern_ms[n], 4),
                      "tflops": round(kern_flops[n] / (kern_ms[n] * 1e-3) / 1e12, 1)
                      if n in kern_flops else None,
                      "share": round(kern_ms[n] / sum(kern_ms.values()), 4)}
                  for n in kern_ms}
    fwd_tflops = fl["fwd"] / (kern_ms["fwd"] * 1e-3) / 1e12

    e2e = None
    if not args.no_e2e:
        # two buffer sets: step i's kernels use set i % 2 while set (i+1) % 2
        # takes the next step's inputs and gives back the previous outputs
        in_names = ["q", "k", "v"] + (["do"] if w.backward else [])
        sets = []
        for b in range(2):
            if b == 0:
                bq, bk, bv, bo, bdo, blse, bdq, bdk, bdv = q, k, v, o, do, lse, dq, dk, dv
            else:
                bq, bk, bv, bo, blse = (torch.empty_like(t) for t in (q, k, v, o, lse))
                bdo = torch.empty_like(do) if w.backward else None
                bdq, bdk, bdv = (torch.empty_like(t) for t in (dq, dk, dv))
            dev_in = [bq, bk, bv] + ([bdo] if w.backward else [])
            sets.append({"ins": dev_in,
                         "outs": [bo, blse] + ([bdq, bdk, bdv] if w.backward else []),
                         "ptrs": (P(bq), P(bk), P(bv), P(bo), P(bdo), P(blse), P(bdq), P(bdk),
                                  P(bdv))})
        e2e = run_e2e(args, fl, world, dev, stream, step, [host(n) for n in in_names], sets,
                      "fa_fwd + fa_bwd_stage x3" if w.backward else "fa_fwd", kernel_ms=ms_step)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, x)

    line = {
        "metric": FWD_FP32_METRIC if fp32 else METRIC, "value": round(value, 2 if not fp32 else 5),
        "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if fp32 else "bf16",
        "data": "synthetic (seeded PCG64, seed 0; no dataset)",
        "config": {"workload": w.name, "desc": w.note, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv,
                   "N": w.N, "d": w.d, "causal": w.causal, "window": w.window,
                   "deterministic_bwd": bool(det), "dkdv_split": kv_split,
                   "alibi": w.alibi, "varlen": w.varlen,
                   "total_tokens": T, "o_dtype": "fp32", "flops_per_step": fl["total"],
                   "pct_of_peak": None if fp32 else round(100.0 * value / world / peak, 2),
                   "fwd_tflops": round(fwd_tflops, 1 if not fp32 else 5),
                   "fwd_pct_of_peak": None if fp32 else round(100.0 * fwd_tflops / peak, 2),
                   "fwd_latency_us": round(kern_ms["fwd"] * 1e3, 2),
                   "l2": l2_note(w, T),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "per_kernel": per_kernel,
        "roofline": roof,
        "secondary_roofs": None if fp32 else secondary_roofs(w, T, fl, kern_ms, dev, hbm, bool(det)),
        "gpu_launches": args.steps * ((5 if kv_split > 1 and det else 4) if w.backward else 1),
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def gpu_numa_cpus(dev):
    """(NUMA node of the GPU, the CPUs of that node this process may use), from
    sysfs; (None, None) when either is unknown."""
    import torch
    try:
        pr = torch.cuda.get_device_properties(dev)
        bus = f"{pr.pci_domain_id:04x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
        node = int(open(f"/sys/bus/pci/devices/{bus}/numa_node").read().strip())
        if node < 0:
            return None, None
        cpus = set()
        for part in open(f"/sys/devices/system/node/node{node}/cpulist").read().strip().split(","):
            lo, _, hi = part.partition("-")
            cpus.update(range(int(lo), int(hi or lo) + 1))
        cpus &= os.sched_getaffinity(0)
        return node, sorted(cpus) if cpus else None
    except (OSError, ValueError, AttributeError):
        return None, None


def copy_rates(dev, hins, dins, houts, douts, s_in, s_out, reps=3):
    """GB/s of one step's input copies alone (host to device), output copies
    alone (device to host), and both at once on their two streams."""
    import torch
    bi = sum(h.numel() * h.element_size() for h in hins)
    bo = sum(h.numel() * h.element_size() for h in houts)

    def timed(do_in, do_out):
        best = None
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            a = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            a[0].record(s_in)
            a[2].record(s_out)
            if do_in:
                with torch.cuda.stream(s_in):
                    for d, h in zip(dins, hins):
                        d.copy_(h, non_blocking=True)
            if do_out:
                with torch.cuda.stream(s_out):
                    for h, d in zip(houts, douts):
                        h.copy_(d, non_blocking=True)
            a[1].record(s_in)
            a[3].record(s_out)
            torch.cuda.synchronize(dev)
            ms = max(a[0].elapsed_time(a[1]) if do_in else 0.0,
                     a[2].elapsed_time(a[3]) if do_out else 0.0)
            best = ms if best is None else min(best, ms)
        return best

    t_in, t_out, t_both = timed(True, False), timed(False, True), timed(True, True)
    return {"h2d_gbs": round(bi / (t_in * 1e-3) / 1e9, 1), "d2h_gbs": round(bo / (t_out * 1e-3) / 1e9, 1),
            "both_gbs": round((bi + bo) / (t_both * 1e-3) / 1e9, 1),
            "h2d_ms": round(t_in, 3), "d2h_ms": round(t_out, 3), "both_ms": round(t_both, 3)}


def run_e2e(args, fl, world, dev, stream, step, host_ins, sets, calls, kernel_ms=None):
    """Same metric through the C ABI with host buffers: every step copies its
    inputs from pinned host memory and its outputs back to pinned host
    memory, and all of those copies are inside the timed region.  The steps
    are pipelined as a serving loop would run them: step i's kernels (on the
    compute stream, buffer set i % 2) overlap the copy of step i+1's inputs
    (copy-in stream) and of step i-1's outputs (copy-out stream).  A set is
    refilled only after the kernels that read it are done, and overwritten
    only after its outputs have been copied out.

    The pinned buffers are allocated with the process bound to the CPUs of
    the GPU's NUMA node (where the system says which that is), so that their
    pages are local to the GPU's host link.  The copy rates of one step's
    inputs and outputs, alone and together, are measured beside the timed
    steps; with the kernels' own time they say how much of the copying the
    pipeline hid."""
    import torch
    node, cpus = gpu_numa_cpus(dev)
    old_aff = os.sched_getaffinity(0)
    if cpus:
        os.sched_setaffinity(0, cpus)
    try:
        hins = [h.pin_memory() for h in host_ins]
        houts = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in sets[0]["outs"]]
        for h in houts:
            h.zero_()                                  # touch the pages on this node
    finally:
        if cpus:
            os.sched_setaffinity(0, old_aff)
    h2d = sum(h.numel() * h.element_size() for h in hins)
    d2h = sum(h.numel() * h.element_size() for h in houts)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    rates = copy_rates(dev, hins, sets[1]["ins"], houts, sets[1]["outs"], s_in, s_out)
    comp_done, out_done = [None, None], [None, None]

    def run(n):
        for i in range(n):
            b = i & 1
            S = sets[b]
            if comp_done[b] is not None:              # kernels of step i-2 read set b
                s_in.wait_event(comp_done[b])
            with torch.cuda.stream(s_in):
                for d, h in zip(S["ins"], hins):
                    d.copy_(h, non_blocking=True)
            in_ev = torch.cuda.Event()
            in_ev.record(s_in)
            stream.wait_event(in_ev)
            if out_done[b] is not None:               # outputs of step i-2 copied out
                stream.wait_event(out_done[b])
            step(None, S["ptrs"])
            ce = torch.cuda.Event()
            ce.record(stream)
            comp_done[b] = ce
            s_out.wait_event(ce)
            with torch.cuda.stream(s_out):
                for d, h in zip(S["outs"], houts):
                    h.copy_(d, non_blocking=True)
            oe = torch.cuda.Event()
            oe.record(s_out)
            out_done[b] = oe

    run(2)
    torch.cuda.synchronize(dev)
    n = max(3, args.steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    run(n)
    stream.wait_event(out_done[(n - 1) & 1])       # the copy-out stream runs in order
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / n
    out = {"value": round(world * fl["total"] / (ms * 1e-3) / 1e9 / 1e3, 2 if fl["total"] > 1e9 else 5),
           "unit": UNIT, "ms_per_step": round(ms, 3), "steps": n, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "copy_rates": rates,
           "pinned_numa_node": node, "pinned_bound_cpus": len(cpus) if cpus else None,
           "path": calls + " through the C ABI; pinned host buffers; copies of step i+1's inputs "
                   "and step i-1's outputs overlap step i's kernels (three streams, two buffer sets)"}
    if kernel_ms is not None:
        # Without overlap a step would take kernels + both copies; fully
        # overlapped, the larger of the kernels and the concurrent copies.
        serial = kernel_ms + rates["h2d_ms"] + rates["d2h_ms"]
        hidden = max(kernel_ms, rates["both_ms"])
        out["kernel_ms_per_step"] = round(kernel_ms, 3)
        out["serial_ms_per_step"] = round(serial, 3)
        out["overlapped_bound_ms"] = round(hidden, 3)
        out["copy_hidden_frac"] = round(min(1.0, max(0.0, (serial - ms) / max(serial - hidden, 1e-9))), 3)
    return out


# ---------------------------------------------------------------- CPU oracle

ORACLE_SAMPLE_TOKENS = 8192


def oracle_sample(w: I.Workload, x):
    """One whole (sequence, query head) of the workload, forward + backward
    in fp64, with the oracle as it stands."""
    from oracle import attention_fp64 as A
    s, e = int(x.cu_seqlens[0]), int(x.cu_seqlens[1])
    h, g = 0, 0
    slope = None if x.alibi_slopes is None else float(x.alibi_slopes[h])
    what = f"1 of {w.B * w.Hq} (sequence, query head) pairs: sequence 0 (L={e - s}), head 0"
    if w.window is not None and e - s > ORACLE_SAMPLE_TOKENS:
        # a causal prefix is a problem of its own; the oracle's dense S and P
        # of a whole 32k head would not fit the host
        e = s + ORACLE_SAMPLE_TOKENS
        what += f", its first {ORACLE_SAMPLE_TOKENS} tokens"
    L = e - s
    pairs = I.attended_pairs(dataclasses.replace(w, B=1, Hq=1, seqlens=None, seqlen_range=None),
                             [L])
    t0 = time.perf_counter()
    if w.backward:
        A.head_backward(x.q[s:e, h], x.k[s:e, g], x.v[s:e, g], x.do[s:e, h], x.scale, w.causal,
                        slope, window=w.window)
    else:
        A.head_forward(x.q[s:e, h], x.k[s:e, g], x.v[s:e, g], x.scale, w.causal, slope,
                       window=w.window)
    dt = time.perf_counter() - t0
    flops = (14.0 if w.backward else 4.0) * w.d * pairs
    return flops, dt, what


def oracle_fp8_baseline(w, x, signs):
    """One whole (sequence, query head) of the workload through the FP8
    oracle: transform, block quantization and attention on the dequantized
    values, in fp64."""
    from oracle import fp8 as F
    s, e = int(x.cu_seqlens[0]), int(x.cu_seqlens[1])
    L = e - s
    cu = np.array([0, L], dtype=np.int64)
    slopes = None if x.alibi_slopes is None else x.alibi_slopes[:1]
    t0 = time.perf_counter()
    qz = F.quantize_inputs(x.q[s:e, :1], x.k[s:e, :1], x.v[s:e, :1], signs, cu, L)
    F.attention_forward_fp8(qz, cu, L, x.scale, w.causal, slopes, window=w.window)
    dt = time.perf_counter() - t0
    pairs = I.attended_pairs(dataclasses.replace(w, B=1, Hq=1, seqlens=None, seqlen_range=None),
                             [L])
    return {"value": round(4.0 * w.d * pairs / dt / 1e12, 6), "unit": UNIT,
            "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"1 of {w.B * w.Hq} (sequence, query head) pairs: sequence 0 (L={L}), head 0",
            "seconds": round(dt, 2),
            "note": "NumPy: float32 transform and e4m3 codes, float64 attention on the "
                    "dequantized values; BLAS threads = all cores"}


def cpu_baseline(w, x):
    fl, dt, sample = oracle_sample(w, x)
    return {"value": round(fl / dt / 1e12, 6), "unit": UNIT, "cores": os.cpu_count(),
            "kind": "oracle", "sample": sample, "seconds": round(dt, 2),
            "note": "NumPy float64, materialises S and P; BLAS threads = all cores"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    if args.workload in I.DECODE_WORKLOADS:
        w = I.DECODE_WORKLOADS[args.workload]
        x = I.make_decode_inputs(w, seed=0)
        sample_fn, metric, unit, scale = oracle_decode_sample, DECODE_METRIC, "GB/s", 1e9
        shape = {"B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S_max": w.S_max, "d": w.d, "q_len": w.q_len,
                 "step": "all query rows of one sequence of the decode step per step"}
    else:
        w = I.workload(args.workload)
        x = I.make_inputs(w, seed=0)
        sample_fn, unit, scale = oracle_sample, UNIT, 1e12
        metric = FWD_FP32_METRIC if w.dtype == "fp32" else METRIC
        shape = {"B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": w.d, "causal": w.causal,
                 "step": "one (sequence, head) sample of the workload per step"}
    for _ in range(max(args.warmup, 0)):
        sample_fn(w, x)
    tot_fl, tot_dt, sample = 0.0, 0.0, ""
    for _ in range(args.steps):
        fl, dt, sample = sample_fn(w, x)
        tot_fl += fl
        tot_dt += dt
    value = tot_fl / tot_dt / scale
    line = {
        "metric": metric, "value": round(value, 6), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot_dt / max(args.steps, 1), 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded PCG64, seed 0; no dataset)", "impl": "reference",
        "config": {"workload": w.name, "desc": w.note, **shape},
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": os.cpu_count(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.record_traffic:
        print(json.dumps({traffic_key(args): record_traffic(args.record_traffic, traffic_key(args))}))
        return
    world, rank, local = dist_info()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    try:
        if args.workload in I.DECODE_WORKLOADS:
            run_decode(args, world, rank, local)
        elif args.fp8:
            run_fp8(args, world, rank, local)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
