#!/usr/bin/env python3
"""Benchmark of the FP8 (E4M3) fine-grained-scaled GEMM on GB300.

Workload (one "step"): the dense FP8 GEMM sweep — M in {64, 128, 4096} x (N, K) in {(2112, 7168),
(24576, 1536), (32768, 512), (7168, 16384), (4096, 7168), (7168, 2048)}, A[M,K] and B[N,K] drawn
N(0,1) from seed 0 and quantised to E4M3 (1x128 A scales, 128x128 B scales, amax/448), BF16 D.
Each of the 18 GEMMs is one launch of the sm_103a kernel through the C ABI; an L2 flush precedes
every GEMM and lies outside the CUDA events that time it: a write of a 256 MB buffer, then a read of
a second 256 MB buffer, so that the write's dirty lines have reached HBM (and L2 holds only clean,
unrelated lines) when the GEMM starts.

Metric: useful TFLOP/s = sum(2*M*N*K) / sum(GEMM time). Printed as one JSON line with the
roofline of the dominant kernel, the CPU oracle baseline, the end-to-end number through host
buffers, the SM clocks seen during the timed region and the number of kernel launches.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--scales fp32|ue8m0]

``--scales ue8m0`` runs the same workload with power-of-two scales (the smallest 2^p >= amax/448)
packed as UE8M0 words through the block-scaled entry points; the default, fp32, is the amax/448
FP32-scale GEMM with CUDA-core promotion.

Multi-GPU (torchrun, one rank per GPU): every rank runs the same sweep on its own GPU (replicas,
weak scaling); rank 0 prints the whole-job throughput using the slowest rank's time.
``--impl reference`` times the CPU oracle (the only reference this method has) on a bounded sample
of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

SWEEP_NK = [(2112, 7168), (24576, 1536), (32768, 512), (7168, 16384), (4096, 7168), (7168, 2048)]
SWEEP_M = [64, 128, 4096]
SHAPES = [(M, N, K) for M in SWEEP_M for (N, K) in SWEEP_NK]
WORKLOAD = "dense FP8 E4M3 GEMM sweep, M in {64,128,4096} x (N,K) in {(2112,7168),(24576,1536),(32768,512),(7168,16384),(4096,7168),(7168,2048)}"
METRIC = "FP8 TFLOPS (2MNK/s) per shape; % of GB300 FP8 dense peak or HBM GB/s"
L2_FLUSH_BYTES = 256 << 20
L2_NOTE = ("flushed before every GEMM, outside its CUDA events: a 256 MB write, then a 256 MB read of a "
           "second buffer (the write's dirty lines reach HBM before the GEMM starts)")
CPU_SAMPLE_PER_SHAPE = 196608
UE8M0 = False      # set by --scales ue8m0


class L2Flush:
    """Evicts the GEMM's operands from L2: writes a buffer larger than L2, then reads another one, so
    that the eviction's write-back of dirty lines happens here and not inside the timed GEMM."""

    def __init__(self):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.r = torch.zeros(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def __call__(self, i):
        import torch
        self.w.fill_(i & 0xFF)
        self.sink = self.r.view(torch.float32).sum()   # one reduction kernel reading 256 MB (zeros)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per_config entries (configs 1, 3, 4 and 5 timed after the sweep)")
    ap.add_argument("--cpu-sample", type=int, default=CPU_SAMPLE_PER_SHAPE)
    ap.add_argument("--all-configs", action="store_true",
                    help="time every workload configuration (dense small, sweep, contiguous, masked, stress) "
                         "and print one JSON line per shape instead of the benchmark line")
    ap.add_argument("--configs", default=None,
                    help="with --all-configs: only these configuration numbers (comma-separated), e.g. 4")
    ap.add_argument("--shapes", default=None,
                    help="restrict the sweep to these MxNxK shapes (comma-separated), e.g. for profiling")
    ap.add_argument("--scales", choices=["fp32", "ue8m0"], default="fp32",
                    help="fp32: amax/448 FP32 scales (CUDA-core promotion); ue8m0: power-of-two scales packed "
                         "as UE8M0 (block-scaled tensor-core kernel)")
    args = ap.parse_args()
    global UE8M0
    UE8M0 = args.scales == "ue8m0"
    if args.shapes:
        global SHAPES
        SHAPES = [tuple(int(v) for v in s.lower().split("x")) for s in args.shapes.split(",")]
    return args


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                "sm_mhz_median": (pk.get("clocks_under_load") or {}).get("sm_mhz_median"),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def algorithmic_bytes(M, N, K):
    """Bytes one dense GEMM must move: A, B, their scales (FP32, or UE8M0 packed four K-groups
    to an int32) and the BF16 D."""
    nkb, nnb = -(-K // 128), -(-N // 128)
    nks = -(-nkb // 4) if UE8M0 else nkb
    return M * K + N * K + 4 * M * nks + 4 * nnb * nks + 2 * M * N


def gpu_scales(a, b):
    """The scale arrays a GEMM call takes: FP32, or packed UE8M0 words."""
    import dg_inputs
    if UE8M0:
        return dg_inputs.pack_ue8m0_a(a.sA), dg_inputs.pack_ue8m0_b(b.sB)
    return a.sA, b.sB


def gemm_entry(dg, kind="dense"):
    names = {"dense": "dg_fp8_gemm_nt", "contiguous": "dg_fp8_grouped_contiguous", "masked": "dg_fp8_grouped_masked"}
    return getattr(dg, names[kind] + ("_ue8m0" if UE8M0 else ""))


def query_config(dg, *a):
    return (dg.dg_query_config_ue8m0 if UE8M0 else dg.dg_query_config)(*a)


def quantisation_note():
    if UE8M0:
        return "E4M3, A 1x128 / B 128x128 power-of-two scales (smallest 2^p >= amax/448), packed UE8M0"
    return "E4M3, A 1x128 / B 128x128 FP32 scales, amax/448"


def measured_traffic(shape: str):
    """DRAM bytes (read + write) of one launch of `shape`, from the committed ncu summary, or None
    when the kernel sources have changed since those counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    h = hashlib.sha256()
    for src in rec.get("sources", []):
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != rec.get("source_sha256"):
        return None
    launch = rec.get("launches_ue8m0" if UE8M0 else "launches", {}).get(shape)
    if not launch:
        return None
    return int(launch["dram_read_bytes"] + launch["dram_write_bytes"])


def slowest_rank(value: float, pg) -> float:
    """The largest `value` over all ranks, returned on every rank (the job's time is its slowest
    rank's); `value` itself without a process group. NCCL reduces on the GPU, gloo on the host."""
    if pg is None:
        return value
    import torch
    device = "cuda" if pg.get_backend() == "nccl" else "cpu"
    x = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(x, op=pg.ReduceOp.MAX)
    return float(x.item())


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ---------------------------------------------------------------------------------------------
# Inputs


def make_inputs():
    import dg_inputs
    a_cache, b_cache, out = {}, {}, []
    for (M, N, K) in SHAPES:
        if (M, K) not in a_cache:
            a_cache[(M, K)] = dg_inputs.make_a(M, K, seed=0, ue8m0=UE8M0)
        if (N, K) not in b_cache:
            b_cache[(N, K)] = dg_inputs.make_b(1, N, K, seed=0, ue8m0=UE8M0)
        out.append((M, N, K, a_cache[(M, K)], b_cache[(N, K)]))
    return out


# ---------------------------------------------------------------------------------------------
# Clock sampling during the timed region


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        self.gpu_id = gpu_id
        self._thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self._thread = threading.Thread(target=self._read, daemon=True)
        self._thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=2)

    def summary(self, t0, t1):
        window = [s for (t, s) in self.samples if t0 <= t <= t1]
        if not window and self.samples:   # a very short timed region: take the samples around it
            window = [min(self.samples, key=lambda ts: abs(ts[0] - (t0 + t1) / 2))[1]]
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[0]) for s in window if num(s[0]) is not None]
        smax = [num(s[1]) for s in window if num(s[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in window:
            for name, v in zip(names, s[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(window),
                "power_w_max": max((num(s[2]) or 0.0) for s in window)}


def gpu_id_for_smi(device_index: int) -> str:
    import torch
    try:
        props = torch.cuda.get_device_properties(device_index)
        bus = getattr(props, "pci_bus_id", None)
        dom = getattr(props, "pci_domain_id", None)
        dev = getattr(props, "pci_device_id", None)
        if bus is not None and dom is not None and dev is not None:
            return f"{dom:08x}:{bus:02x}:{dev:02x}.0"
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return vis.split(",")[device_index]
    return str(device_index)


# ---------------------------------------------------------------------------------------------
# Our arm


def run_ours(args, rank, world, local):
    import torch
    import moe_grouped_gemm_e4m3_gb300 as dg

    torch.cuda.set_device(local)
    dg.load()
    pg = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        pg = tdist

    problems = make_inputs()
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    tensors = []
    gemm = gemm_entry(dg)
    for (M, N, K, a, b) in problems:
        gsA, gsB = gpu_scales(a, b)
        tensors.append(dict(M=M, N=N, K=K, A=dev(a.A), sA=dev(gsA), B=dev(b.B[0]), sB=dev(gsB[0]),
                            D=torch.empty(M, N, dtype=torch.bfloat16, device="cuda"),
                            cfg=query_config(dg, 0, M, N, K)))
    flush = L2Flush()
    stream = torch.cuda.current_stream()

    def one_step(events):
        for i, t in enumerate(tensors):
            flush(i)
            if events is not None:
                events[i][0].record(stream)
            gemm(t["A"], t["sA"], t["B"], t["sB"], t["D"], stream)
            if events is not None:
                events[i][1].record(stream)

    for _ in range(args.warmup):
        one_step(None)
    torch.cuda.synchronize()
    status = dg.dg_get_device_status()
    if status:
        raise RuntimeError(f"device status 0x{status:x} after warm-up")

    sampler = ClockSampler(gpu_id_for_smi(local)) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    ev = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in tensors]
          for _ in range(args.steps)]
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for s in range(args.steps):
        one_step(ev[s])
    torch.cuda.synchronize()
    t1 = time.time()
    if pg:
        pg.barrier()
    if sampler:
        time.sleep(0.1)
        sampler.stop()
    per_shape_ms = np.array([[ev[s][i][0].elapsed_time(ev[s][i][1]) for i in range(len(tensors))]
                             for s in range(args.steps)])   # [steps, shapes]
    ms_per_step_local = float(per_shape_ms.sum(axis=1).mean())
    ms_per_step = slowest_rank(ms_per_step_local, pg)
    status = dg.dg_get_device_status()
    if status:
        raise RuntimeError(f"device status 0x{status:x} after the timed region")

    flops_step = sum(2.0 * t["M"] * t["N"] * t["K"] for t in tensors)
    value = world * flops_step / (ms_per_step * 1e-3) / 1e12

    # The floor of this timing method: an empty kernel (torch.cuda._sleep(0)) between the same pair
    # of events after the same L2 flush. Short, HBM-bound launches spend a fixed part of their
    # event time on it.
    floor = []
    for r in range(max(5, args.steps)):
        flush(r)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        torch.cuda._sleep(0)
        e1.record(stream)
        torch.cuda.synchronize()
        floor.append(e0.elapsed_time(e1) * 1e3)
    floor_us = float(np.median(floor))

    # e2e through host buffers (pinned), copies inside the timed region
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(dg, problems, args, stream)
        if pg:
            e2e["value"] = world * flops_step / (slowest_rank(e2e["ms_per_step"], pg) * 1e-3) / 1e12

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return

    peaks = load_peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops"]           # dense FP8 = 2x dense BF16 (nominal ratio)
    mean_ms = per_shape_ms.mean(axis=0)
    per_shape = []
    for i, t in enumerate(tensors):
        M, N, K = t["M"], t["N"], t["K"]
        tflops = 2.0 * M * N * K / (mean_ms[i] * 1e-3) / 1e12
        gbs = algorithmic_bytes(M, N, K) / (mean_ms[i] * 1e-3) / 1e9
        t_tc = 2.0 * M * N * K / (fp8_peak * 1e12)
        t_hbm = algorithmic_bytes(M, N, K) / (peaks["hbm_gbs"] * 1e9)
        bound = "tensor" if t_tc >= t_hbm else "hbm"
        frac = (tflops / fp8_peak) if bound == "tensor" else (gbs / peaks["hbm_gbs"])
        entry = {"M": M, "N": N, "K": K, "us": round(float(mean_ms[i]) * 1e3, 2), "tflops": round(tflops, 1),
                 "gbs": round(gbs, 1), "bound": bound, "roof_frac": round(frac, 3),
                 "block_n": t["cfg"]["block_n"], "splits": t["cfg"]["splits"]}
        if bound == "hbm" and mean_ms[i] * 1e3 > floor_us:
            # the same fraction with the empty-kernel floor taken out of the event time
            entry["roof_frac_above_floor"] = round(algorithmic_bytes(M, N, K) / ((mean_ms[i] * 1e3 - floor_us) * 1e-6) / 1e9
                                                   / peaks["hbm_gbs"], 3)
        per_shape.append(entry)
    # Dominant kernel: the instantiation (tile width, split-K or not) with the largest share of the
    # step. Its roofline is reported for its longest launch (per-launch figures, as ncu sees them).
    groups = {}
    for i, t in enumerate(tensors):
        key = (t["cfg"]["block_n"], t["cfg"]["splits"] > 1)
        g = groups.setdefault(key, {"ms": 0.0, "flops": 0.0, "launches": []})
        g["ms"] += float(mean_ms[i])
        g["flops"] += 2.0 * t["M"] * t["N"] * t["K"]
        g["launches"].append(i)
    dom_key = max(groups, key=lambda k: groups[k]["ms"])
    dom = groups[dom_key]
    li = max(dom["launches"], key=lambda i: float(mean_ms[i]))
    lt = tensors[li]
    shape = f"{lt['M']}x{lt['N']}x{lt['K']}"
    l_ms = float(mean_ms[li])
    l_flops = 2.0 * lt["M"] * lt["N"] * lt["K"]
    l_bytes = algorithmic_bytes(lt["M"], lt["N"], lt["K"])
    kname = (f"fp8_gemm_bs_kernel<dense,bf16> ({'split-K' if dom_key[1] else 'no split'}, BN=256)" if UE8M0 else
             f"fp8_gemm_kernel<BN={dom_key[0]},{'split-K' if dom_key[1] else 'no split'},dense,bf16>")
    if l_flops / (fp8_peak * 1e12) >= l_bytes / (peaks["hbm_gbs"] * 1e9):
        achieved = l_flops / (l_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                "frac": round(achieved / fp8_peak, 4)}
    else:
        achieved = l_bytes / (l_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4)}
    roof.update({"traffic": measured_traffic(shape), "kernel": kname, "launch": shape,
                 "launch_share_of_step": round(l_ms / float(mean_ms.sum()), 3),
                 "kernel_share_of_step": round(dom["ms"] / float(mean_ms.sum()), 3),
                 "kernel_achieved_all_launches": round(dom["flops"] / (dom["ms"] * 1e-3) / 1e12, 1),
                 "peak_source": f"{peaks['source']}: 2 x bf16_tflops (dense FP8 = 2x BF16 nominal)"})

    clocks = sampler.summary(t0, t1) if sampler else None
    # The measured peak was taken under the power cap at a lower SM clock than the bench usually
    # runs at; the same peak scaled to the bench's median clock shows how much of the fraction is
    # clock, not kernel (a tensor-bound kernel's rate scales with the SM clock; HBM does not).
    pk_mhz = peaks.get("sm_mhz_median")
    if roof["bound"] == "tensor" and pk_mhz and clocks and clocks.get("sm_mhz"):
        scaled = fp8_peak * clocks["sm_mhz"] / pk_mhz
        roof.update({"peak_sm_mhz": pk_mhz, "bench_sm_mhz": clocks["sm_mhz"],
                     "peak_at_bench_clock": round(scaled, 1), "frac_at_bench_clock": round(roof["achieved"] / scaled, 4)})

    per_config, per_config_s = None, None
    if not args.no_per_config and world == 1:
        tp = time.time()
        per_config = per_config_measure(dg, max(3, min(args.steps, 10)))
        per_config_s = round(time.time() - tp, 1)

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(problems, args.cpu_sample)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "data": "synthetic",
        "dtype": ("e4m3 x e4m3 block-scaled by ue8m0 -> f32 accumulate -> bf16" if UE8M0 else
                  "e4m3 x e4m3 -> f32 accumulate (fine-grained scales) -> bf16"),
        "config": {"workload": WORKLOAD if len(tensors) == 18 else f"subset {SHAPES}", "shapes": len(tensors), "seed": 0, "values": "N(0,1)",
                   "quantisation": quantisation_note(),
                   "l2": L2_NOTE,
                   "e2e": ("every step: H2D of each GEMM's A, sA, B, sB from pinned host memory, the GEMM, D2H "
                           "of D to pinned host memory; copies on two copy streams, overlapping the GEMMs"),
                   "parallelism": f"replicas x{world}", "wall_ms_per_step": round((t1 - t0) * 1e3 / args.steps, 4)},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": ({k: e2e[k] for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step", "host_buffers_pinned")}
                if e2e else None),
        "clocks": clocks,
        "gpu_launches": len(tensors) * args.steps,
        "launch_floor_us": round(floor_us, 2),
        "per_shape": per_shape,
        "per_config": per_config,
        "per_config_wall_s": per_config_s,
    }
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


def per_config_measure(dg, reps):
    """The workload configurations other than the sweep, each timed like the sweep's GEMMs (CUDA
    events around the launch, L2 flushed before each repetition, mean over `reps`): config 1 (dense
    128x512x1024), config 3 (contiguous grouped, G = 4 and 8, 8192 rows a group), config 4 (masked
    decode, G = 16, M_max = 256) and config 5 (Student-t inputs with outlier channels). Returns one
    entry per shape: time, TFLOP/s, algorithmic GB/s, the binding roof and the fraction of it."""
    import torch
    import dg_inputs
    peaks = load_peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    flush = L2Flush()
    out = []

    def timeit(fn):
        fn()
        ts = []
        for r in range(reps):
            flush(r)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return float(np.mean(ts))

    def add(config, shape, flops, nbytes, ms, cfg=None):
        t_tc, t_hbm = flops / (fp8_peak * 1e12), nbytes / (peaks["hbm_gbs"] * 1e9)
        bound = "tensor" if t_tc >= t_hbm else "hbm"
        tflops, gbs = flops / (ms * 1e-3) / 1e12, nbytes / (ms * 1e-3) / 1e9
        frac = tflops / fp8_peak if bound == "tensor" else gbs / peaks["hbm_gbs"]
        e = {"config": config, "shape": shape, "us": round(ms * 1e3, 2), "tflops": round(tflops, 1),
             "gbs": round(gbs, 1), "bound": bound, "roof_frac": round(frac, 3)}
        if cfg:
            e.update({"block_n": cfg["block_n"], "splits": cfg["splits"]})
        out.append(e)

    def nks(K):
        nkb = -(-K // 128)
        return -(-nkb // 4) if UE8M0 else nkb

    def dense(config, M, N, K, dist=dg_inputs.NORMAL, outliers=0.0):
        a = dg_inputs.make_a(M, K, seed=0, dist=dist, outlier_frac=outliers, ue8m0=UE8M0)
        b = dg_inputs.make_b(1, N, K, seed=0, dist=dist, ue8m0=UE8M0)
        gsA, gsB = gpu_scales(a, b)
        A, sA, B, sB = dev(a.A), dev(gsA), dev(b.B[0]), dev(gsB[0])
        D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        gemm = gemm_entry(dg)
        ms = timeit(lambda: gemm(A, sA, B, sB, D))
        add(config, f"{M}x{N}x{K}", 2.0 * M * N * K, algorithmic_bytes(M, N, K), ms, query_config(dg, 0, M, N, K))

    dense("1 dense small", 128, 512, 1024)
    # config 3: the G = 4 problem is the first four groups of the G = 8 one
    for (N, K) in ((4096, 7168), (7168, 2048)):
        a8 = dg_inputs.make_a(8 * 8192, K, seed=0, ue8m0=UE8M0)
        b8 = dg_inputs.make_b(8, N, K, seed=0, ue8m0=UE8M0)
        gsA8, gsB8 = gpu_scales(a8, b8)
        for G in (4, 8):
            M = G * 8192
            A, B = dev(a8.A[:M]), dev(b8.B[:G])
            sA, sB = dev(np.ascontiguousarray(gsA8[:, :M])), dev(gsB8[:G])
            idx = dev(np.repeat(np.arange(G, dtype=np.int32), 8192))
            D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
            gemm = gemm_entry(dg, "contiguous")
            ms = timeit(lambda: gemm(A, sA, B, sB, idx, D))
            nbytes = M * K + G * N * K + 4 * M * nks(K) + 4 * G * (-(-N // 128)) * nks(K) + 2 * M * N
            add("3 contiguous", f"G={G} M={M} N={N} K={K}", 2.0 * M * N * K, nbytes, ms, query_config(dg, 1, M, N, K, G))
            del A, B, D
        del a8, b8
    for (N, K) in ((4096, 7168), (7168, 2048)):
        G, M_max = 16, 256
        mm = dg_inputs.make_masked_m(G, M_max, seed=0)
        a = dg_inputs.make_masked_a(G, M_max, K, seed=0, ue8m0=UE8M0)
        b = dg_inputs.make_b(G, N, K, seed=0, ue8m0=UE8M0)
        gsA, gsB = gpu_scales(a, b)
        A, sA, B, sB, MM = dev(a.A), dev(gsA), dev(b.B), dev(gsB), dev(mm)
        D = torch.empty(G, M_max, N, dtype=torch.bfloat16, device="cuda")
        gemm = gemm_entry(dg, "masked")
        ms = timeit(lambda: gemm(A, sA, B, sB, MM, D))
        valid, active = int(mm.sum()), int((mm > 0).sum())
        nbytes = valid * K + active * N * K + 4 * valid * nks(K) + 4 * G * (-(-N // 128)) * nks(K) + 2 * valid * N
        add("4 masked", f"G=16 M_max=256 sum(masked_m)={valid} N={N} K={K}", 2.0 * valid * N * K, nbytes, ms,
            query_config(dg, 2, M_max, N, K, G))
    for (M, N, K) in ((4096, 2112, 7168), (4096, 576, 7168), (4096, 7168, 32768)):
        dense("5 stress (Student-t, outliers)", M, N, K, dist=dg_inputs.STUDENT_T3, outliers=0.01)
    return out


def measure_e2e(dg, problems, args, stream):
    """Same sweep through host buffers: every step copies each GEMM's A, sA, B, sB from pinned host
    memory, runs the GEMM and copies D back to pinned host memory, all inside the timed region.
    The copies are pipelined across three streams (host-to-device, compute, device-to-host), so the
    two copy directions overlap each other and the GEMMs; a step ends when its last D is on the host."""
    import torch
    host = []
    h2d = d2h = 0
    gemm = gemm_entry(dg)
    for (M, N, K, a, b) in problems:
        h = dict(M=M, N=N, K=K)
        gsA, gsB = gpu_scales(a, b)
        for name, arr in (("A", a.A), ("sA", gsA), ("B", b.B[0]), ("sB", gsB[0])):
            ht = torch.from_numpy(np.ascontiguousarray(arr)).pin_memory()
            h[name] = ht
            h["d" + name] = torch.empty_like(ht, device="cuda")
            h2d += ht.numel() * ht.element_size()
        h["dD"] = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        h["D"] = torch.empty(M, N, dtype=torch.bfloat16).pin_memory()
        d2h += M * N * 2
        host.append(h)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    done = [torch.cuda.Event() for _ in host]       # the GEMM of shape i has finished (inputs read, D written)
    out_done = [torch.cuda.Event() for _ in host]   # D of shape i is on the host
    steps = max(3, min(args.steps, 10))

    def one_step():
        ev_in = []
        for i, h in enumerate(host):
            with torch.cuda.stream(s_in):
                s_in.wait_event(done[i])             # the previous step's GEMM i no longer reads them
                for name in ("A", "sA", "B", "sB"):
                    h["d" + name].copy_(h[name], non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_in)
                ev_in.append(e)
        for i, h in enumerate(host):
            stream.wait_event(ev_in[i])
            stream.wait_event(out_done[i])            # the previous step's D2H no longer reads D
            gemm(h["dA"], h["dsA"], h["dB"], h["dsB"], h["dD"], stream)
            done[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done[i])
                h["D"].copy_(h["dD"], non_blocking=True)
                out_done[i].record(s_out)

    one_step()
    one_step()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(s_in)
    for _ in range(steps):
        one_step()
    t_end.record(s_out)
    torch.cuda.synchronize()
    ms = t_start.elapsed_time(t_end) / steps
    flops = sum(2.0 * h["M"] * h["N"] * h["K"] for h in host)
    pinned = all(h[n].is_pinned() for h in host for n in ("A", "sA", "B", "sB", "D"))
    return {"value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": ms, "host_buffers_pinned": pinned}


# ---------------------------------------------------------------------------------------------
# CPU oracle (baseline and the reference arm)


def oracle_scales(a, b, K):
    """The FP32 scales the oracle uses: the arrays themselves, or the UE8M0 words the GPU gets,
    unpacked by the oracle."""
    if not UE8M0:
        return a.sA, b.sB
    import oracle
    pa, pb = gpu_scales(a, b)
    nkb = -(-K // 128)
    return oracle.unpack_ue8m0_a(pa, nkb), oracle.unpack_ue8m0_b(pb, nkb)


def cpu_sample_plan(problems, per_shape, seed=0):
    import dg_inputs
    rng = np.random.default_rng(seed)
    plan = []
    for (M, N, K, a, b) in problems:
        ms = rng.integers(0, M, per_shape)
        ns = rng.integers(0, N, per_shape)
        sA, sB = oracle_scales(a, b, K)
        plan.append((M, N, K, dg_inputs.OperandA(a.A, sA), dg_inputs.OperandB(b.B, sB), ms, ns))
    return plan


def cpu_baseline(problems, per_shape):
    import oracle
    plan = cpu_sample_plan(problems, per_shape)
    threads = oracle.hardware_threads()
    flops = 0.0
    t0 = time.perf_counter()
    for (M, N, K, a, b, ms, ns) in plan:
        oracle.gemm_nt_sampled(a.A, a.sA, b.B[0], b.sB[0], ms, ns, threads=threads)
        flops += 2.0 * K * len(ms)
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "extrapolated": True,
            "sample": f"a rate extrapolated from a sample: {per_shape} random output elements of each of the "
                      f"{len(plan)} sweep GEMMs ({flops / 1e9:.2f} GFLOP in {dt:.1f} s; the whole sweep would take "
                      f"about {sum(2.0 * M * N * K for (M, N, K, a, b, ms, ns) in plan) / (flops / dt) / 60:.0f} "
                      f"min), FP64 two-level accumulation, std::thread"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    problems = make_inputs()
    threads = oracle.hardware_threads()
    # Size each step's sample so that the whole --warmup W --steps K run takes about a minute:
    # calibrate the oracle's rate on a small sample first.
    calib = cpu_sample_plan(problems, 64, seed=2)
    t0 = time.perf_counter()
    cal_flops = 0.0
    for (M, N, K, a, b, ms, ns) in calib:
        oracle.gemm_nt_sampled(a.A, a.sA, b.B[0], b.sB[0], ms, ns, threads=threads)
        cal_flops += 2.0 * K * len(ms)
    rate = cal_flops / max(time.perf_counter() - t0, 1e-6)
    flops_per_element = sum(2.0 * K for (M, N, K, a, b) in problems)
    per_step_budget_s = 60.0 / max(1, args.steps + args.warmup)
    per_shape = int(min(max(16, rate * per_step_budget_s / flops_per_element), 1 << 20))
    plan = cpu_sample_plan(problems, per_shape, seed=1)

    def one_step():
        fl = 0.0
        for (M, N, K, a, b, ms, ns) in plan:
            oracle.gemm_nt_sampled(a.A, a.sA, b.B[0], b.sB[0], ms, ns, threads=threads)
            fl += 2.0 * K * len(ms)
        return fl

    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    flops = 0.0
    for _ in range(args.steps):
        flops += one_step()
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "shapes": len(plan), "seed": 0, "values": "N(0,1)",
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"each step: {per_shape} random output elements of each of the {len(plan)} sweep "
                                   f"GEMMs ({flops / args.steps / 1e9:.3f} GFLOP)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_all_configs(args):
    """One JSON line per shape of every workload configuration: time (CUDA events, mean over reps,
    L2 flushed before each, with the median beside it), TFLOP/s, the binding roof and the fraction
    of it."""
    import torch
    import dg_inputs
    import moe_grouped_gemm_e4m3_gb300 as dg
    dg.load()
    peaks = load_peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    flush = L2Flush()
    reps = max(3, min(args.steps, 20))

    def timeit(fn):
        fn()
        ts = []
        for r in range(reps):
            flush(r)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        medians.append(float(np.median(ts)))
        return float(np.mean(ts))

    medians = []   # the median of each timeit call, reported beside the mean (a rep can be an outlier)

    def report(config, shape, flops, nbytes, ms, extra=None):
        t_tc, t_hbm = flops / (fp8_peak * 1e12), nbytes / (peaks["hbm_gbs"] * 1e9)
        bound = "tensor" if t_tc >= t_hbm else "hbm"
        frac = (flops / (ms * 1e-3) / 1e12 / fp8_peak) if bound == "tensor" else (nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"])
        line = {"config": config, "shape": shape, "us": round(ms * 1e3, 2), "tflops": round(flops / (ms * 1e-3) / 1e12, 1),
                "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "bound": bound, "roof_frac": round(frac, 3),
                "us_median": round(medians[-1] * 1e3, 2) if medians else None}
        line.update(extra or {})
        print(json.dumps(line), flush=True)

    scales = {"scales": "ue8m0" if UE8M0 else "fp32"}
    chosen = None if args.configs is None else {int(c) for c in args.configs.split(",")}
    want = lambda n: chosen is None or n in chosen

    def dense(config, M, N, K, dist=dg_inputs.NORMAL, outliers=0.0):
        a = dg_inputs.make_a(M, K, seed=0, dist=dist, outlier_frac=outliers, ue8m0=UE8M0)
        b = dg_inputs.make_b(1, N, K, seed=0, dist=dist, ue8m0=UE8M0)
        gsA, gsB = gpu_scales(a, b)
        A, sA, B, sB = dev(a.A), dev(gsA), dev(b.B[0]), dev(gsB[0])
        D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        gemm = gemm_entry(dg)
        ms = timeit(lambda: gemm(A, sA, B, sB, D))
        report(config, f"{M}x{N}x{K}", 2.0 * M * N * K, algorithmic_bytes(M, N, K), ms,
               dict(scales, cfg=query_config(dg, 0, M, N, K)))

    if want(1):
        dense("1 dense small", 128, 512, 1024)
    for (M, N, K) in [(M, N, K) for M in SWEEP_M for (N, K) in SWEEP_NK] if want(2) else []:
        dense("2 dense sweep", M, N, K)
    for G in (4, 8) if want(3) else ():
        for (N, K) in ((4096, 7168), (7168, 2048)):
            M = G * 8192
            a = dg_inputs.make_a(M, K, seed=0, ue8m0=UE8M0)
            b = dg_inputs.make_b(G, N, K, seed=0, ue8m0=UE8M0)
            gsA, gsB = gpu_scales(a, b)
            idx = dev(np.repeat(np.arange(G, dtype=np.int32), 8192))
            A, sA, B, sB = dev(a.A), dev(gsA), dev(b.B), dev(gsB)
            D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
            gemm = gemm_entry(dg, "contiguous")
            ms = timeit(lambda: gemm(A, sA, B, sB, idx, D))
            nkb, nnb = -(-K // 128), -(-N // 128)
            nks = -(-nkb // 4) if UE8M0 else nkb
            nbytes = M * K + G * N * K + 4 * M * nks + 4 * G * nnb * nks + 2 * M * N
            report("3 contiguous", f"G={G} M={M} N={N} K={K}", 2.0 * M * N * K, nbytes, ms,
                   dict(scales, cfg=query_config(dg, 1, M, N, K, G)))
            del A, B, D
    for (N, K) in ((4096, 7168), (7168, 2048)) if want(4) else ():
        G, M_max = 16, 256
        mm = dg_inputs.make_masked_m(G, M_max, seed=0)
        a = dg_inputs.make_masked_a(G, M_max, K, seed=0, ue8m0=UE8M0)
        b = dg_inputs.make_b(G, N, K, seed=0, ue8m0=UE8M0)
        gsA, gsB = gpu_scales(a, b)
        A, sA, B, sB, MM = dev(a.A), dev(gsA), dev(b.B), dev(gsB), dev(mm)
        D = torch.empty(G, M_max, N, dtype=torch.bfloat16, device="cuda")
        gemm = gemm_entry(dg, "masked")
        ms = timeit(lambda: gemm(A, sA, B, sB, MM, D))
        valid = int(mm.sum())
        nkb, nnb = -(-K // 128), -(-N // 128)
        nks = -(-nkb // 4) if UE8M0 else nkb
        active = int((mm > 0).sum())
        nbytes = valid * K + active * N * K + 4 * valid * nks + 4 * G * nnb * nks + 2 * valid * N
        report("4 masked", f"G=16 M_max=256 sum(masked_m)={valid} N={N} K={K}", 2.0 * valid * N * K, nbytes, ms,
               dict(scales, cfg=query_config(dg, 2, M_max, N, K, G)))
    for (M, N, K) in ((4096, 2112, 7168), (4096, 576, 7168), (4096, 7168, 32768)) if want(5) else ():
        dense("5 stress (Student-t, outliers)", M, N, K, dist=dg_inputs.STUDENT_T3, outliers=0.01)
    # the masked form fused with SwiGLU (both scale forms): B holds 2I rows, H has I columns
    if want(7):
        for (N2, K) in ((4096, 7168),):
            G, M_max, I = 16, 256, N2 // 2
            mm = dg_inputs.make_masked_m(G, M_max, seed=0)
            a = dg_inputs.make_masked_a(G, M_max, K, seed=0, ue8m0=UE8M0)
            b = dg_inputs.make_b(G, N2, K, seed=0, ue8m0=UE8M0)
            gsA, gsB = gpu_scales(a, b)
            A, sA, B, sB, MM = dev(a.A), dev(gsA), dev(b.B), dev(gsB), dev(mm)
            H = torch.empty(G, M_max, I, dtype=torch.bfloat16, device="cuda")
            fn = dg.dg_fp8_grouped_masked_swiglu_ue8m0 if UE8M0 else dg.dg_fp8_grouped_masked_swiglu
            ms = timeit(lambda: fn(A, sA, B, sB, MM, H))
            valid = int(mm.sum())
            nkb = -(-K // 128)
            nks = -(-nkb // 4) if UE8M0 else nkb
            active = int((mm > 0).sum())
            nbytes = valid * K + active * N2 * K + 4 * valid * nks + 4 * G * (N2 // 128) * nks + 2 * valid * I
            report("7 masked + SwiGLU (fused)", f"G=16 M_max=256 sum(masked_m)={valid} 2I={N2} K={K}",
                   2.0 * valid * N2 * K, nbytes, ms, dict(scales))
            if not UE8M0:   # H cast to FP8 in the epilogue (1x128 groups): the down projection's A and sA
                Hq = torch.empty(G, M_max, I, dtype=torch.uint8, device="cuda")
                sH = torch.empty(G, I // 128, -(-M_max // 4) * 4, dtype=torch.float32, device="cuda")
                ms = timeit(lambda: dg.dg_fp8_grouped_masked_swiglu_fp8(A, sA, B, sB, MM, Hq, sH))
                nbytes += -2 * valid * I + valid * I + 4 * valid * (I // 128)
                report("7 masked + SwiGLU + FP8 H (fused)", f"G=16 M_max=256 sum(masked_m)={valid} 2I={N2} K={K}",
                       2.0 * valid * N2 * K, nbytes, ms, dict(scales))
                del Hq, sH
            del A, B, H
    # the NN / TN / TT layouts (both scale forms): A stored [K,M] and/or B stored [K,N]
    if want(8):
        M, N, K = 4096, 7168, 2048
        a = dg_inputs.make_a(M, K, seed=0, ue8m0=UE8M0)
        b = dg_inputs.make_b(1, N, K, seed=0, ue8m0=UE8M0)
        gsA, gsB = gpu_scales(a, b)
        for layout, (a_t, b_t) in (("nn", (False, True)), ("tn", (True, True)), ("tt", (True, False))):
            A = dev(np.ascontiguousarray(a.A.T) if a_t else a.A)
            B = dev(np.ascontiguousarray(b.B[0].T) if b_t else b.B[0])
            sA, sB = dev(gsA), dev(gsB[0])
            D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
            fn = getattr(dg, f"dg_fp8_gemm_{layout}_ue8m0" if UE8M0 else f"dg_fp8_gemm_{layout}")
            ms = timeit(lambda: fn(A, sA, B, sB, D, M, N, K))
            report(f"8 layout {layout}", f"{M}x{N}x{K}", 2.0 * M * N * K, algorithmic_bytes(M, N, K), ms,
                   dict(scales, cfg=query_config(dg, 0, M, N, K)))
            del A, B, D
    # the K-grouped form (weight gradients): 4 experts with 1024, 0, 2048 and 512 tokens
    if want(9):
        M, N = 2048, 7168
        off = np.array([0, 1024, 1024, 3072, 3584], np.int32)
        K = int(off[-1])
        a = dg_inputs.make_a(M, K, seed=0, ue8m0=UE8M0)
        b = dg_inputs.make_b(1, N, K, seed=0, ue8m0=UE8M0)
        gsA, gsB = gpu_scales(a, b)
        A, B = dev(np.ascontiguousarray(a.A.T)), dev(np.ascontiguousarray(b.B[0].T))
        sA, sB, O = dev(gsA), dev(gsB[0]), dev(off)
        G = len(off) - 1
        D = torch.empty(G, M, N, dtype=torch.bfloat16, device="cuda")
        fn = dg.dg_fp8_k_grouped_gemm_tn_contiguous_ue8m0 if UE8M0 else dg.dg_fp8_k_grouped_gemm_tn_contiguous
        ms = timeit(lambda: fn(A, sA, B, sB, O, D))
        nkb, nnb = K // 128, -(-N // 128)
        nks = -(-nkb // 4) if UE8M0 else nkb
        nbytes = M * K + N * K + 4 * M * nks + 4 * nnb * nks + 2 * G * M * N
        report("9 K-grouped (weight gradient)", f"G=4 M={M} N={N} K_total={K} (1024,0,2048,512)", 2.0 * M * N * K,
               nbytes, ms, dict(scales))
        del A, B, D
    # the accumulating form D = C + A·Bᵀ (FP32 C = D, in place): C is read and D written in FP32
    for (M, N, K) in ((4096, 7168, 16384), (4096, 7168, 2048)) if want(6) else ():
        a = dg_inputs.make_a(M, K, seed=0, ue8m0=UE8M0)
        b = dg_inputs.make_b(1, N, K, seed=0, ue8m0=UE8M0)
        gsA, gsB = gpu_scales(a, b)
        A, sA, B, sB = dev(a.A), dev(gsA), dev(b.B[0]), dev(gsB[0])
        D = torch.zeros(M, N, dtype=torch.float32, device="cuda")
        acc = dg.dg_fp8_gemm_nt_ue8m0_acc_f32 if UE8M0 else dg.dg_fp8_gemm_nt_acc_f32
        ms = timeit(lambda: acc(A, sA, B, sB, D, D))
        nbytes = algorithmic_bytes(M, N, K) - 2 * M * N + 8 * M * N
        report("6 accumulate D = C + A·Bᵀ (FP32, in place)", f"{M}x{N}x{K}", 2.0 * M * N * K, nbytes, ms,
               dict(scales, cfg=query_config(dg, 0, M, N, K)))
        del A, B, D


def main():
    args = parse_args()
    rank, world, local = dist_info()
    if args.all_configs:
        run_all_configs(args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
