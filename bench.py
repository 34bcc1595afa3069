"""Benchmark of the GB300 tiled GEMM  C = A·Bᵀ  (TFLOP/s = 2MNK / t).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl tkg|reference]

Default: the GEMM suite.  Every GEMM workload of the study (bf16 256^3, 4096^3,
8192^3 and 16384x8192x2048, FP8 e4m3 8192^3, NVFP4 16384^3) is measured in
turn; the JSON line's headline fields are those of the largest, NVFP4
M=N=K=16384, and `configs` carries one entry per workload with its own value,
roofline, cpu_baseline, e2e, clocks and parity check.  For each workload a step
is one batch of independent GEMMs run back to back through the C ABI with
operands resident in HBM; operands rotate over copies whose total exceeds the
129 MB L2, so every GEMM reads its inputs from HBM.  After the timed steps the
output is compared with the CPU oracle on sampled rows at the contract's
tolerance; a mismatch makes the run exit non-zero.

--workload NAME measures one workload (a GEMM, an input encoder or attention)
and prints its own line.  Rank 0 prints one JSON line.  Under torchrun each
rank runs its own replica (weak scaling, no collective on the data path); the
time is the maximum over ranks.  --gpus N without torchrun relaunches the
script under torchrun with N processes.

--impl reference times the CPU oracle (the plain C reference) on the host
cores on a bounded sample of the same workload, with the same metric.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from tiled_tensor_core_gb300 import synth  # noqa: E402

METRIC = "GEMM TFLOP/s (2MNK/t) bf16/FP8/NVFP4 on 1 GB300; % of dense tensor peak"
L2_BYTES = 129 * 2 ** 20
# GEMMs per step, sized so that a step is tens of milliseconds of GPU work
BATCH = {"bf16_256": 2000, "bf16_4096": 400, "bf16_8192": 60, "bf16_skinny": 100, "fp8_8192": 100,
         "nvfp4_16384": 30, "bf16_4096_k64": 4000, "bf16_4096_k128": 3000, "bf16_4096_k256": 2000,
         "bf16_4096_k512": 1500, "bf16_4096_k1024": 1000}
SCHEDULE = {"static": 1, "dynamic": 2, "single": 3}
# the default run: every GEMM workload of the study, headline on the largest
SUITE = ["bf16_256", "bf16_4096", "bf16_8192", "bf16_skinny", "fp8_8192", "nvfp4_16384"]
HEADLINE = "nvfp4_16384"
# dense tensor-core peak relative to bf16 (nominal GB300 ratios: bf16 2.25, fp8 4.5, fp4 13.5 PFLOP/s)
PEAK_RATIO = {"bf16": 1.0, "fp8": 2.0, "nvfp4": 6.0}
DTYPE = {"bf16": "bf16", "fp8": "e4m3", "nvfp4": "e2m1+e4m3"}


# DRAM bytes (read + write) per launch of the dominant kernel, from one full-size ncu capture
# (profiles/gemm_*_ncu.md, profiles/attention_fwd_4096_d128_ncu.md), valid only while the sources of
# that kernel hash to the value recorded with it.
TRAFFIC = {
    "bf16_4096": {"bytes": 93_633_792, "src": "4bed562ab90fb120"},
    "bf16_8192": {"bytes": 834_269_952, "src": "4bed562ab90fb120"},
    "bf16_skinny": {"bytes": 448_839_936, "src": "4bed562ab90fb120"},
    "fp8_8192": {"bytes": 393_207_552, "src": "0ee1790daf721892"},
    "nvfp4_16384": {"bytes": 1_604_999_936, "src": "0ef3cf4e1cc09e5e"},
    "attn_n4096_d128": {"bytes": 1_061_352_448, "src": "83fdd4522b9cd05c"},
}
KERNEL_SOURCES = {
    "bf16": ("tkg_device.cuh", "gemm_kernel.cuh", "gemm_bf16.cu"),
    "fp8": ("tkg_device.cuh", "gemm_kernel.cuh", "gemm_fp8.cu"),
    "nvfp4": ("tkg_device.cuh", "gemm_kernel.cuh", "gemm_nvfp4.cu"),
    "attn": ("tkg_device.cuh", "attention.cu"),
}


def kernel_source_hash(files) -> str:
    """Hash of kernel sources with comments, blank lines and indentation removed, so that a
    comment or layout edit does not invalidate a recorded capture but any code change does."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tiled_tensor_core_gb300", "csrc")
    for f in files:
        with open(os.path.join(csrc, f)) as fh:
            text = re.sub(r"/\*.*?\*/", "", fh.read(), flags=re.S)
        for line in text.splitlines():
            line = re.sub(r"//.*$", "", line).strip()
            if line:
                h.update(line.encode() + b"\n")
    return h.hexdigest()[:16]


def traffic_bytes(workload: str):
    rec = TRAFFIC.get(workload)
    if rec is None:
        return None
    kind = "attn" if workload.startswith("attn_") else workload.split("_")[0]
    if rec["src"] == kernel_source_hash(KERNEL_SOURCES[kind]):
        return rec["bytes"]
    return None


def algorithmic_bytes(w) -> int:
    """Minimal HBM bytes of one GEMM: A and B read once (plus, NVFP4, the per-16
    block scales and the two fp32 tensor scales), C written once."""
    if w.kind == "bf16":
        ab = 2 * (w.M + w.N) * w.K
    elif w.kind == "fp8":
        ab = (w.M + w.N) * w.K + 8
    else:
        ab = (w.M + w.N) * w.K // 2 + (w.M + w.N) * w.K // 16 + 8
    return ab + 2 * w.M * w.N


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"bf16_tflops": float(d["bf16_tflops"]), "bf16_tflops_sustained": float(d["bf16_tflops_sustained"]),
                "hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="tkg_clocks_", suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
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
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), max=float(parts[2]), power=float(parts[3]), active=parts[4],
                                 hw=parts[5], hw_thermal=parts[6], sw_thermal=parts[7], sw_power=parts[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


# ---------------------------------------------------------------- distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "tkg" else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- oracle timing

def oracle_sample(ops, target_s: float):
    """Time the oracle as it stands on a row sample of the workload sized to
    about target_s seconds of host work.  Returns (TFLOP/s, seconds, rows, threads)."""
    import oracle
    M, N, K = ops.M, ops.N, ops.K
    threads = oracle.num_threads()
    wave = np.linspace(0, M - 1, min(M, threads)).astype(np.int64)
    t0 = time.perf_counter()
    oracle.gemm(ops, rows=wave)
    t_wave = max(time.perf_counter() - t0, 1e-6)
    waves = max(1, int(target_s / t_wave))
    n_rows = int(min(M, len(wave) * waves))
    rows = np.linspace(0, M - 1, n_rows).astype(np.int64)
    t0 = time.perf_counter()
    oracle.gemm(ops, rows=rows)
    dt = time.perf_counter() - t0
    return 2.0 * n_rows * N * K / dt / 1e12, dt, n_rows, threads


# ---------------------------------------------------------------- parity gate

# Tolerances of the GEMM contract: bf16 output against the oracle's bf16 output
# (relative Frobenius <= 1e-3, |delta| <= 1e-2 (|ref| + 1) elementwise); FP8 /
# NVFP4 against the oracle's fp32 accumulation of the same decoded values times
# the per-tensor scales (relative Frobenius <= 2e-3).
BF16_REL_FRO, BF16_ELEM, SCALED_REL_FRO = 1e-3, 1e-2, 2e-3
PARITY_ROWS = 32


def parity_rows(M: int, seed: int) -> np.ndarray:
    """At least PARITY_ROWS rows: the edges of 128-row CTA tiles and 256-row pair
    tiles, every 32-row TMEM lane quarter of the first tile, the last rows, and
    seeded random rows."""
    fixed = [0, 1, 31, 32, 63, 64, 95, 96, 127, 128, 159, 160, 191, 192, 223, 224, 255, 256, 383, 511,
             M // 2, M // 2 + 127, M - 129, M - 128, M - 2, M - 1]
    rows = sorted({r for r in fixed if 0 <= r < M})
    rng = np.random.default_rng(seed)
    while len(rows) < min(M, PARITY_ROWS + 8):
        rows = sorted(set(rows) | {int(r) for r in rng.integers(0, M, size=8)})
    return np.array(rows, dtype=np.int64)


def parity_check(ops, c_rows_bits: np.ndarray, rows: np.ndarray) -> dict:
    """Compare sampled output rows (bf16 bits) with the oracle at the contract tolerance."""
    import oracle
    acc, c_ref = oracle.gemm(ops, rows=rows)
    to64 = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)  # noqa: E731
    got = to64(c_rows_bits)
    out = {"rows": int(len(rows)), "finite": bool(np.isfinite(got).all())}
    if ops.kind == "bf16":
        ref = to64(c_ref)
        out["rel_fro"] = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
        out["max_elem"] = float((np.abs(got - ref) / (np.abs(ref) + 1.0)).max())
        out["tol"] = {"rel_fro": BF16_REL_FRO, "elem": BF16_ELEM, "against": "oracle bf16 output"}
        out["pass"] = out["finite"] and out["rel_fro"] <= BF16_REL_FRO and out["max_elem"] <= BF16_ELEM
    else:
        ref = acc.astype(np.float64) * ops.scale_a * ops.scale_b
        out["rel_fro"] = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
        out["tol"] = {"rel_fro": SCALED_REL_FRO, "against": "oracle fp32 accumulation x scales"}
        out["pass"] = out["finite"] and out["rel_fro"] <= SCALED_REL_FRO
    return out


# ---------------------------------------------------------------- reference arm

def run_reference(args, world, rank):
    if rank != 0:
        return 0
    if args.workload in ENCODERS:
        return run_reference_encoder(args)
    name = args.workload or HEADLINE
    w = synth.WORKLOADS[name]
    ops = synth.workload_operands(name)
    for _ in range(args.warmup):
        oracle_sample(ops, 0.1)
    times = []
    flops = 0.0
    n_rows = threads = 0
    for _ in range(args.steps):
        _, dt, n_rows, threads = oracle_sample(ops, args.ref_step_s)
        times.append(dt)
        flops += 2.0 * n_rows * w.N * w.K
    value = flops / sum(times) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE[w.kind],
        "data": "synthetic",
        "config": {"workload": w.description, "M": w.M, "N": w.N, "K": w.K,
                   "sample_rows_per_step": n_rows},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n_rows} of {w.M} output rows (x {w.N} cols x K={w.K}) per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

def set_options(tkg, args):
    tkg.tkg_set_option(tkg.TKG_OPT_VARIANT, args.variant)
    tkg.tkg_set_option(tkg.TKG_OPT_GROUP_M, args.group_m)
    tkg.tkg_set_option(tkg.TKG_OPT_SCHEDULE, SCHEDULE[args.schedule])
    tkg.tkg_set_option(tkg.TKG_OPT_LAUNCH_OVERLAP,
                       tkg.TKG_OVERLAP_ON if args.overlap == "on" else tkg.TKG_OVERLAP_OFF)
    tkg.tkg_set_option(tkg.TKG_OPT_SPLIT_K, tkg.TKG_SPLIT_ON if args.split == "on" else tkg.TKG_SPLIT_OFF)
    tkg.tkg_set_option(tkg.TKG_OPT_K_ORDER,
                       tkg.TKG_K_ORDER_SERPENTINE if args.k_order == "serpentine" else tkg.TKG_K_ORDER_FORWARD)


def operand_sets(footprint: int) -> int:
    """Copies of a workload's operands (and output) that the timed launches rotate over: enough
    that a GEMM never finds its operands in L2 from the last time they were used (a footprint of
    twice the 129 MB L2 needs one; the 256^3 workload ~1400 of its 0.4 MB sets)."""
    return 1 if footprint >= 2 * L2_BYTES else math.ceil(4 * L2_BYTES / footprint)


def measure_gemm(name, args, world, rank, local, cpu_s):
    """Warm-up, timed steps, parity gate, e2e, cuBLAS context and oracle timing of one
    GEMM workload.  Returns its entry (a dict); entry["parity"]["pass"] is False on a
    mismatch with the oracle."""
    import torch
    from tiled_tensor_core_gb300 import tkg
    from tiled_tensor_core_gb300.device import DeviceGemm

    dev = torch.device("cuda", local)
    w = synth.WORKLOADS[name]
    ops = synth.workload_operands(name)
    base = DeviceGemm(ops, dev)
    footprint = base.input_bytes() + base.output_bytes()
    n_sets = operand_sets(footprint)
    sets = [base]
    for _ in range(n_sets - 1):
        g = DeviceGemm.__new__(DeviceGemm)
        g.__dict__.update(base.__dict__)
        g.a, g.b = base.a.clone(), base.b.clone()
        if base.sfa is not None:
            g.sfa, g.sfb = base.sfa.clone(), base.sfb.clone()
        if base.scale_a is not None:
            g.scale_a, g.scale_b = base.scale_a.clone(), base.scale_b.clone()
        g.c = torch.empty_like(base.c)
        sets.append(g)
    batch = args.batch or BATCH[name]
    stream = torch.cuda.Stream(device=dev)
    sptr = int(stream.cuda_stream)
    launches_per_gemm = 2 if w.kind == "nvfp4" else 1

    def step(events=None):
        for i in range(batch):
            g = sets[i % n_sets]
            if events is not None:
                events[2 * i].record(stream)
            g.run(stream=sptr)
            if events is not None:
                events[2 * i + 1].record(stream)

    for g in sets:
        g.c.fill_(float("nan"))
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    st = tkg.tkg_check_status(sptr)
    if st != tkg.TKG_OK:
        raise RuntimeError(f"{name}: warm-up failed: {tkg.status_string(st)}")

    # Launch-bound workloads replay the step from a CUDA graph (captured after the
    # warm-up, so every lazy set-up is done); the GEMM launches are unchanged.
    use_graph = args.graph == "on" or (args.graph == "auto" and w.flops < 5e10 and w.kind != "nvfp4")
    graph = None
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        with torch.cuda.stream(stream):
            for _ in range(2):
                graph.replay()
        torch.cuda.synchronize(dev)

    step_ms, kern_ms, host_ms = [], [], []
    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    for g in sets:  # the parity check below reads outputs written inside the timed region
        g.c.fill_(float("nan"))
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)  # let the sampler take its first reading
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    # The steps are enqueued back to back (no host synchronisation between them, so the GPU never
    # waits for the host at a step boundary); per-step and per-launch events are read afterwards.
    per_launch = graph is None and args.overlap == "off"
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    launch_ev = ([[torch.cuda.Event(enable_timing=True) for _ in range(2 * batch)] for _ in range(args.steps)]
                 if per_launch else None)
    t_start.record(stream)
    for s_ in range(args.steps):
        step_ev[s_][0].record(stream)
        h0 = time.perf_counter()
        if graph is not None:
            with torch.cuda.stream(stream):
                graph.replay()
        else:
            # an event between two launches would end their overlap: with it on, the step is timed whole
            step(launch_ev[s_] if per_launch else None)
        host_ms.append((time.perf_counter() - h0) * 1e3)
        step_ev[s_][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    for s_ in range(args.steps):
        step_ms.append(step_ev[s_][0].elapsed_time(step_ev[s_][1]))
        if per_launch:
            kern_ms.extend(launch_ev[s_][2 * i].elapsed_time(launch_ev[s_][2 * i + 1]) for i in range(batch))
        else:
            # no per-launch events (inside a graph, or between overlapped launches): the step is
            # nothing but GEMM launches (and, NVFP4, the scale re-layout before each), so spread its
            # time over the GEMMs
            kern_ms.extend([step_ms[-1] / batch] * batch)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    barrier(world)
    st = tkg.tkg_check_status(sptr)
    if st != tkg.TKG_OK:
        raise RuntimeError(f"{name}: timed run failed: {tkg.status_string(st)}")
    total_ms = t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(total_ms, world, dev)
    gemms = args.steps * batch
    value = world * gemms * w.flops / (total_ms * 1e-3) / 1e12
    kern_avg_ms = sum(kern_ms) / len(kern_ms)
    achieved = w.flops / (kern_avg_ms * 1e-3) / 1e12

    # parity gate on every rank: sampled rows of an output written by the timed steps
    rows = parity_rows(w.M, seed=w.M + w.N + w.K)
    last = sets[(gemms - 1) % n_sets] if graph is None else sets[(batch - 1) % n_sets]
    c_rows = last.c[torch.from_numpy(rows).to(dev)].view(torch.int16).cpu().numpy().view(np.uint16)
    parity = parity_check(ops, c_rows, rows) if not args.no_check else {"skipped": True, "pass": True}

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(ops, dev, w, args)

    # context: cuBLAS on the same shape, operands and stream (the pages' "matches cuBLAS" claim)
    cublas = None
    if not args.no_cublas:
        cublas = run_cublas(sets, w, batch, stream, args)
        if cublas is not None and "value" in cublas:
            cublas["ours_over_cublas"] = value / world / cublas["value"]

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and cpu_s > 0:
        v, dt, n_rows, threads = oracle_sample(ops, cpu_s)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{n_rows} of {w.M} output rows of the same workload ({dt:.1f} s)"}

    peaks = load_peaks()
    # Denominators: the measured bf16 peak x the nominal dtype ratio.  The timed region is about a
    # second of back-to-back launches: `frac` uses the burst figure (the lower fraction), and the
    # fraction of the sustained (power-capped, seconds-long) figure is given beside it.
    peak_burst = peaks["bf16_tflops"] * PEAK_RATIO[w.kind]
    peak_sust = peaks["bf16_tflops_sustained"] * PEAK_RATIO[w.kind]
    kid = {"bf16": 0, "fp8": 1, "nvfp4": 2}[w.kind]
    info = tkg.tkg_debug_variant_info(kid, tkg.tkg_debug_pick_variant(kid, w.M, w.N, w.K))
    alg_bytes = algorithmic_bytes(w)
    entry = {
        "workload": name, "description": w.description, "M": w.M, "N": w.N, "K": w.K, "dtype": DTYPE[w.kind],
        "value": value, "unit": "TFLOP/s", "ms_per_step": total_ms / args.steps, "gemms_per_step": batch,
        "median_gemm_ms": statistics.median(kern_ms),
        "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms), "max": max(step_ms)},
        "host_enqueue_ms_per_step": statistics.median(host_ms),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_burst, "unit": "TFLOP/s",
                     "frac": achieved / peak_burst, "traffic": traffic_bytes(name),
                     "algorithmic_bytes": alg_bytes,
                     "peak_sustained": peak_sust, "frac_of_sustained_peak": achieved / peak_sust,
                     "peak_source": (f"{peaks['source']} bf16 burst (cuBLAS) x {PEAK_RATIO[w.kind]:g} "
                                     "(nominal dtype ratio); sustained beside it")},
        "achieved_hbm_gbs_algorithmic": alg_bytes / (kern_avg_ms * 1e-3) / 1e9,
        "cpu_baseline": cpu, "e2e": e2e, "cublas": cublas, "clocks": clocks, "parity": parity,
        "gpu_launches": gemms * launches_per_gemm,
        "kernel": info,
        "l2": (f"{n_sets} rotating operand sets, {n_sets * footprint / 2**20:.0f} MiB > 129 MiB L2"
               if n_sets > 1 else f"operands {footprint / 2**20:.0f} MiB > 129 MiB L2"),
        "cuda_graph": graph is not None,
        "inputs_sha256": ops.digest()[:16],
    }
    del sets, base
    torch.cuda.empty_cache()
    return entry


def tkg_group_m() -> int:
    from tiled_tensor_core_gb300 import tkg
    return int(tkg.tkg_get_option(tkg.TKG_OPT_GROUP_M))


def line_from_entry(e, args, world, extra_config=None):
    """The contract's JSON line for one measured GEMM entry."""
    w = synth.WORKLOADS[e["workload"]]
    config = {"workload": w.description, "M": w.M, "N": w.N, "K": w.K, "gemms_per_step": e["gemms_per_step"],
              "global_batch": e["gemms_per_step"] * world, "parallelism": f"replicas{world}", "l2": e["l2"],
              "kernel": e["kernel"], "group_m": tkg_group_m(), "schedule": args.schedule,
              "split_k_tail": args.split, "k_order": args.k_order,
              "launch_overlap": "programmatic dependent launch" if args.overlap == "on" else "off",
              "cuda_graph": e["cuda_graph"]}
    if extra_config:
        config.update(extra_config)
    return {
        "metric": METRIC, "value": e["value"], "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": e["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": e["dtype"], "data": "synthetic", "config": config,
        "roofline": e["roofline"], "cpu_baseline": e["cpu_baseline"], "e2e": e["e2e"],
        "gpu_launches": e["gpu_launches"], "clocks": e["clocks"], "parity": e["parity"],
        "median_gemm_ms": e["median_gemm_ms"], "step_ms": e["step_ms"],
        "host_enqueue_ms_per_step": e["host_enqueue_ms_per_step"], "cublas": e["cublas"],
        "inputs_sha256": e["inputs_sha256"], "device": device_record(),
    }


def device_record() -> dict:
    """The GPU the line was measured on, from its device properties (the SM clocks under load
    and their maximum are in `clocks`)."""
    import torch
    p = torch.cuda.get_device_properties(torch.cuda.current_device())
    return {"name": p.name, "sm_count": p.multi_processor_count, "cc": f"{p.major}.{p.minor}",
            "memory_gib": round(p.total_memory / 2**30, 1)}


def run_tkg(args, world, rank, local):
    import torch
    from tiled_tensor_core_gb300 import tkg

    torch.cuda.set_device(local)
    set_options(tkg, args)
    if args.workload:
        e = measure_gemm(args.workload, args, world, rank, local, args.cpu_s)
        if rank == 0:
            print(json.dumps(line_from_entry(e, args, world)), flush=True)
        return 0 if e["parity"]["pass"] else 3
    entries = []
    for name in SUITE:
        cpu_s = args.cpu_s if name == HEADLINE else args.cpu_s_other
        entries.append(measure_gemm(name, args, world, rank, local, cpu_s))
    head = next(e for e in entries if e["workload"] == HEADLINE)
    line = line_from_entry(head, args, world, {"suite": SUITE, "headline": HEADLINE})
    line["configs"] = entries
    line["gpu_launches_all_configs"] = sum(e["gpu_launches"] for e in entries)
    line["parity_all_pass"] = all(e["parity"]["pass"] for e in entries)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0 if line["parity_all_pass"] else 3


# ---------------------------------------------------------------- input encoders

ENCODERS = {
    # name: (kind, rows, cols, seed) — the fp32 data the FP8 8192^3 and NVFP4 16384^3 workloads encode
    "encode_fp8_8192": ("fp8", 8192, 8192, 1004),
    "encode_nvfp4_16384": ("nvfp4", 16384, 16384, 1005),
}


def run_encoder(args, world, rank, local):
    """One step = one on-device encoding (tkg_quantize_fp8 / tkg_quantize_nvfp4)
    of an fp32 [rows][cols] tensor resident in HBM.  HBM-bound: the algorithmic
    bytes are two reads of x (the tensor amax must be known before any element
    is encoded) plus the encoded output."""
    import torch
    from tiled_tensor_core_gb300 import tkg

    import oracle

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kind, rows, cols, seed = ENCODERS[args.workload]
    x_host = synth.draw_fp32(seed, rows, cols, "normal")
    x = torch.from_numpy(x_host).to(dev)
    n = rows * cols
    if kind == "fp8":
        outs = [torch.empty((rows, cols), dtype=torch.uint8, device=dev), torch.empty(1, dtype=torch.float32, device=dev)]
        call = lambda st: tkg.tkg_quantize_fp8(rows, cols, x, outs[0], outs[1], stream=st)  # noqa: E731
        out_bytes = n + 4
    else:
        outs = [torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev),
                torch.empty((rows, cols // 16), dtype=torch.uint8, device=dev),
                torch.empty(1, dtype=torch.float32, device=dev)]
        call = lambda st: tkg.tkg_quantize_nvfp4(rows, cols, x, outs[0], outs[1], outs[2], stream=st)  # noqa: E731
        out_bytes = n // 2 + n // 16 + 4
    alg_bytes = 2 * 4 * n + out_bytes
    stream = torch.cuda.Stream(device=dev)
    sptr = int(stream.cuda_stream)
    for _ in range(args.warmup):
        call(sptr)
    if tkg.tkg_check_status(sptr) != tkg.TKG_OK:
        raise RuntimeError("encoder warm-up failed")
    spot = None
    if rank == 0 and not args.no_check:  # full bit-exact comparison with the oracle's encoder
        if kind == "fp8":
            q_ref, s_ref = oracle.quantize_fp8(x_host)
            spot = bool(np.array_equal(outs[0].cpu().numpy(), q_ref) and outs[1].item() == s_ref)
        else:
            q_ref, sf_ref, g_ref = oracle.quantize_nvfp4(x_host)
            spot = bool(np.array_equal(outs[0].cpu().numpy(), q_ref) and np.array_equal(outs[1].cpu().numpy(), sf_ref)
                        and outs[2].item() == g_ref)
        if not spot:
            raise RuntimeError("encoder output differs from the oracle")
    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]
    for i in range(args.steps):
        ev[2 * i].record(stream)
        call(sptr)
        ev[2 * i + 1].record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    barrier(world)
    if tkg.tkg_check_status(sptr) != tkg.TKG_OK:
        raise RuntimeError("encoder timed run failed")
    step_ms = [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(args.steps)]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    value = world * args.steps * alg_bytes / (total_ms * 1e-3) / 1e9
    achieved = alg_bytes / (statistics.mean(step_ms) * 1e-3) / 1e9

    e2e = None
    if not args.no_e2e:  # pinned host x -> device, encode, encoded operand -> host
        xh = torch.from_numpy(x_host).pin_memory()
        oh = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
        torch.cuda.synchronize(dev)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k = max(1, args.e2e_steps)
        with torch.cuda.stream(stream):
            t0.record(stream)
            for _ in range(k):
                x.copy_(xh, non_blocking=True)
                call(sptr)
                for o, h in zip(outs, oh):
                    h.copy_(o, non_blocking=True)
            t1.record(stream)
        t1.synchronize()
        ms = t0.elapsed_time(t1) / k
        e2e = {"value": alg_bytes / (ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": 4 * n,
               "d2h_bytes_per_step": out_bytes, "ms_per_step": ms}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r = max(1, min(rows, int(rows * min(1.0, args.cpu_s / 10.0))))
        xs = np.ascontiguousarray(x_host[:r])
        t = time.perf_counter()
        (oracle.quantize_fp8 if kind == "fp8" else oracle.quantize_nvfp4)(xs)
        dt = time.perf_counter() - t
        nb = 2 * 4 * r * cols + (r * cols if kind == "fp8" else r * cols // 2 + r * cols // 16)
        cpu = {"value": nb / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{r} of {rows} rows of the same tensor ({dt:.1f} s)"}

    peaks = load_peaks()
    line = {
        "metric": "encoder GB/s (algorithmic bytes: 2 reads of fp32 x + encoded output, / time)",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{kind} encoder of an fp32 [{rows}][{cols}] N(0,1) tensor", "rows": rows, "cols": cols,
                   "l2": f"input {4 * n / 2**20:.0f} MiB > 129 MiB L2"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                     "peak_source": f"{peaks['source']} copy bandwidth"},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 3 * args.steps, "clocks": clocks,
        "bit_exact_vs_oracle": spot,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_cublas(sets, w, batch, stream, args):
    """cuBLAS (through torch.matmul for bf16, torch._scaled_mm for FP8 with the same per-tensor
    scales) on the same operand sets, timed like our step: `batch` products back to back per
    step, events around the steps.  Context only: no part of the library path."""
    import torch
    outs = [torch.empty_like(g.c) for g in sets]
    if w.kind == "bf16":
        mats = [(g.a.view(torch.bfloat16), g.b.view(torch.bfloat16)) for g in sets]

        def one(i):
            a, b = mats[i % len(sets)]
            torch.matmul(a, b.t(), out=outs[i % len(sets)])
    elif w.kind == "fp8":
        if not hasattr(torch, "_scaled_mm"):
            return None
        mats = [(g.a.view(torch.float8_e4m3fn), g.b.view(torch.float8_e4m3fn), g.scale_a, g.scale_b) for g in sets]

        def one(i):
            a, b, sa, sb = mats[i % len(sets)]
            outs[i % len(sets)] = torch._scaled_mm(a, b.t(), scale_a=sa, scale_b=sb, out_dtype=torch.bfloat16)
    else:
        # NVFP4: the same packed e2m1 operands and e4m3 block scales, the scales re-laid out (once,
        # untimed) into the 128 x 4 blocked order cuBLAS documents for 16-element block scaling;
        # cuBLAS applies the block scales only (the two per-tensor scales are one multiply in the
        # epilogue)
        if not hasattr(torch, "_scaled_mm") or not hasattr(torch, "float4_e2m1fn_x2"):
            return {"unavailable": "this torch build has no float4_e2m1fn_x2 / _scaled_mm"}
        mats = [(g.a.view(torch.float4_e2m1fn_x2), g.b.view(torch.float4_e2m1fn_x2),
                 cublas_blocked_scales(g.sfa).view(torch.float8_e4m3fn),
                 cublas_blocked_scales(g.sfb).view(torch.float8_e4m3fn)) for g in sets]

        def one(i):
            a, b, sa, sb = mats[i % len(sets)]
            outs[i % len(sets)] = torch._scaled_mm(a, b.t(), scale_a=sa, scale_b=sb, out_dtype=torch.bfloat16)
    try:
        with torch.cuda.stream(stream):
            for i in range(batch * max(1, args.warmup)):
                one(i)
            torch.cuda.synchronize()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            for s in range(args.steps):
                ev[s][0].record(stream)
                for i in range(batch):
                    one(i)
                ev[s][1].record(stream)
            torch.cuda.synchronize()
    except RuntimeError as e:  # a cuBLAS path torch does not offer on this build
        return {"unavailable": str(e).splitlines()[0][:200]}
    ms = statistics.median(a.elapsed_time(b) for a, b in ev) / batch
    how = {"bf16": "torch.matmul (bf16)", "fp8": "torch._scaled_mm (e4m3, per-tensor scales)",
           "nvfp4": "torch._scaled_mm (e2m1, e4m3 scales per 16 elements)"}[w.kind]
    return {"value": w.flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "how": how}


def cublas_blocked_scales(sf):
    """Row-major [rows][K/16] e4m3 block scales -> cuBLAS's blocked layout: the matrix padded to
    128-row x 4-column blocks, blocks in row-major order, and inside a block the scale of row r,
    column c at byte 16 * (r % 32) + 4 * (r // 32) + c."""
    import torch
    rows, cols = sf.shape
    pr, pc = -(-rows // 128) * 128, -(-cols // 4) * 4
    padded = torch.zeros((pr, pc), dtype=torch.uint8, device=sf.device)
    padded[:rows, :cols] = sf.view(torch.uint8)
    blocks = padded.view(pr // 128, 128, pc // 4, 4).permute(0, 2, 1, 3)  # [row block][col block][128][4]
    inner = blocks.reshape(pr // 128, pc // 4, 4, 32, 4).transpose(2, 3)  # [..][r % 32][r // 32][c]
    return inner.reshape(pr, pc).contiguous()


def run_e2e(ops, dev, w, args):
    """End to end through the public API with host buffers: every step copies
    its inputs from pinned host memory to the device, runs the GEMM and copies
    C back to pinned host memory.  Steps are pipelined over two device buffer
    sets and three streams (H2D of step i+1 and D2H of step i-1 overlap the
    GEMM of step i); the timed region spans all copies of all steps."""
    import torch
    from tiled_tensor_core_gb300.device import DeviceGemm

    sets = [DeviceGemm(ops, dev), DeviceGemm(ops, dev)]
    names = [n for n in ("a", "b", "sfa", "sfb", "scale_a", "scale_b") if getattr(sets[0], n) is not None]
    host = {n: getattr(sets[0], n).cpu().pin_memory() for n in names}
    c_host = [torch.empty(sets[0].c.shape, dtype=sets[0].c.dtype).pin_memory() for _ in range(2)]
    h2d_s, gemm_s, d2h_s = (torch.cuda.Stream(device=dev) for _ in range(3))
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = c_host[0].numel() * c_host[0].element_size()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    inputs_free = [ev(), ev()]   # GEMM of the set finished reading its inputs
    inputs_ready = [ev(), ev()]
    out_free = [ev(), ev()]      # D2H of the set finished reading C
    out_ready = [ev(), ev()]
    for e in inputs_free + out_free:
        e.record(gemm_s)

    def one(i):
        k = i % 2
        g = sets[k]
        h2d_s.wait_event(inputs_free[k])
        with torch.cuda.stream(h2d_s):
            for n in names:
                getattr(g, n).copy_(host[n], non_blocking=True)
        inputs_ready[k].record(h2d_s)
        gemm_s.wait_event(inputs_ready[k])
        gemm_s.wait_event(out_free[k])
        g.run(stream=int(gemm_s.cuda_stream))
        inputs_free[k].record(gemm_s)
        out_ready[k].record(gemm_s)
        d2h_s.wait_event(out_ready[k])
        with torch.cuda.stream(d2h_s):
            c_host[k].copy_(g.c, non_blocking=True)
        out_free[k].record(d2h_s)

    for i in range(4):
        one(i)
    torch.cuda.synchronize(dev)
    n = args.e2e_steps
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(h2d_s)
    for i in range(n):
        one(i)
    d2h_s.wait_stream(h2d_s)
    d2h_s.wait_stream(gemm_s)
    t1.record(d2h_s)
    t1.synchronize()
    ms = t0.elapsed_time(t1) / n
    return {"value": w.flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": ms, "pipelined": "2 buffer sets, 3 streams"}


# ---------------------------------------------------------------- attention forward

ATTN_METRIC = "attention forward TFLOP/s (4·B·H·Nq·Nkv·D / t), bf16, non-causal, 1 GB300"
ATTN_BATCH = {"attn_n1024_d128": 40, "attn_n4096_d128": 6, "attn_n4096_d64": 8}


def attn_oracle_sample(x, w, target_s: float):
    """The attention oracle, as it stands, on a sample of query rows of a few heads
    (about target_s seconds).  Returns (TFLOP/s, seconds, rows, heads)."""
    from oracle import attention as oa
    heads = [(b, h) for b in range(w.B) for h in range(w.H)][:: max(1, (w.B * w.H) // 8)][:8]
    probe = np.arange(0, w.Nq, max(1, w.Nq // 16))
    t0 = time.perf_counter()
    oa.attention_forward(x.q, x.k, x.v, heads=heads[:1], rows=probe)
    per_row = max(time.perf_counter() - t0, 1e-6) / len(probe)
    n_rows = int(max(16, min(w.Nq, target_s / per_row / len(heads))))
    rows = np.linspace(0, w.Nq - 1, n_rows).astype(np.int64)
    t0 = time.perf_counter()
    oa.attention_forward(x.q, x.k, x.v, heads=heads, rows=rows)
    dt = time.perf_counter() - t0
    flops = 4.0 * len(heads) * n_rows * w.Nkv * w.D
    return flops / dt / 1e12, dt, n_rows, len(heads)


def run_reference_attention(args):
    w = synth.ATTN_WORKLOADS[args.workload]
    x = synth.attn_workload_inputs(args.workload)
    for _ in range(args.warmup):
        attn_oracle_sample(x, w, 0.05)
    times, flops = [], 0.0
    n_rows = n_heads = 0
    for _ in range(args.steps):
        _, dt, n_rows, n_heads = attn_oracle_sample(x, w, args.ref_step_s)
        times.append(dt)
        flops += 4.0 * n_heads * n_rows * w.Nkv * w.D
    value = flops / sum(times) / 1e12
    line = {"impl": "reference", "metric": ATTN_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.description, "B": w.B, "H": w.H, "Nq": w.Nq, "Nkv": w.Nkv, "D": w.D},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"{n_rows} query rows x {n_heads} heads per step (numpy float64, "
                                       "BLAS threads on all host cores)"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_attention(args, world, rank, local):
    import torch
    from tiled_tensor_core_gb300 import tkg

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tkg.tkg_set_option(tkg.TKG_OPT_LAUNCH_OVERLAP,
                       tkg.TKG_OVERLAP_ON if args.overlap == "on" else tkg.TKG_OVERLAP_OFF)
    w = synth.ATTN_WORKLOADS[args.workload]
    x = synth.attn_workload_inputs(args.workload)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)  # noqa: E731
    base = {"q": t(x.q), "k": t(x.k), "v": t(x.v)}
    per_set = sum(v.numel() * 2 for v in base.values()) + base["q"].numel() * 2
    n_sets = 1 if per_set >= 2 * L2_BYTES else min(8, math.ceil(4 * L2_BYTES / per_set))
    sets = []
    for i in range(n_sets):
        d = {k: (v if i == 0 else v.clone()) for k, v in base.items()}
        d["o"] = torch.empty_like(d["q"])
        d["lse"] = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
        sets.append(d)
    batch = args.batch or ATTN_BATCH[args.workload]
    stream = torch.cuda.Stream(device=dev)
    sptr = int(stream.cuda_stream)

    def call(d, s):
        tkg.tkg_attention_fwd(w.B, w.H, w.Nq, w.Nkv, w.D, d["q"], d["k"], d["v"], d["o"], d["lse"], stream=s)

    def step():
        for i in range(batch):
            call(sets[i % n_sets], sptr)

    for _ in range(args.warmup):
        step()
    st = tkg.tkg_check_status(sptr)
    if st != tkg.TKG_OK:
        raise RuntimeError(f"warm-up failed: {tkg.status_string(st)}")

    spot = None
    if rank == 0 and not args.no_check:
        from oracle import attention as oa
        rows = np.array([0, w.Nq // 2, w.Nq - 1])
        ref = oa.attention_forward(x.q, x.k, x.v, heads=[(0, 0)], rows=rows)
        d = sets[(batch - 1) % n_sets]
        got = d["o"][0, 0][torch.from_numpy(rows).to(dev)].cpu().numpy().view(np.uint16)
        g = oa.bf16_decode(got)
        spot = float(np.linalg.norm(g - ref["o"][0]) / np.linalg.norm(ref["o"][0]))

    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    t0.record(stream)
    for s in range(args.steps):  # enqueued back to back; read afterwards
        step_ev[s][0].record(stream)
        step()
        step_ev[s][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    barrier(world)
    st = tkg.tkg_check_status(sptr)
    if st != tkg.TKG_OK:
        raise RuntimeError(f"timed run failed: {tkg.status_string(st)}")
    total_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    calls = args.steps * batch
    value = world * calls * w.flops / (total_ms * 1e-3) / 1e12
    per_call_ms = statistics.median(step_ms) / batch
    achieved = w.flops / (per_call_ms * 1e-3) / 1e12

    e2e = None
    if not args.no_e2e:
        host = {k: base[k].cpu().pin_memory() for k in ("q", "k", "v")}
        o_host = torch.empty(base["q"].shape, dtype=torch.int16).pin_memory()
        d = sets[0]
        h2d = sum(v.numel() * 2 for v in host.values())
        ea = torch.cuda.Event(enable_timing=True)
        eb = torch.cuda.Event(enable_timing=True)
        n = max(2, args.e2e_steps // 2)
        with torch.cuda.stream(stream):
            ea.record(stream)
            for _ in range(n):
                for k in ("q", "k", "v"):
                    d[k].copy_(host[k], non_blocking=True)
                call(d, sptr)
                o_host.copy_(d["o"], non_blocking=True)
            eb.record(stream)
        eb.synchronize()
        ms = ea.elapsed_time(eb) / n
        e2e = {"value": w.flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(o_host.numel() * 2), "ms_per_step": ms, "pipelined": "no (one stream)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt, n_rows, n_heads = attn_oracle_sample(x, w, args.cpu_s)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{n_rows} query rows x {n_heads} heads of the same workload ({dt:.1f} s, numpy float64, "
                         "BLAS threads on all host cores)"}

    peaks = load_peaks()
    peak = peaks["bf16_tflops_sustained"]
    line = {
        "metric": ATTN_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.description, "B": w.B, "H": w.H, "Nq": w.Nq, "Nkv": w.Nkv, "D": w.D,
                   "calls_per_step": batch, "parallelism": f"replicas{world}",
                   "l2": f"{n_sets} rotating input sets, {n_sets * per_set / 2**20:.0f} MiB > 129 MiB L2",
                   "launch_overlap": "programmatic dependent launch" if args.overlap == "on" else "off"},
        "median_call_ms": per_call_ms,
        "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms), "max": max(step_ms)},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic_bytes(args.workload),
                     "frac_of_burst_peak": achieved / peaks["bf16_tflops"],
                     "peak_source": f"{peaks['source']} bf16 sustained (back-to-back cuBLAS)"},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": calls, "clocks": clocks, "spot_check_rel_err": spot,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def relaunch_under_torchrun(n: int, argv) -> int:
    """--gpus N without torchrun: run this script under torchrun with N processes
    (one replica per GPU; rank 0 prints the line)."""
    import socket
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def main(argv=None):
    argv = list(sys.argv[1:] if argv is None else argv)
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["tkg", "reference"], default="tkg")
    p.add_argument("--workload", choices=sorted(synth.WORKLOADS) + sorted(ENCODERS) + sorted(synth.ATTN_WORKLOADS),
                   default=None, help="one workload (default: the GEMM suite, headline NVFP4 16384^3)")
    p.add_argument("--batch", type=int, default=0, help="GEMMs per step (default: per workload)")
    p.add_argument("--variant", type=int, default=0)
    p.add_argument("--group-m", type=int, default=0)
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--cpu-s", type=float, default=20.0,
                   help="seconds of oracle work for the headline's (or --workload's) cpu_baseline")
    p.add_argument("--cpu-s-other", type=float, default=2.0,
                   help="seconds of oracle work for each other suite workload's cpu_baseline")
    p.add_argument("--ref-step-s", type=float, default=3.0, help="seconds of oracle work per reference step")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-check", action="store_true", help="skip the parity gate (never for a reported number)")
    p.add_argument("--no-cublas", action="store_true", help="skip the cuBLAS comparison")
    p.add_argument("--graph", choices=["auto", "on", "off"], default="auto",
                   help="replay each step from a CUDA graph (auto: launch-bound workloads)")
    p.add_argument("--schedule", choices=sorted(SCHEDULE), default="static",
                   help="tile schedule: persistent static grid, dynamic (cluster launch control), one cluster per tile")
    p.add_argument("--overlap", choices=["on", "off"], default="on",
                   help="launch GEMMs as programmatic dependents of the previous kernel (on) or plainly (off)")
    p.add_argument("--split", choices=["on", "off"], default="on",
                   help="split the tiles of a persistent grid's last, at most half-full round along K")
    p.add_argument("--k-order", choices=["serpentine", "forward"], default="serpentine",
                   help="K walk of a CTA's odd-numbered tiles: from the last K block down (serpentine) or up")
    args = p.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    world_env = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return relaunch_under_torchrun(args.gpus, argv)
    if args.gpus != world_env:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world_env}; launch one process per GPU", file=sys.stderr)
        return 2
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        if args.workload in synth.ATTN_WORKLOADS:
            return run_reference_attention(args) if rank == 0 else 0
        return run_reference(args, world_env, rank)
    world, rank, local = dist_setup(args)
    if args.workload in ENCODERS:
        return run_encoder(args, world, rank, local)
    if args.workload in synth.ATTN_WORKLOADS:
        return run_attention(args, world, rank, local)
    return run_tkg(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
