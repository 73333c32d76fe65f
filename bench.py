#!/usr/bin/env python
"""(O, P) SDPA forward benchmark on one GB300 (or N independent replicas).

One step = one materialised-probability SDPA forward over the workload: scores,
masking, row statistics, exact P = exp(S - lse), P V and the stores of O and P,
all in the library's CUDA kernels, called through the C ABI.

Default workload: prefill 2k D128 (fp16, B=1, H=16, Sq=Skv=2048, D=128,
causal), the shape FlagOS-OP PR #10 "feat: add sdpa_math operator" quotes its
headline numbers on (first report's table: Ascend 910 Triton 1.369 ms against
2.776 ms for the native math backend; the P800 table: 2.392 ms), and the
largest single-GPU workload.  ``--config`` selects another of the synthetic
workloads.

Timing: W warm-up steps, then exactly K timed steps, each bracketed by CUDA
events on the launching stream.  Before every step L2 is flushed by writing a
256 MiB buffer and then reading another (the workloads' inputs and outputs
are smaller than the 129 MB L2, and the read leaves no dirty lines to write
back during the step), and a ~100 us device sleep keeps the GPU busy while the
host enqueues the step, so the events time the kernel, not the host call.  The
timed region is bracketed by a barrier and a device synchronise on both sides;
the reported time is the max over ranks.

``--impl reference`` times the CPU oracle as it stands (fp64 C, OpenMP over the
host cores) on a bounded sample of the same workload, extrapolated to the full
workload by rows.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sdpa_forward_materialised_gb300 import workloads as W  # noqa: E402

METRIC = "(O,P) fwd ms, TFLOPS and HBM GB/s; % of roofline (1×GB300)"
FLUSH_BYTES = 256 << 20
# Pages' own number for the default workload (Ascend 910, Triton, fp16): context only.
PAGES_MS = {"prefill1k_d64_f16": 0.515, "prefill2k_d128_f16": 1.369, "gqa1k_d128_f16": 0.810,
            "tail100_mask_f16": 0.219}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- accounting

def elem(dtype) -> int:
    return torch.empty((), dtype=dtype).element_size()


def algorithmic_bytes(w: W.Workload) -> int:
    """Q, K, V read once, mask read once at its broadcast shape, O and the full P written."""
    e = elem(w.torch_dtype)
    q = w.B * w.Hq * w.Sq * w.D * e
    kv = 2 * w.B * w.Hkv * w.Skv * w.D * e
    o = w.B * w.Hq * w.Sq * w.D * e
    p = w.B * w.Hq * w.Sq * w.Skv * e
    m = w.B * 1 * w.Sq * w.Skv if w.mask else 0
    return q + kv + o + p + m


def live_scores(w: W.Workload) -> int:
    per = 0
    for i in range(w.Sq):
        per += min(i + 1, w.Skv) if w.is_causal else w.Skv
    return w.B * w.Hq * per


def flops(w: W.Workload):
    """(algorithmic, dense) FLOPs: QK^T and PV, 2 per MAC; algorithmic counts
    live (causally visible) scores only, dense counts every score (the pages'
    TFLOPS convention)."""
    alg = 4 * w.D * live_scores(w)
    dense = 4 * w.D * w.B * w.Hq * w.Sq * w.Skv
    return alg, dense


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- clocks

class NvmlClocks:
    """In-process NVML queries (read-only: clocks, power, clock-event reasons)
    through ctypes, so the timed region gets samples however short it is."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        ok = False
        try:  # the physical GPU behind the torch device, by UUID
            uuid = str(torch.cuda.get_device_properties(torch_index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            ok = self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) == 0
        except Exception:
            ok = False
        if not ok:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES")
            idx = int(vis.split(",")[torch_index]) if vis and vis.split(",")[0].isdigit() else torch_index
            if self.lib.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(self.h)) != 0:
                raise OSError("no NVML handle")
        self.reason_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sample(self):
        ct = self.ct
        sm, mx, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(sm))        # NVML_CLOCK_SM
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ct.byref(mx))
        self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw))
        self.reason_fn(self.h, ct.byref(rs))
        return float(sm.value), float(mx.value), mw.value / 1000.0, int(rs.value)


class ClockSampler:
    """SM clock and clock-event reasons sampled every ~1 ms by a host thread
    through NVML while the timed region runs (falls back to nvidia-smi at
    100 ms when NVML cannot be loaded)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, torch_index: int, smi_index: int):
        self.torch_index = torch_index
        self.gpu = smi_index
        self.samples = []  # (time, sm_mhz, max_mhz, watts, [reasons])
        self.proc = None
        self.thread = None
        self.stop_flag = threading.Event()
        self.source = None

    def start(self):
        try:
            nv = NvmlClocks(self.torch_index)
            self.source = "nvml (in-process, ~1 ms)"
            self.thread = threading.Thread(target=self._poll_nvml, args=(nv,), daemon=True)
            self.thread.start()
            return
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi (100 ms)"
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read_smi, daemon=True)
        self.thread.start()

    def _poll_nvml(self, nv):
        while not self.stop_flag.is_set():
            try:
                sm, mx, w, rs = nv.sample()
            except Exception:
                return
            self.samples.append((time.perf_counter(), sm, mx, w,
                                 [n for bit, n in NvmlClocks.REASONS.items() if rs & bit]))
            time.sleep(0.001)

    def _read_smi(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm, mx = float(p[1]), float(p[2])
            except ValueError:
                continue
            try:
                w = float(p[3])
            except ValueError:
                w = None
            self.samples.append((time.perf_counter(), sm, mx, w,
                                 [n for n, val in zip(names, p[5:9]) if val.lower().startswith("active")]))

    def stop(self):
        self.stop_flag.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        rows = list(self.samples)
        inside = [r for r in rows if t0 <= r[0] <= t1]
        use = inside if inside else sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:1]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples_in_region": 0,
                    "source": self.source}
        reasons = sorted({n for r in use for n in r[4]})
        watts = [r[3] for r in use if r[3] is not None]
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "sm_mhz_min": min(r[1] for r in use), "power_w_max": max(watts) if watts else None,
                "reasons": reasons, "samples_in_region": len(inside), "source": self.source}


# ----------------------------------------------------------------------------- distributed

def smi_index(local: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis and vis.split(",")[0].strip().isdigit():
        return int(vis.split(",")[local])
    return local


def dist_setup(backend: str):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle

def oracle_sample_ms(w: W.Workload, budget_s: float, inputs=None):
    """Time the oracle on a row sample sized for ~budget_s; return
    (ms extrapolated to the full workload, threads, sample description)."""
    import numpy as np
    import oracle
    q, k, v, m = inputs if inputs is not None else W.make_inputs(w)
    threads = max(1, os.cpu_count() or 1)
    total = w.B * w.Hq * w.Sq
    rng = np.random.default_rng(0)
    probe = np.sort(rng.choice(total, size=min(total, max(threads * 2, 16)), replace=False))
    t0 = time.perf_counter()
    oracle.oracle_fwd(q, k, v, m, is_causal=w.is_causal, scale=w.scale, rows=probe, nthreads=threads)
    per_row = (time.perf_counter() - t0) / len(probe)
    n = int(min(total, max(len(probe), budget_s / max(per_row, 1e-9))))
    rows = np.sort(rng.choice(total, size=n, replace=False))
    t0 = time.perf_counter()
    oracle.oracle_fwd(q, k, v, m, is_causal=w.is_causal, scale=w.scale, rows=rows, nthreads=threads)
    dt = time.perf_counter() - t0
    if n < total:
        ms = dt * 1e3 * total / n
        sample = (f"{n} of {total} query rows (each over all {w.Skv} keys), fp64 C oracle, "
                  f"{threads} OpenMP threads, {dt:.2f} s, extrapolated to all rows")
        return ms, threads, sample
    # the whole workload fits the budget: repeat it to fill the budget, report the mean pass
    reps = int(min(1000, max(1, budget_s / max(dt, 1e-6))))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.oracle_fwd(q, k, v, m, is_causal=w.is_causal, scale=w.scale, rows=rows, nthreads=threads)
    dt = time.perf_counter() - t0
    ms = dt * 1e3 / reps
    sample = (f"all {total} query rows (each over all {w.Skv} keys), fp64 C oracle, {threads} OpenMP threads, "
              f"{reps} passes in {dt:.2f} s, mean pass")
    return ms, threads, sample


def run_reference_bwd(args, w: W.Workload):
    """The oracle backward (on one (batch, KV head) group, extrapolated), as the
    reference arm of --pass bwd."""
    import oracle
    q, k, v, m = W.make_inputs(w)
    _, Po, _ = oracle.oracle_fwd(q, k, v, m, is_causal=w.is_causal, scale=w.scale,
                                 nthreads=max(1, os.cpu_count() or 1))
    P = torch.from_numpy(Po).to(w.torch_dtype)
    g = torch.Generator().manual_seed(w.seed + 100)
    go = torch.randn(w.B, w.Hq, w.Sq, w.D, generator=g).to(w.torch_dtype)
    gp = torch.randn(P.shape, generator=g).to(w.torch_dtype)
    vals = [oracle_bwd_sample_ms(w, q, k, v, P, go, gp) for _ in range(max(1, args.steps))]
    ms = statistics.mean(x[0] for x in vals)
    line = {
        "impl": "reference", "metric": METRIC_BWD, "value": ms, "unit": "ms", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "pass": "bwd"},
        "cpu_baseline": {"value": ms, "unit": "ms", "cores": 1, "kind": "oracle", "sample": vals[0][2]},
        "e2e": {"value": ms, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args, w: W.Workload):
    world, rank, _ = dist_setup("gloo")
    if rank != 0:
        return 0
    if args.pass_ == "bwd":
        return run_reference_bwd(args, w)
    inputs = W.make_inputs(w)
    per_step = max(0.05, min(args.cpu_budget, 10.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample_ms(w, per_step / 4, inputs)
    vals, threads, sample = [], 1, ""
    for _ in range(args.steps):
        ms, threads, sample = oracle_sample_ms(w, per_step, inputs)
        vals.append(ms)
    ms = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": ms, "unit": "ms", "n_gpus": max(world, args.gpus),
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, **{k: v for k, v in w.describe().items() if k != "name"}},
        "cpu_baseline": {"value": ms, "unit": "ms", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": ms, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm

def run_ours(args, w: W.Workload):
    import sdpa_forward_materialised_gb300 as sm
    world, rank, local = dist_setup("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sm.load_library()

    q, k, v, m = W.make_inputs(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    md = m.to(dev) if m is not None else None
    kind = sm.MASK_NONE if md is None else (sm.MASK_BOOL if md.dtype == torch.bool else sm.MASK_ADDITIVE)
    O, P = sm.empty_outputs(qd, vd, w.Skv)
    plan = sm.sdpa_math_plan(qd, kd, vd, md, is_causal=w.is_causal, scale=w.scale, out=O, probs=P,
                             variant=args.variant)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_rd = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # write 256 MiB (evicts the workload from L2), then read another 256 MiB
        # so the write-back of those dirty lines does not land inside the timed
        # step; then keep the GPU busy for ~100 us while the host enqueues the
        # step, so host-side call overhead stays outside the events
        flush.zero_()
        flush_rd.sum()
        torch.cuda._sleep(200_000)

    def step():
        sm.sdpa_math_fwd_ex(qd, kd, vd, md, kind, w.is_causal, w.scale, O, P, None, args.variant, stream)

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize(dev)
    sm.sdpa_math_device_status(stream)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local, smi_index(local))
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(args.steps):
        flush_l2()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    t1 = time.perf_counter()
    time.sleep(0.15)
    sampler.stop()
    sm.sdpa_math_device_status(stream)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = max_over_ranks(statistics.mean(step_ms), world, dev)
    clocks = sampler.summary(t0, t1)

    # end to end through the same C-ABI call, host buffers in pinned memory
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    hm = m.pin_memory() if m is not None else None
    hO = torch.empty(O.shape, dtype=O.dtype).pin_memory()
    hP = torch.empty(P.shape, dtype=P.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv) + ((hm,) if hm is not None else ()))
    d2h = hO.numel() * hO.element_size() + hP.numel() * hP.element_size()
    e2e_steps = max(3, min(args.steps, 50))

    def e2e_step():
        qd.copy_(hq, non_blocking=True)
        kd.copy_(hk, non_blocking=True)
        vd.copy_(hv, non_blocking=True)
        if hm is not None:
            md.copy_(hm, non_blocking=True)
        step()
        hO.copy_(O, non_blocking=True)
        hP.copy_(P, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    es.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    ee.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = max_over_ranks(es.elapsed_time(ee) / e2e_steps, world, dev)

    peaks, peak_src = load_peaks()
    nbytes = algorithmic_bytes(w)
    alg, dense = flops(w)
    gbs = nbytes / (ms * 1e-3) / 1e9
    hbm_peak = float(peaks["hbm_gbs"])
    traffic = ncu_traffic(w, plan["variant"])
    line = {
        "metric": METRIC, "value": ms, "unit": "ms", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": (ms / PAGES_MS[w.name]) if w.name in PAGES_MS else None,
        "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Skv": w.Skv,
                   "D": w.D, "is_causal": w.is_causal, "mask": w.mask, "seed": w.seed,
                   "variant": plan["variant"], "l2": "flushed before every step (256 MiB write, then 256 MiB read)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "vs_baseline_ref": "Ascend 910 Triton ms from the pages (other hardware, context only)"},
        "tflops_alg": alg / (ms * 1e-3) / 1e12, "tflops_dense": dense / (ms * 1e-3) / 1e12,
        "hbm_gbs": gbs, "algorithmic_bytes": nbytes,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": gbs / hbm_peak, "traffic": traffic,
                     "traffic_kind": ("ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch; DRAM only: "
                                      "ncu flushes the caches before its replay, and P lines still dirty in the "
                                      "129 MB L2 when the kernel ends are written back after it, uncounted"),
                     "peak_source": f"{peak_src} (copy bandwidth, burst)"},
        "e2e": {"value": e2e_ms, "unit": "ms", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * plan["launches"],
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cms, threads, sample = oracle_sample_ms(w, args.cpu_budget, (q, k, v, m))
        line["cpu_baseline"] = {"value": cms, "unit": "ms", "cores": threads, "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------- backward

METRIC_BWD = "(dq,dk,dv) bwd ms and HBM GB/s; % of roofline (1×GB300)"


def bwd_bytes(w: W.Workload) -> int:
    """Algorithmic bytes of the backward: q, k, v, P, dout, dprobs read once;
    dq, dk, dv and the fp32 per-row sums written once."""
    e = 4 if w.dtype == "f32" else 2
    rows = w.B * w.Hq * w.Sq
    # D == Dv for every workload: q, dout, dq rows; k, v, dk, dv rows; P and dprobs
    return e * (3 * rows * w.D + 4 * w.B * w.Hkv * w.Skv * w.D + 2 * rows * w.Skv) + 4 * rows


def bwd_tc_eligible(w: W.Workload) -> bool:
    """Whether sdpa_math_bwd runs this workload on the tensor-core kernels
    (f16/bf16, D == Dv in {64, 128}, contiguous P rows on 16-byte boundaries)."""
    return w.dtype in ("f16", "bf16") and w.D in (64, 128) and w.Skv % 8 == 0


def oracle_bwd_sample_ms(w: W.Workload, q, k, v, P, go, gp):
    """The oracle backward on one (batch, KV head) group, extrapolated to all
    B * Hkv groups (groups are independent and equal in size)."""
    import oracle
    g = w.Hq // w.Hkv
    sl = lambda t, H: t[:1, :H].contiguous()
    qs, ks, vs = sl(q, g), sl(k, 1), sl(v, 1)
    Ps, gos, gps = sl(P, g), sl(go, g), sl(gp, g)
    threads = max(1, os.cpu_count() or 1)
    t0 = time.perf_counter()
    oracle.oracle_bwd(qs, ks, vs, Ps, gos, gps, scale=w.scale, nthreads=threads)
    dt = time.perf_counter() - t0
    groups = w.B * w.Hkv
    sample = (f"1 of {groups} (batch, KV head) groups ({g} query heads x {w.Sq} rows x {w.Skv} keys), "
              f"fp64 C oracle backward, {dt:.2f} s, extrapolated to all groups (one thread per group)")
    return dt * 1e3 * groups, 1, sample


def run_ours_bwd(args, w: W.Workload):
    import sdpa_forward_materialised_gb300 as sm
    world, rank, local = dist_setup("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sm.load_library()
    q, k, v, m = W.make_inputs(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    md = m.to(dev) if m is not None else None
    O, P = sm.sdpa_math(qd, kd, vd, md, is_causal=w.is_causal, scale=w.scale)  # the forward's map
    g = torch.Generator().manual_seed(w.seed + 100)
    go = torch.randn(O.shape, generator=g).to(w.torch_dtype)
    gp = torch.randn(P.shape, generator=g).to(w.torch_dtype)
    god, gpd = go.to(dev), gp.to(dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    rowsum = torch.empty(qd.shape[:3], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_rd = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        flush.zero_()
        flush_rd.sum()
        torch.cuda._sleep(200_000)

    def step():
        sm.sdpa_math_bwd(qd, kd, vd, P, god, gpd, w.scale, dq, dk, dv, rowsum, stream)

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize(dev)
    sm.sdpa_math_device_status(stream)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local, smi_index(local))
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(args.steps):
        flush_l2()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    t1 = time.perf_counter()
    time.sleep(0.15)
    sampler.stop()
    sm.sdpa_math_device_status(stream)
    ms = max_over_ranks(statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends)), world, dev)
    clocks = sampler.summary(t0, t1)

    # end to end: inputs from pinned host memory, gradients back to it
    hosts = [t.pin_memory() for t in (q, k, v, P.cpu(), go, gp)]
    devs = [qd, kd, vd, P, god, gpd]
    outs = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk, dv)]
    h2d = sum(t.numel() * t.element_size() for t in hosts)
    d2h = sum(t.numel() * t.element_size() for t in outs)
    e2e_steps = max(3, min(args.steps, 50))

    def e2e_step():
        for d, h in zip(devs, hosts):
            d.copy_(h, non_blocking=True)
        step()
        for o, d in zip(outs, (dq, dk, dv)):
            o.copy_(d, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    es.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    ee.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(es.elapsed_time(ee) / e2e_steps, world, dev)

    peaks, peak_src = load_peaks()
    nbytes = bwd_bytes(w)
    gbs = nbytes / (ms * 1e-3) / 1e9
    hbm_peak = float(peaks["hbm_gbs"])
    line = {
        "metric": METRIC_BWD, "value": ms, "unit": "ms", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "pass": "bwd", "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq,
                   "Skv": w.Skv, "D": w.D, "is_causal": w.is_causal, "mask": w.mask, "seed": w.seed,
                   "kernels": ("tensor-core (tcgen05) rows + keys kernels" if bwd_tc_eligible(w)
                               else "CUDA-core rows + keys kernels"),
                   "l2": "flushed before every step (256 MiB write, then 256 MiB read)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "hbm_gbs": gbs, "algorithmic_bytes": nbytes,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": gbs / hbm_peak,
                     # DRAM bytes of the rows + keys kernels per step, from the ncu summary
                     "traffic": ncu_traffic(w, "bwd", key=f"{w.name}:bwd") if bwd_tc_eligible(w) else None,
                     "peak_source": f"{peak_src} (copy bandwidth, burst)"},
        "e2e": {"value": e2e_ms, "unit": "ms", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * 2,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cms, threads, sample = oracle_bwd_sample_ms(w, q, k, v, P.cpu(), go, gp)
        line["cpu_baseline"] = {"value": cms, "unit": "ms", "cores": threads, "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def ncu_traffic(w: W.Workload, variant: str, key: str = None):
    """DRAM bytes per launch from the committed ncu summary, only when it was
    taken on the kernel sources as they are now (else None).  ``key`` names a
    summary other than the workload's forward one (e.g. its backward)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        from sdpa_forward_materialised_gb300 import _build
        fp = _build.source_fingerprint()
        with open(path) as f:
            d = json.load(f)
        ent = d.get(key or w.name)
        if ent and ent.get("sources") == fp and ent.get("variant") == variant:
            return ent["dram_bytes_per_launch"]
    except Exception:
        return None
    return None


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="prefill2k_d128_f16", choices=sorted(W.BY_NAME))
    ap.add_argument("--variant", default="auto",
                    choices=["auto", "simt", "twopass", "paired", "fused", "onesweep", "decode", "split", "tcdecode"])
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd"], default="fwd",
                    help="fwd: the (O, P) forward (the headline); bwd: the backward for dout and dprobs")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps
    w = W.BY_NAME[args.config]
    if args.impl == "reference":
        return run_reference(args, w)
    if args.pass_ == "bwd":
        return run_ours_bwd(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
