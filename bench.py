#!/usr/bin/env python
"""Throughput of the fused attention forward on one GB300 (or N, as replicas).

A step is one pass of the hot path over one batch: the non-causal and the
causal forward of the headline workload (B=1, H=32, N=4096, d=128, bf16 Q/K/V
i.i.d. N(0,1), scale 1/sqrt(d)).  FLOPs are counted as 4*B*H*N^2*d for the
non-causal pass and half that for the causal one.  Inputs are resident in
device memory when timing starts; L2 is flushed (a 256 MiB write) before
every step, outside the per-step CUDA events.  The JSON line also carries the
roofline of the dominant kernel, the fp64 oracle timed on the host as a CPU
baseline, an end-to-end figure through host buffers, clocks sampled with
nvidia-smi, and the number of kernels launched.

--impl reference times the oracle itself on the host (bounded samples of the
same workload); under torchrun only rank 0 does so.
"""
import os

os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_attention_20_gb300.inputs import HEADLINE, WORKLOADS, make_grad, make_qkv  # noqa: E402

METRIC = "attn fwd TFLOP/s (bf16, causal/non-causal) N=4096 d=128; % of GB300 BF16 peak"
KERNEL_SOURCES = [
    os.path.join(ROOT, "exact_attention_20_gb300", "csrc", n)
    for n in ("fa_fwd_kernel.cuh", "sm103_ptx.cuh", "fa_api.cu")
]
BWD_KERNEL_SOURCES = [
    os.path.join(ROOT, "exact_attention_20_gb300", "csrc", n)
    for n in ("fa_bwd_kernel.cuh", "sm103_ptx.cuh", "fa_bwd.cu")
]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")
FLUSH_BYTES = 256 << 20
# tcgen05.mma (M = 128, kind::f16, bf16 in, fp32 accumulate) retires
# 8,192 flop per clock per SM (measured on this GPU by a probe of the
# instruction alone); times the SMs and the SM clock it is the per-clock peak
TC_FLOP_PER_CLK_SM = 8192
# NVIDIA's dense bf16 figure per GB300 GPU
SPEC_BF16_TFLOPS = 2250.0


def median(xs):
    ys = sorted(xs)
    n = len(ys)
    return ys[n // 2] if n % 2 else 0.5 * (ys[n // 2 - 1] + ys[n // 2])


def flops(w, causal):
    f = 4.0 * w.B * w.H * w.N * w.N * w.d
    return f / 2 if causal else f


def kernel_hash(sources=None):
    h = hashlib.sha256()
    for p in sources or KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("bf16_tflops", 1900.0), d.get("bf16_tflops_sustained"), "measured"
    return 1900.0, 1700.0, "fallback"


def recorded_traffic(workload, causal):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel sources changed since those counters were taken."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    if d.get("kernel_hash") != kernel_hash():
        return None
    return d.get("bytes_per_launch", {}).get(f"{workload}:{'causal' if causal else 'non-causal'}")


def recorded_bwd_traffic(workload, causal):
    """The same for fa_bwd_kernel (its own sources and record)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f).get("backward", {})
    if d.get("kernel_hash") != kernel_hash(BWD_KERNEL_SOURCES):
        return None
    return d.get("bytes_per_launch", {}).get(f"{workload}:{'causal' if causal else 'non-causal'}")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        # samples inside the timed region (second resolution), else the last
        # second of warm-up before it
        inside = [r for r in rows if self.t0 - 1 <= r[0] <= self.t1 + 1]
        use = inside or rows
        mhz = sorted(r[1] for r in use)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use),
                "window": "timed region +-1 s" if inside else "whole run"}


def dist_setup(n_gpus):
    if n_gpus <= 1 or "RANK" not in os.environ:
        return 0, 1, 0
    import torch.distributed as dist
    rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    torch.cuda.set_device(local)
    dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample_rate(w, n_heads, seed=0):
    """Runs the fp64 oracle on n_heads heads of the workload, both masks;
    returns (TFLOP/s on the sample, seconds, description)."""
    import numpy as np

    import oracle

    q, k, v = make_qkv(1, n_heads, w.N, w.d, seed=seed, values=w.values)
    qf, kf, vf = (t.float().numpy().astype(np.float64) for t in (q, k, v))
    masks = [c for c in (False, True) if c in w.causal]
    t0 = time.perf_counter()
    for causal in masks:
        oracle.attention(qf, kf, vf, w.scale, causal)
    dt = time.perf_counter() - t0
    fl = sum(4.0 * n_heads * w.N * w.N * w.d / (2 if c else 1) for c in masks)
    names = " and ".join("causal" if c else "non-causal" for c in masks)
    desc = f"{n_heads} of {w.B * w.H} heads of {w.name}, {names}, fp64 numpy"
    return fl / dt / 1e12, dt, desc


def cpu_sample_heads(w, requested=None):
    """Heads for the oracle's timed sample: as requested, else about 100
    GFLOP of work (eight heads of the headline shape), at least one."""
    if requested:
        return requested
    per_head = sum(4.0 * w.N * w.N * w.d / (2 if c else 1) for c in w.causal)
    return max(1, min(w.B * w.H, int(round(1.03e11 / per_head))))


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    for _ in range(args.warmup):
        oracle_sample_rate(w, 1)
    times, rates = [], []
    desc = ""
    for i in range(args.steps):
        r, dt, desc = oracle_sample_rate(w, 1, seed=i)
        rates.append(r)
        times.append(dt)
    fl = sum(4.0 * w.N * w.N * w.d / (2 if c else 1) for c in w.causal)
    value = fl * len(times) / sum(times) / 1e12
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "masks": ["causal" if c else "non-causal" for c in w.causal], "sample": "1 head per step"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": desc + " per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def time_workload(fa, w, dev, steps, warmup, flush, peak_burst, sms, mhz):
    """Median ms per mask of one fa_fwd call on workload w (L2 flushed before
    each call, outside the events), with its fractions of the peaks."""
    q, k, v = make_qkv(w.B, w.H, w.N, w.d, seed=4321, values=w.values, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=dev)
    out = {}
    for causal in [c for c in (False, True) if c in w.causal]:
        for _ in range(warmup):
            fa.fa_fwd(q, k, v, o, lse, causal=causal, scale=w.scale)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for e0, e1 in evs:
            flush.zero_()
            e0.record()
            fa.fa_fwd(q, k, v, o, lse, causal=causal, scale=w.scale)
            e1.record()
        torch.cuda.synchronize(dev)
        ms = median([a.elapsed_time(b) for a, b in evs])
        tf = flops(w, causal) / (ms * 1e-3) / 1e12
        clock_peak = sms * TC_FLOP_PER_CLK_SM * mhz * 1e6 / 1e12 if mhz else None
        out["causal" if causal else "non-causal"] = {
            "ms": ms, "tflops": tf, "frac_of_measured_peak": tf / peak_burst,
            "frac_of_clock_peak": tf / clock_peak if clock_peak else None,
            "frac_of_spec_peak": tf / SPEC_BF16_TFLOPS}
    del q, k, v, o, lse
    return out


def run_ours(args):
    from exact_attention_20_gb300 import build as fa_build

    rank, world, local = dist_setup(args.gpus)
    if rank == 0 or world == 1:
        fa_build.build()
    barrier(world)
    from exact_attention_20_gb300 import fa

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    masks = [c for c in (False, True) if c in w.causal]
    q, k, v = make_qkv(w.B, w.H, w.N, w.d, seed=1234 + rank, values=w.values, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(evs=None):
        for i, causal in enumerate(masks):
            if evs is not None:
                evs[i][0].record(stream)
            fa.fa_fwd(q, k, v, o, lse, causal=causal, scale=w.scale, stream=stream)
            if evs is not None:
                evs[i][1].record(stream)

    sampler = ClockSampler(local)
    if not args.quick:
        sampler.start()
    # warm-up: at least args.warmup steps and (unless --quick) one second of work
    t_warm = time.time()
    n = 0
    while n < args.warmup or (not args.quick and time.time() - t_warm < 1.0):
        flush.zero_()
        step()
        n += 1
        if n % 8 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)

    evs = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
            for _ in masks] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.mark("t0")
    wall0 = time.perf_counter()
    for s in range(args.steps):
        flush.zero_()
        step(evs[s])
    torch.cuda.synchronize(dev)
    wall1 = time.perf_counter()
    sampler.mark("t1")
    barrier(world)
    per_mask_ms = [[evs[s][i][0].elapsed_time(evs[s][i][1]) for s in range(args.steps)]
                   for i in range(len(masks))]
    # the median step (the masks run interleaved, one call each per step)
    step_ms = median([sum(per_mask_ms[i][s] for i in range(len(masks))) for s in range(args.steps)])
    step_ms = max_over_ranks(step_ms, world)
    step_flops = sum(flops(w, c) for c in masks)
    value = world * step_flops / (step_ms * 1e-3) / 1e12
    if args.quick:
        if rank == 0:
            print(json.dumps({"quick": True, "workload": w.name, "ms_per_step": step_ms,
                              "value": value, "unit": "TFLOP/s"}), flush=True)
        return

    # end to end through the public API from pinned host buffers
    qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
    oh = [torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True) for _ in masks]
    lh = [torch.empty(lse.shape, dtype=torch.float32, pin_memory=True) for _ in masks]
    ws = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))

    def e2e_step():
        for t_d, t_h in zip(ws, (qh, kh, vh)):
            t_d.copy_(t_h, non_blocking=True)
        for i, causal in enumerate(masks):
            fa.fa_fwd(ws[0], ws[1], ws[2], o, lse, causal=causal, scale=w.scale, stream=stream)
            oh[i].copy_(o, non_blocking=True)
            lh[i].copy_(lse, non_blocking=True)

    for _ in range(max(3, args.warmup)):
        e2e_step()
    torch.cuda.synchronize(dev)
    e_steps = max(3, min(args.steps, 20))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(e_steps):
        flush.zero_()
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, world)
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = sum(t.numel() * t.element_size() for t in oh + lh)

    clocks = sampler.stop()
    if rank != 0:
        return

    launches_per_step = fa.KERNELS_PER_CALL * len(masks)
    peak_burst, peak_sustained, peak_kind = measured_peaks()
    # the per-clock peak: every SM's tensor core at the SM clock sampled
    # during the timed region (the pages define 100 % as operations per clock
    # per SM times the clock the kernel ran at)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = clocks["sm_mhz"] if clocks else None
    clock_peak = sms * TC_FLOP_PER_CLK_SM * mhz * 1e6 / 1e12 if mhz else None
    dom = 0  # the first mask of the step: non-causal where the workload has it
    dom_ms = median(per_mask_ms[dom])
    achieved = flops(w, masks[dom]) / (dom_ms * 1e-3) / 1e12
    per_mask = {}
    for i, c in enumerate(masks):
        ms = median(per_mask_ms[i])
        tf = flops(w, c) / (ms * 1e-3) / 1e12
        per_mask["causal" if c else "non-causal"] = {
            "ms": ms, "ms_mean": sum(per_mask_ms[i]) / len(per_mask_ms[i]), "tflops": tf,
            "frac_of_measured_peak": tf / peak_burst,
            "frac_of_clock_peak": tf / clock_peak if clock_peak else None,
            "frac_of_spec_peak": tf / SPEC_BF16_TFLOPS}

    # the other configurations of the method (parity cases; reported beside
    # the headline, not part of its value), same protocol, after the timed
    # region and its clock samples
    others = {}
    if world == 1 and not args.no_other_workloads:
        for name, ow in WORKLOADS.items():
            if name == w.name:
                continue
            others[name] = time_workload(fa, ow, dev, max(10, min(args.steps, 50)), 3, flush, peak_burst, sms, mhz)

    cpu = None
    if not args.no_cpu_baseline:
        rate, dt, desc = oracle_sample_rate(w, cpu_sample_heads(w, args.cpu_heads))
        cpu = {"value": rate, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{desc}; {dt:.1f} s; BLAS products on all cores, elementwise steps single-threaded"}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "masks": ["causal" if c else "non-causal" for c in masks],
                   "scale": w.scale, "l2": "flushed before every step (256 MiB write, outside the events)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "per_mask": per_mask,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_burst,
                     "unit": "TFLOP/s", "frac": achieved / peak_burst,
                     "peak_kind": f"{peak_kind} bf16 dense, burst",
                     "clock_peak": clock_peak, "frac_of_clock_peak": achieved / clock_peak if clock_peak else None,
                     "clock_peak_kind": (f"{sms} SMs x {TC_FLOP_PER_CLK_SM} flop/clk/SM (tcgen05.mma M=128 kind::f16, "
                                         f"measured by a probe on this GPU) x the median SM clock sampled in the "
                                         f"timed region"),
                     "spec_peak": SPEC_BF16_TFLOPS, "frac_of_spec_peak": achieved / SPEC_BF16_TFLOPS,
                     "spec_peak_kind": "NVIDIA's dense bf16 figure per GB300 GPU (36 PFLOP/s per 8 GPUs with 2:4 sparsity)",
                     "statistic": "median of the timed steps",
                     "kernel": f"fa_fwd_kernel<{w.d},{str(masks[dom]).lower()}>",
                     "timed_span": "one fa_fwd call = one launch of this kernel (split items merged inside it)",
                     "traffic": recorded_traffic(w.name, masks[dom])},
        "other_workloads": others or None,
        "cpu_baseline": cpu,
        "e2e": {"value": world * step_flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clocks,
        "wall_s_timed_region": wall1 - wall0,
    }
    print(json.dumps(line), flush=True)


DECODE_SHAPES = [(1, 32, 1, 32768, 128), (1, 32, 128, 32768, 128)]  # B, H, Nq, Nk, d


def run_decode(args):
    """Few query rows over long keys (fa_fwd_rect, non-causal): HBM-bound.

    The algorithmic bytes are Q, K, V read once and O, LSE written once; the
    useful FLOPs (4 B H Nq Nk d) are negligible.  The value is the bytes per
    second of the one-query-row shape against the measured copy bandwidth.
    """
    from exact_attention_20_gb300 import build as fa_build

    fa_build.build()
    from exact_attention_20_gb300 import fa

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    # L2 is evicted before every call by READING a 256 MiB buffer: a written
    # flush would leave up to an L2's worth of dirty lines, whose write-back
    # then competes with this HBM-bound kernel's reads inside the timed
    # region.  K and V (537 MB) are larger than L2 in any case.
    flush = torch.zeros(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        hbm = json.load(f).get("hbm_gbs", 6800.0)
    sampler = ClockSampler(0)
    sampler.start()
    per_shape = {}
    for B, H, Nq, Nk, d in DECODE_SHAPES:
        q, _, _ = make_qkv(B, H, Nq, d, seed=1, device=dev)
        _, k, v = make_qkv(B, H, Nk, d, seed=2, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
        for _ in range(args.warmup):
            fa.fa_fwd_rect(q, k, v, o, lse, scale=d ** -0.5)
        torch.cuda.synchronize(dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        sampler.mark("t0")
        for e0, e1 in evs:
            flush.max()
            e0.record()
            fa.fa_fwd_rect(q, k, v, o, lse, scale=d ** -0.5)
            e1.record()
        torch.cuda.synchronize(dev)
        sampler.mark("t1")
        ms = median([a.elapsed_time(b) for a, b in evs])
        nbytes = B * H * (2 * Nq * d * 2 + 2 * Nk * d * 2 + Nq * 4)
        grid, nsplit = fa.plan(B, H, Nq, d, False, n_keys=Nk)
        per_shape[f"B{B}-H{H}-Nq{Nq}-Nk{Nk}-d{d}"] = {
            "ms": ms, "gbs": nbytes / (ms * 1e-3) / 1e9, "frac_of_measured_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm,
            "algorithmic_bytes": nbytes, "useful_tflops": 4.0 * B * H * Nq * Nk * d / (ms * 1e-3) / 1e12,
            "ctas": grid, "split_items": nsplit}
    clocks = sampler.stop()
    first = next(iter(per_shape.values()))
    print(json.dumps({
        "metric": "attn fwd decode: algorithmic bytes per second, few query rows over 32768 keys (bf16, non-causal)",
        "value": first["gbs"], "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "decode", "shapes": list(per_shape),
                   "l2": "evicted before every call by reading a 256 MiB buffer (outside the events); "
                         "K and V (537 MB) are larger than L2"},
        "per_shape": per_shape,
        "roofline": {"bound": "hbm", "achieved": first["gbs"], "peak": hbm, "unit": "GB/s",
                     "frac": first["gbs"] / hbm, "peak_kind": "measured copy bandwidth"},
        "clocks": clocks}), flush=True)


def run_backward(args):
    """dQ, dK, dV of the workload through fa_bwd, both masks, L2 flushed before every call.

    One fa_bwd call is three launches (prep: D, L and the zeroed dQ
    accumulator; the fused backward kernel; the dQ conversion), all inside
    the timed span.  The algorithmic FLOPs are the backward's five products
    (S, dP, dV, dK, dQ), 10 B H N^2 d non-causal and half that causal.
    """
    from exact_attention_20_gb300 import build as fa_build

    fa_build.build()
    from exact_attention_20_gb300 import fa

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    peak, _, peak_src = measured_peaks()
    q, k, v = make_qkv(w.B, w.H, w.N, w.d, seed=0, values=w.values, device=dev)
    do = make_grad(w.B, w.H, w.N, w.d, seed=1, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    sampler = ClockSampler(0)
    sampler.start()
    per_mask = {}
    for causal in w.causal:
        o, lse = fa.attention(q, k, v, causal=causal, scale=w.scale)
        for _ in range(args.warmup):
            fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal=causal, scale=w.scale)
        torch.cuda.synchronize(dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        sampler.mark("t0")
        for e0, e1 in evs:
            flush.zero_()
            e0.record()
            fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal=causal, scale=w.scale)
            e1.record()
        torch.cuda.synchronize(dev)
        sampler.mark("t1")
        ms = median([a.elapsed_time(b) for a, b in evs])
        f = 2.5 * flops(w, causal)
        per_mask["causal" if causal else "non-causal"] = {
            "ms": ms, "tflops": f / (ms * 1e-3) / 1e12, "frac_of_measured_peak": f / (ms * 1e-3) / 1e12 / peak}
    clocks = sampler.stop()
    total_f = sum(2.5 * flops(w, c) for c in w.causal)
    total_ms = sum(m["ms"] for m in per_mask.values())
    value = total_f / (total_ms * 1e-3) / 1e12
    dom = max(per_mask, key=lambda m: per_mask[m]["ms"])
    print(json.dumps({
        "metric": "attn bwd TFLOP/s (bf16, dQ dK dV, causal/non-causal); % of GB300 BF16 peak",
        "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "masks": list(per_mask),
                   "l2": "flushed before every call (256 MiB write, outside the events)"},
        "per_mask": per_mask,
        "roofline": {"bound": "tensor", "achieved": per_mask[dom]["tflops"], "peak": peak, "unit": "TFLOP/s",
                     "frac": per_mask[dom]["frac_of_measured_peak"], "peak_kind": f"{peak_src} bf16 dense, burst",
                     "timed_span": "one fa_bwd call: prep, fa_bwd_kernel, dQ conversion", "mask": dom,
                     "kernel": "fa_bwd_kernel", "traffic": recorded_bwd_traffic(w.name, dom == "causal")},
        "gpu_launches": args.steps * len(per_mask) * fa.BWD_KERNELS_PER_CALL,
        "clocks": clocks}), flush=True)


def run_fp8(args):
    """The forward on FP8 operands (fa_fwd_fp8), both masks, L2 flushed before every call.

    Inputs are quantised once (fa_quantize_fp8) and stay resident; the timed
    span is one fa_fwd_fp8 call, the same single kernel launch as fa_fwd.
    FLOPs are the forward's (4 B H N^2 d, half causal); the roofline peak is
    the measured bf16 peak times the nominal FP8 / bf16 ratio (2).  The
    quantisation of Q, K and V is timed separately.
    """
    from exact_attention_20_gb300 import build as fa_build

    fa_build.build()
    from exact_attention_20_gb300 import fa

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    peak16, _, peak_src = measured_peaks()
    peak8 = 2.0 * peak16
    q, k, v = make_qkv(w.B, w.H, w.N, w.d, seed=0, values=w.values, device=dev)
    q8, sq = fa.quantize_fp8(q, 0)
    k8, sk = fa.quantize_fp8(k, 0)
    vt8, sv = fa.quantize_fp8(v, 1)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    sampler = ClockSampler(0)
    sampler.start()
    per_mask = {}
    for causal in w.causal:
        for _ in range(args.warmup):
            fa.fa_fwd_fp8(q8, k8, vt8, sq, sk, sv, o, lse, causal=causal, scale=w.scale)
        torch.cuda.synchronize(dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        sampler.mark("t0")
        for e0, e1 in evs:
            flush.zero_()
            e0.record()
            fa.fa_fwd_fp8(q8, k8, vt8, sq, sk, sv, o, lse, causal=causal, scale=w.scale)
            e1.record()
        torch.cuda.synchronize(dev)
        sampler.mark("t1")
        ms = median([a.elapsed_time(b) for a, b in evs])
        f = flops(w, causal)
        per_mask["causal" if causal else "non-causal"] = {
            "ms": ms, "tflops": f / (ms * 1e-3) / 1e12, "frac_of_fp8_peak": f / (ms * 1e-3) / 1e12 / peak8}
    # the quantisation of all three inputs, one call each, L2 flushed first
    qevs = []
    for _ in range(max(3, args.steps // 10)):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fa.quantize_fp8(q, 0)
        fa.quantize_fp8(k, 0)
        fa.quantize_fp8(v, 1)
        e1.record()
        qevs.append((e0, e1))
    torch.cuda.synchronize(dev)
    quant_ms = sum(a.elapsed_time(b) for a, b in qevs) / len(qevs)
    clocks = sampler.stop()
    total_f = sum(flops(w, c) for c in w.causal)
    total_ms = sum(m["ms"] for m in per_mask.values())
    dom = max(per_mask, key=lambda m: per_mask[m]["ms"])
    print(json.dumps({
        "metric": "attn fwd TFLOP/s on FP8 (e4m3) operands, causal/non-causal; % of GB300 FP8 peak",
        "value": total_f / (total_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms, "higher_is_better": True, "dtype": "e4m3 (fp32 accumulate)",
        "data": "synthetic", "config": {"workload": w.name, "masks": list(per_mask),
                                        "l2": "flushed before every call (256 MiB write, outside the events)"},
        "per_mask": per_mask, "quantize_qkv_ms": quant_ms,
        "roofline": {"bound": "tensor", "achieved": per_mask[dom]["tflops"], "peak": peak8, "unit": "TFLOP/s",
                     "frac": per_mask[dom]["frac_of_fp8_peak"],
                     "peak_kind": f"{peak_src} bf16 dense burst x 2 (nominal FP8 / bf16 ratio)",
                     "kernel": "fa_fwd_kernel<128, *, e4m3>", "mask": dom, "traffic": None},
        "gpu_launches": args.steps * len(per_mask),
        "clocks": clocks}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-heads", type=int, default=None,
                    help="heads of the oracle's CPU sample (default: about 100 GFLOP of work)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip timing the other configurations after the headline")
    ap.add_argument("--decode", action="store_true",
                    help="the few-query-rows shapes through fa_fwd_rect (HBM-bound), "
                         "instead of the headline step")
    ap.add_argument("--fp8", action="store_true",
                    help="the forward on FP8 (e4m3) operands through fa_fwd_fp8 instead of the bf16 step")
    ap.add_argument("--backward", action="store_true",
                    help="dQ, dK, dV of the workload through fa_bwd instead of the forward step")
    ap.add_argument("--quick", action="store_true",
                    help="only the timed kernel steps (for profiler runs): no clock sampling, "
                         "no end-to-end leg, no CPU baseline, no one-second warm-up floor")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.decode:
        run_decode(args)
    elif args.backward:
        run_backward(args)
    elif args.fp8:
        run_fp8(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
