#!/usr/bin/env python
"""Benchmark of the FlashAttention-2 backward on GB300.

One step = one backward pass over the workload's batch: fa_bwd_preprocess
(D = rowsum(O * dO), zero the dQ accumulator), fa_bwd (the tcgen05 kernel),
fa_convert_dq.  O and L come from fa_fwd once, before timing (the forward is
the backward's producer and is timed separately under "fa_fwd").

Throughput counts the five backward GEMMs, 10 B H N^2 d FLOPs, halved under
the causal mask.  Default workload: B=1, H=32, N=8192, d=128, causal, bf16.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the float64 CPU oracle arm

Prints one JSON line (rank 0).  Under torchrun every rank runs an
independent replica (the problem shards over (b, h) with no exchange), times
are the max over ranks and `value` aggregates all ranks (weak scaling).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FA2 backward TFLOPS (10·BHN²d, ½ if causal) and % of GB300 bf16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CSRC = os.path.join(ROOT, "flashattention_backward_gb300", "csrc")
# per fa_bwd kernel: (kernel name, source file, committed ncu traffic record)
BWD_KERNELS = {
    "sm103": ("bwd_sm103_kernel", os.path.join(CSRC, "fa_bwd_sm103.cu"),
              os.path.join(ROOT, "profiles", "fa_bwd_sm103_traffic.txt")),
    "d256": ("bwd_d256_kernel", os.path.join(CSRC, "fa_bwd_d256_sm103.cu"),
             os.path.join(ROOT, "profiles", "fa_bwd_d256_sm103_traffic.txt")),
}


def bwd_kernel(w):
    """The fa_bwd kernel that serves workload w (bf16)."""
    return BWD_KERNELS["d256" if w.d == 256 else "sm103"]


# ----------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_sha(src: str) -> str:
    with open(src, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def recorded_traffic(w):
    """DRAM bytes per fa_bwd launch from the committed ncu summary, or None
    when the kernel source changed since the capture."""
    _, src, record = bwd_kernel(w)
    try:
        with open(record) as f:
            kv = dict(line.split(None, 1) for line in f.read().splitlines() if line and not line.startswith("#"))
    except (OSError, ValueError):
        return None
    if kv.get("kernel_sha256", "").strip() != kernel_sha(src):
        return None
    val = kv.get(f"bytes_per_launch_{w.name}")
    return float(val) if val else None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.lines: list[str] = []
        self.proc = None
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "20",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5.0 and self.proc.poll() is None:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def mark(self):
        return len(self.lines)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, first: int):
        rows = [l.split(", ") for l in self.lines[first:]]
        rows = [r for r in rows if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip().lower() == "active"})
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


def aggregate_max(value: float, dist_mod=None) -> float:
    """Max of `value` over all ranks (identity without a process group)."""
    if dist_mod is None or not dist_mod.is_available() or not dist_mod.is_initialized():
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if dist_mod.get_backend() == "nccl" else "cpu")
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank_step: float, world: int, steps: int, max_ms_total: float) -> float:
    """Units all ranks processed over the slowest rank's time."""
    return flops_per_rank_step * world * steps / (max_ms_total * 1e-3) / 1e12


# ----------------------------------------------------------------- oracle arm
def oracle_sample_tflops(w, heads: int, repeat: int = 1):
    """Time the float64 oracle on `heads` heads of the workload (host cores).
    Returns (TFLOPS in the metric's accounting, seconds, sample description)."""
    from fa_inputs import make_inputs, to_f64
    from oracle import attention_backward

    small = w.with_(B=1, H=heads)
    q, k, v, g = make_inputs(small)
    arrays = [to_f64(t) for t in (q, k, v, g)]
    t0 = time.perf_counter()
    for _ in range(repeat):
        attention_backward(*arrays, w.scale, w.causal)
    dt = (time.perf_counter() - t0) / repeat
    return small.counted_flops / dt / 1e12, dt, f"{heads} head(s) of B={w.B} H={w.H} N={w.N} d={w.d}" \
        f"{' causal' if w.causal else ''}, full rows, float64 NumPy/BLAS"


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def run_reference(args, w, rank: int) -> int:
    if rank != 0:
        return 0
    for _ in range(args.warmup):
        oracle_sample_tflops(w, args.ref_heads)
    times = []
    for _ in range(args.steps):
        _, dt, sample = oracle_sample_tflops(w, args.ref_heads)
        times.append(dt)
    small = w.with_(B=1, H=args.ref_heads)
    total = sum(times)
    value = small.counted_flops * args.steps / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args.gpus),
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": host_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, n_gpus):
    return {"workload": f"{w.name}: B={w.B} H={w.H} N={w.N} d={w.d} {'causal' if w.causal else 'non-causal'} "
                        f"{w.dtype}", "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
            "parallelism": f"replicas x{n_gpus}",
            "l2": "inputs larger than L2 (Q, K, V, dO, O, dQ/dK/dV, fp32 dQ accumulator: >0.5 GB per step)"}


# ----------------------------------------------------------------- GPU arm
def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="causal")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-heads", type=int, default=1, help="heads per oracle step (reference arm)")
    ap.add_argument("--cpu-heads", type=int, default=2, help="heads in the cpu_baseline sample")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--e2e-group", type=int, default=0, help="heads per group in the end-to-end leg (0: auto)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--deterministic", action="store_true", help="bitwise reproducible dQ (per-key-block slices)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)

    from fa_inputs import workload

    w = workload(args.workload)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return run_reference(args, w, rank)

    import torch
    import torch.distributed as dist

    import flashattention_backward_gb300 as fa
    from fa_inputs import make_inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    fa.load_library()

    # inputs: seeded on the host, copied once; O and L from fa_fwd
    q_h, k_h, v_h, g_h = make_inputs(w)
    q, k, v, g = (t.to(dev) for t in (q_h, k_h, v_h, g_h))
    stream = torch.cuda.current_stream()
    p = fa.problem_for(q, w.scale, w.causal, args.deterministic)
    o = torch.empty_like(q)
    L = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=dev)
    D = torch.empty_like(L)
    acc = torch.empty(fa.fa_dq_accum_elems(p), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)

    # companion forward, timed on its own
    fwd_ms = []
    for it in range(4):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fa.fa_fwd(p, q, k, v, o, L, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        if it:
            fwd_ms.append(e0.elapsed_time(e1))

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fa.fa_bwd_preprocess(p, o, g, D, acc, stream)
        if ev is not None:
            ev[1].record(stream)
        fa.fa_bwd(p, q, k, v, g, L, D, acc, dk, dv, stream)
        if ev is not None:
            ev[2].record(stream)
        fa.fa_convert_dq(p, acc, dq, stream)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if fa.get_device_status() != 0:
        raise RuntimeError("device status set during warm-up")

    sampler = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    sampler.start()
    mark = sampler.mark()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    time.sleep(0.15)
    sampler.stop()
    clocks = sampler.summary(mark)
    total_ms = aggregate_max(t_start.elapsed_time(t_end), dist if world > 1 else None)
    status = fa.get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    pre_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    cvt_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)

    # the same step as one launch (fa_backward_fused), timed after the timed
    # region for comparison; the three launches above are faster on this GPU
    fused = None
    sync_n = fa.fa_backward_fused_sync_elems(p)
    if sync_n > 0:
        sync = torch.empty(sync_n, dtype=torch.int32, device=dev)
        for _ in range(3):
            fa.fa_backward_fused(p, q, k, v, o, g, L, D, acc, sync, dq, dk, dv, stream)
        n_fused = max(5, args.steps // 10)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n_fused):
            fa.fa_backward_fused(p, q, k, v, o, g, L, D, acc, sync, dq, dk, dv, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        if fa.get_device_status() != 0:
            raise RuntimeError("device status set by the single-launch backward")
        fused_ms = e0.elapsed_time(e1) / n_fused
        fused = {"ms": fused_ms, "TFLOPS": w.counted_flops / (fused_ms * 1e-3) / 1e12,
                 "note": "preprocess + bwd + convert in one launch; not the step timed above"}

    # end to end through the public API with host buffers: fa_backward_host
    # streams groups of heads through a device workspace, copies overlapped
    # with compute; every input crosses host->device and every gradient
    # device->host inside the timed region.
    e2e = None
    if args.e2e_steps > 0:
        pin = lambda t: t.contiguous().pin_memory()
        hq, hk, hv, hg = (pin(t) for t in (q_h, k_h, v_h, g_h))
        ho, hL = pin(o.cpu()), pin(L.cpu())
        houts = tuple(torch.empty_like(hq).pin_memory() for _ in range(3))
        ws = torch.empty(fa.fa_backward_host_workspace_bytes(p, args.e2e_group), dtype=torch.uint8, device=dev)
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, ho, hg, hL))
        d2h = sum(t.numel() * t.element_size() for t in houts)

        def e2e_step():
            fa.attention_backward_host(hq, hk, hv, ho, hg, hL, w.scale, w.causal, args.e2e_group, workspace=ws,
                                       out=houts, stream=stream, deterministic=args.deterministic)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = aggregate_max(e0.elapsed_time(e1), dist if world > 1 else None)
        if fa.get_device_status() != 0:
            raise RuntimeError("device status set during the end-to-end leg")
        e2e = {"value": whole_job_tflops(w.counted_flops, world, args.e2e_steps, e2e_ms), "unit": "TFLOPS",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / args.e2e_steps,
               "api": "fa_backward_host (pinned host buffers, %s heads per group)" % (args.e2e_group or "auto")}

    peaks, peak_src = load_peaks()
    flops = w.counted_flops
    value = whole_job_tflops(flops, world, args.steps, total_ms)
    bwd_tflops = flops / (bwd_ms * 1e-3) / 1e12
    bhnd = w.B * w.H * w.N * w.d
    slice_bytes = fa.fa_dq_accum_elems(fa.problem_for(q, w.scale, w.causal)) * 4  # one accumulator slice
    n_slices = fa.fa_dq_accum_elems(p) * 4 // slice_bytes
    pre_bytes = 2 * bhnd * 2 + w.B * w.H * w.N * 4 + (0 if args.deterministic else slice_bytes)
    # convert reads every slice that holds a contribution (half of them under the causal mask)
    live = n_slices if not w.causal else (n_slices + 1) / 2
    cvt_bytes = slice_bytes * live + bhnd * 2
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(workload_config(w, world), dq_mode="deterministic" if args.deterministic else "atomic"),
        "e2e": e2e,
        "gpu_launches": 3 * args.steps,
        "roofline": {"kernel": f"fa_bwd ({bwd_kernel(w)[0]})", "bound": "tensor", "achieved": bwd_tflops,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": bwd_tflops / peaks["bf16_tflops"],
                     "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json)" if peak_src == "measured"
                     else "fallback 1.9 PFLOP/s bf16 burst",
                     "frac_of_sustained": bwd_tflops / peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]),
                     "traffic": recorded_traffic(w), "ms": bwd_ms},
        "kernels": {
            "fa_bwd_preprocess": {"ms": pre_ms, "GB/s": pre_bytes / (pre_ms * 1e-3) / 1e9,
                                  "frac_hbm": pre_bytes / (pre_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]},
            "fa_bwd": {"ms": bwd_ms, "TFLOPS": bwd_tflops},
            "fa_convert_dq": {"ms": cvt_ms, "GB/s": cvt_bytes / (cvt_ms * 1e-3) / 1e9,
                              "frac_hbm": cvt_bytes / (cvt_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]},
            "fa_backward_fused": fused,
            "fa_fwd": {"ms": statistics.mean(fwd_ms),
                       "TFLOPS": 0.4 * flops / (statistics.mean(fwd_ms) * 1e-3) / 1e12,
                       "note": "companion forward, not part of the step; 4 B H N^2 d (half if causal)"},
        },
        "clocks": clocks,
        # ch.16 §16.7's cost model: the backward's 5 GEMMs against the
        # forward's 2 are 2.5x the FLOPs (the page quotes ~2.9x in time)
        "bwd_fwd_time_ratio": {"value": bwd_ms / statistics.mean(fwd_ms), "flop_ratio_model": 2.5,
                               "note": "fa_bwd time / fa_fwd time on this workload"},
    }
    if rank == 0 and not args.no_cpu_baseline:
        tf, dt, sample = oracle_sample_tflops(w, args.cpu_heads)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOPS", "cores": host_cores(), "kind": "oracle",
                                "sample": sample, "seconds": dt}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
