#!/usr/bin/env python3
"""Benchmark: p=8 bf16 AllReduce throughput on one GPU, against HBM peak.

One step = one ccl_allreduce call through the C ABI (argument checks,
schedule selection and table build on the host, one fused kernel on the
device) over p=8 rank buffers of 2^27 bf16 elements (256 MiB per rank,
2 GiB in, 2 GiB out).  Throughput counts the algorithmic minimum bytes of an
AllReduce in which every rank receives the result: p*n*s read + p*n*s written.

Printed JSON line (rank 0): value = whole-job GB/s over K timed steps (CUDA
events on the launching stream, barrier + synchronize on both sides, max over
ranks), plus roofline (the fused kernel against the measured HBM copy peak),
e2e (same metric with pinned host buffers, every byte crossing the host link
inside the timed region: the kernel on the host buffers, or staged copies),
the CPU oracle baseline, clocks sampled during the timed region, and the
message-size sweep (1 KiB .. 256 MiB per rank, ring and all-pairs).

Multi-GPU: one process per GPU (torchrun), each an independent replica of the
workload (the collective's p ranks are buffers in one GPU's memory; there is
no exchange between GPUs).  value = all replicas' bytes / max time.

--impl reference times the CPU oracle on the host cores instead (rank 0
only), each step a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "p=8 bf16 AllReduce GB/s and % of GB300 HBM peak vs message size (1 GPU)"
P = 8
N = 1 << 27            # bf16 elements per rank: 256 MiB
S = 2
WORKLOAD = "p=8 bf16 AllReduce sum, 256 MiB per rank (n=2^27), N(0,1), schedule auto (ring at this size)"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["reducescatter_reduction_gb300/csrc/reduce.cuh",
                  "reducescatter_reduction_gb300/csrc/device.cuh",
                  "reducescatter_reduction_gb300/csrc/reduce_bf16.cu"]
# ncu's DRAM bytes per launch of the headline kernel, with the hash of the
# kernel source it was taken on (written beside the ncu summary it comes from)
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "roofline_traffic.json")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--schedule", default="auto", choices=["auto", "ring", "allpairs"])
    ap.add_argument("--variant", default="ldst", choices=["ldst", "tma", "tma_bulkred"])
    ap.add_argument("--sm-budget", type=int, default=0)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--no-budgets", action="store_true")
    ap.add_argument("--rmsnorm-tokens", type=int, default=0,
                    help="profiling mode: only the fused AllReduce + residual + RMSNorm, p=8 bf16, "
                         "[tokens, 8192], warmup + steps calls")
    ap.add_argument("--ranks", type=int, default=0,
                    help="profiling: one bf16 AllReduce of this many ranks of --n elements, with --variant and "
                         "--sm-budget, timed alone")
    ap.add_argument("--moe-rows", type=int, default=0,
                    help="profiling mode: only the p=16 bf16 [rows, 7168] ring AllReduce with --variant and "
                         "--sm-budget, warmup + steps calls")
    ap.add_argument("--host-buffers", action="store_true",
                    help="profiling mode: only the zero-copy AllReduce, p=8 bf16 rank buffers of --n elements in "
                         "pinned host memory (inputs and outputs), --sm-budget, warmup + steps calls")
    ap.add_argument("--collective", choices=["rs", "ag"], default=None,
                    help="profiling mode: only the p=8 bf16 ReduceScatter (rank r's output = chunk r of a second "
                         "buffer, as in the rs_ag rows) or the in-place AllGather, --n elements per rank, "
                         "warmup + steps calls")
    ap.add_argument("--calibrate", action="store_true",
                    help="fit t = alpha + bytes/B per variant and SM budget (p=8 bf16) and print the table")
    ap.add_argument("--n", type=int, default=N,
                    help="bf16 elements per rank (default 2^27; smaller only for profiling runs)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# multi-process plumbing (timing only: no data moves between GPUs)
# ---------------------------------------------------------------------------

class Dist:
    def __init__(self):
        self.rank = int(os.environ.get("RANK", "0"))
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = False

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = True

    def barrier(self):
        if self.pg:
            import torch.distributed as dist
            dist.barrier()

    def reduce(self, value: float, op: str) -> float:
        """max or sum of a float over ranks (every rank gets the result)."""
        if not self.pg:
            return value
        import torch
        import torch.distributed as dist
        dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
        t = torch.tensor([value], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            import torch.distributed as dist
            dist.destroy_process_group()


def aggregate(dist: Dist, local_ms: float, local_bytes: float):
    """Whole-job throughput: every replica's bytes over the slowest replica's time."""
    t = dist.reduce(local_ms, "max")
    b = dist.reduce(local_bytes, "sum")
    return t, b, (b / (t * 1e-3) / 1e9 if t > 0 else 0.0)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
            if self.gpu_id:
                cmd.insert(1, f"--id={self.gpu_id}")
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.seek(0)
        rows = [line.strip().split(",") for line in self.file.read().splitlines() if line.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for row in rows:
            row = [c.strip() for c in row]
            if len(row) < 8:
                continue
            try:
                sm.append(float(row[0]))
                mx.append(float(row[1]))
            except ValueError:
                continue
            for name, flag in zip(names, row[4:8]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def gpu_uuid(torch, dev) -> str | None:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ---------------------------------------------------------------------------
# peaks and the committed ncu summary
# ---------------------------------------------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs: bf16 copy, read+write bytes)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 measurement)"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """(DRAM bytes per launch, where they come from): ncu's dram__bytes_read.sum
    + dram__bytes_write.sum per launch of the headline kernel, as recorded in
    TRAFFIC_FILE -- only if that capture was taken on the current kernel source
    (else None, and the reason)."""
    rel = os.path.relpath(TRAFFIC_FILE, ROOT)
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
        traffic = float(rec["dram_bytes_per_launch"])
        src = str(rec["kernel_source_sha256_16"])
    except (OSError, KeyError, ValueError, TypeError):
        return None, f"no ncu record ({rel} missing or unreadable)"
    cur = kernel_source_hash()
    if src != cur:
        return None, f"{rel} was taken on kernel source {src}; the current source is {cur}: not reported"
    how = rec.get("how", "")
    return traffic, f"ncu dram__bytes_read.sum + dram__bytes_write.sum, {rel} (kernel source {src}); {how}".rstrip("; ")


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------

def run_ours(args, dist: Dist):
    import numpy as np
    import torch

    import __graft_entry__
    import reducescatter_reduction_gb300 as ccl

    __graft_entry__.build()
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    dist.init("nccl")
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or 0

    # inputs: seeded N(0,1) bf16 on the device (2 GiB), outputs beside them
    gen = torch.Generator(device=dev)
    gen.manual_seed(2 + 1000 * dist.rank)
    n = args.n
    ins = [torch.randn(n, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
           for _ in range(P)]
    outs = [torch.empty_like(t) for t in ins]
    comm = ccl.ccl_comm_create(P, [t.data_ptr() for t in ins])
    ccl.ccl_comm_set_outputs(comm, [t.data_ptr() for t in outs])
    ccl.ccl_set_launch(comm, args.sm_budget, args.variant, 0)
    alg_bytes = 2.0 * P * n * S

    for _ in range(args.warmup):
        ccl.ccl_allreduce(comm, "sum", "bf16", n, args.schedule, sptr)
    torch.cuda.synchronize()
    launch_desc = ccl.ccl_comm_last_launch(comm)

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_uuid(torch, dev))
    sampler.start()
    time.sleep(0.3)                       # let the sampler take its first reading
    dist.barrier()
    torch.cuda.synchronize()
    launches0 = ccl.ccl_comm_launch_count(comm)
    e0.record(stream)
    for _ in range(args.steps):
        ccl.ccl_allreduce(comm, "sum", "bf16", n, args.schedule, sptr)
    e1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    clocks = sampler.stop()
    launches = ccl.ccl_comm_launch_count(comm) - launches0
    local_ms = e0.elapsed_time(e1)
    ccl.ccl_comm_check(comm)

    t_ms, job_bytes, job_gbs = aggregate(dist, local_ms, alg_bytes * args.steps)
    ms_per_step = t_ms / args.steps
    per_launch_ms = local_ms / max(1, launches)
    achieved = alg_bytes / (per_launch_ms * 1e-3) / 1e9
    peak, peak_src = hbm_peak()
    traffic, traffic_src = profiled_traffic() if n == N else (None, "profiling size: no record")

    result = {
        "metric": METRIC,
        "value": round(job_gbs, 2),
        "unit": "GB/s",
        "n_gpus": dist.world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "frac_of_hbm_peak": round(job_gbs / dist.world / peak, 4),
        "config": {
            "workload": WORKLOAD if n == N else f"p=8 bf16 AllReduce sum, n={n} per rank (profiling size)",
            "p": P, "n_per_rank": n, "element": "bf16 (fp32 accumulation)",
            "bytes_per_rank": n * S,
            "algorithmic_bytes_per_step": int(alg_bytes),
            "schedule": args.schedule, "variant": args.variant, "sm_budget": args.sm_budget,
            "launch": launch_desc,
            "l2": f"inputs ({P * n * S >> 20} MiB) larger than L2 ({l2 >> 20} MiB): no flush",
            "parallelism": f"replicas x{dist.world} (no inter-GPU exchange)",
        },
        "roofline": {
            "bound": "hbm",
            "achieved": round(achieved, 2),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "traffic_source": traffic_src,
            "algorithmic_bytes_per_launch": int(alg_bytes),
            "peak_source": peak_src,
            "kernel": launch_desc.split()[0] if launch_desc else None,
        },
        "gpu_launches": int(launches),
        "clocks": clocks,
    }

    if not args.no_e2e:
        result["e2e"] = run_e2e(args, dist, comm, ins, outs, sptr, stream, alg_bytes, n)
    if not args.no_sweep:
        result["rs_ag"] = run_rs_ag(args, ins, outs, sptr, stream, peak, n)
        result["variants"] = run_variants(comm, sptr, stream, peak, n, args)

    ccl.ccl_comm_destroy(comm)
    if not args.no_sweep:
        del outs
        torch.cuda.empty_cache()
        result["sweep"] = run_sweep(dist, dev, sptr, stream, peak, l2, ins)
        result["launch_floor"] = launch_floor()
    if not args.no_sweep:
        result["op_coverage"] = run_ops(dev, sptr, stream, peak)
    if not args.no_budgets:
        torch.cuda.empty_cache()
        result["sm_budgets"] = run_budgets(dev, sptr, stream, peak)
        result["sm_budgets_p8"] = run_budgets(dev, sptr, stream, peak, p=8, n=1 << 25, variants=("ldst", "tma", "auto"),
                                              budgets=(8, 16, 32, 76, 0))
        result["fused_rmsnorm"] = run_rmsnorm(dev, peak)
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline_from(ins)
    del ins
    dist.close()
    return result


def run_e2e(args, dist, comm, ins, outs, sptr, stream, alg_bytes, n):
    """Same metric with host buffers: every step copies its p inputs from
    pinned host memory, runs the AllReduce through the C ABI, and copies its
    p results back to pinned host memory, all inside the timed region.

    Three ways of running a stream of such steps are timed: double-buffered
    (two device buffer sets; host->device copies on one stream, AllReduce on
    another, device->host on a third, ordered by events), so that step i+1's
    input copy overlaps step i's AllReduce and output copy; serial, one step
    at a time on one stream; and zero-copy, where the communicator's rank
    buffers are the pinned host buffers themselves and the AllReduce kernel
    reads the inputs and writes the results over the host link (NVLink-C2C on
    Grace-Blackwell), one kernel per step.  Every mode moves p*n*s bytes each
    way per step.  value is the fastest; the others are kept beside it."""
    import torch
    import reducescatter_reduction_gb300 as ccl

    h_in = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True) for _ in range(P)]
    for h, d in zip(h_in, ins):
        h.copy_(d)
    h_out = [[torch.empty(n, dtype=torch.bfloat16, pin_memory=True) for _ in range(P)] for _ in range(2)]
    ins2 = [torch.empty_like(t) for t in ins]
    outs2 = [torch.empty_like(t) for t in outs]
    comm2 = ccl.ccl_comm_create(P, [t.data_ptr() for t in ins2])
    ccl.ccl_comm_set_outputs(comm2, [t.data_ptr() for t in outs2])
    sets = [(comm, ins, outs), (comm2, ins2, outs2)]

    def timed(fn, steps):
        for i in range(2):
            fn(i)
        torch.cuda.synchronize()
        dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        start_stream = torch.cuda.current_stream()
        for i in range(steps):
            fn(i)
        end_stream = last_stream[0] or start_stream
        e1.record(end_stream)
        torch.cuda.synchronize()
        dist.barrier()
        return e0.elapsed_time(e1)

    last_stream = [None]

    def serial_step(i):
        for h, d in zip(h_in, ins):
            d.copy_(h, non_blocking=True)
        ccl.ccl_allreduce(comm, "sum", "bf16", n, args.schedule, sptr)
        for h, d in zip(h_out[0], outs):
            h.copy_(d, non_blocking=True)

    s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev_h2d = [torch.cuda.Event() for _ in range(2)]
    ev_ar = [torch.cuda.Event() for _ in range(2)]
    ev_d2h = [torch.cuda.Event() for _ in range(2)]
    issued = [False, False]

    def piped_step(i):
        k = i % 2
        h, d_in, d_out = sets[k]
        s_h2d.wait_stream(stream) if i == 0 else None
        if issued[k]:
            s_h2d.wait_event(ev_ar[k])            # the AllReduce two steps back read d_in
        with torch.cuda.stream(s_h2d):
            for hh, dd in zip(h_in, d_in):
                dd.copy_(hh, non_blocking=True)
        ev_h2d[k].record(s_h2d)
        stream.wait_event(ev_h2d[k])
        if issued[k]:
            stream.wait_event(ev_d2h[k])          # the output copy two steps back read d_out
        ccl.ccl_allreduce(h, "sum", "bf16", n, args.schedule, sptr)
        ev_ar[k].record(stream)
        s_d2h.wait_event(ev_ar[k])
        with torch.cuda.stream(s_d2h):
            for hh, dd in zip(h_out[k], d_out):
                hh.copy_(dd, non_blocking=True)
        ev_d2h[k].record(s_d2h)
        issued[k] = True
        last_stream[0] = s_d2h

    zc = ccl.ccl_comm_create(P, [t.data_ptr() for t in h_in])
    ccl.ccl_comm_set_outputs(zc, [t.data_ptr() for t in h_out[0]])

    def zero_copy_step(i):
        ccl.ccl_allreduce(zc, "sum", "bf16", n, args.schedule, sptr)

    t_serial = timed(serial_step, args.e2e_steps)
    last_stream[0] = None
    t_piped = timed(piped_step, args.e2e_steps)
    last_stream[0] = None
    t_zc = timed(zero_copy_step, args.e2e_steps)
    ccl.ccl_comm_check(zc)
    ccl.ccl_comm_destroy(zc)
    ccl.ccl_comm_destroy(comm2)
    modes = []
    for t, name in ((t_zc, "zero-copy: the AllReduce reads the pinned host inputs and writes the pinned host "
                           "outputs over the host link, one kernel per step"),
                    (t_piped, "double-buffered: H2D, AllReduce and D2H on three streams"),
                    (t_serial, "serial: H2D, AllReduce, D2H on one stream")):
        t_ms, _, gbs = aggregate(dist, t, alg_bytes * args.e2e_steps)
        modes.append({"value": round(gbs, 2), "ms_per_step": round(t_ms / args.e2e_steps, 4), "mode": name})
    # All run the same AllReduce on the same host buffers; which is fastest
    # depends on how the machine's host link takes both directions at once,
    # so the line reports the fastest and keeps the others beside it.
    modes.sort(key=lambda m: -m["value"])
    best = modes[0]
    return {"value": best["value"], "unit": "GB/s", "h2d_bytes_per_step": P * n * S,
            "d2h_bytes_per_step": P * n * S, "steps": args.e2e_steps,
            "ms_per_step": best["ms_per_step"], "mode": best["mode"], "other_modes": modes[1:]}


def run_variants(comm, sptr, stream, peak, n, args):
    """The benchmark AllReduce through each kernel variant and comparison
    executor (all SMs).  GBps counts the AllReduce's algorithmic bytes 2*p*n*s
    for all of them; bytes_moved is what each one actually moves: 2(p+1)ns for
    bulk-reduce (ReduceScatter then AllGather), 5(p-1)ns for the stepwise
    ring, (p^2+p)ns for one-phase all-pairs."""
    import torch
    import reducescatter_reduction_gb300 as ccl

    rows = {}
    moved = {"ldst": 2 * P, "tma": 2 * P, "tma_bulkred": 2 * (P + 1), "ring_stepwise": 5 * (P - 1),
             "one_phase": P * P + P}                       # bytes moved per n*s
    for variant in ("ldst", "tma", "tma_bulkred", "ring_stepwise", "one_phase"):
        ccl.ccl_set_launch(comm, 0, variant, 0)
        for _ in range(3):
            ccl.ccl_allreduce(comm, "sum", "bf16", n, "ring", sptr)
        torch.cuda.synchronize()
        iters = 50
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(iters):
            ccl.ccl_allreduce(comm, "sum", "bf16", n, "ring", sptr)
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / iters
        gbs = 2 * P * n * S / (us * 1e-6) / 1e9
        moved_gbs = moved[variant] * n * S / (us * 1e-6) / 1e9
        rows[variant] = {"us": round(us, 1), "GBps": round(gbs, 1), "frac_of_hbm_peak": round(gbs / peak, 4),
                         "bytes_moved": moved[variant] * n * S, "moved_GBps": round(moved_gbs, 1),
                         "launch": ccl.ccl_comm_last_launch(comm)}
    ccl.ccl_set_launch(comm, args.sm_budget, args.variant, 0)
    ccl.ccl_comm_check(comm)
    return rows


def run_ops(dev, sptr, stream, peak):
    """The op-coverage workload: p=8 rank buffers of 64 Mi elements, ring,
    every op in int32 (uniform in [-1000, 1000]; prod over {-1, 1, 2}), fp32
    and fp16 (N(0,1)), drawn on the device.  GB/s over 2*p*n*s per call."""
    import torch
    import reducescatter_reduction_gb300 as ccl
    from reducescatter_reduction_gb300 import inputs

    p, n = 8, inputs.COVERAGE_N
    gen = torch.Generator(device=dev)
    gen.manual_seed(4)
    rows = {}
    for dtype, tdt, s in (("i32", torch.int32, 4), ("f32", torch.float32, 4), ("f16", torch.float16, 2)):
        for op in ("sum", "prod", "min", "max", "avg"):
            if dtype == "i32":
                if op == "prod":
                    vals = torch.tensor([-1, 1, 2], device=dev, dtype=torch.int32)
                    ins = [vals[torch.randint(0, 3, (n,), generator=gen, device=dev)] for _ in range(p)]
                else:
                    ins = [torch.randint(-1000, 1001, (n,), generator=gen, device=dev, dtype=torch.int32)
                           for _ in range(p)]
            else:
                ins = [torch.randn(n, generator=gen, device=dev).to(tdt) for _ in range(p)]
            outs = [torch.empty_like(t) for t in ins]
            h = ccl.ccl_comm_create(p, [t.data_ptr() for t in ins])
            ccl.ccl_comm_set_outputs(h, [t.data_ptr() for t in outs])
            for _ in range(3):
                ccl.ccl_allreduce(h, op, dtype, n, "ring", sptr)
            torch.cuda.synchronize()
            iters = 20
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(iters):
                ccl.ccl_allreduce(h, op, dtype, n, "ring", sptr)
            e1.record(stream)
            torch.cuda.synchronize()
            ccl.ccl_comm_check(h)
            us = e0.elapsed_time(e1) * 1e3 / iters
            gbs = 2 * p * n * s / (us * 1e-6) / 1e9
            rows[f"{dtype}_{op}"] = {"us": round(us, 1), "GBps": round(gbs, 1), "frac_of_hbm_peak": round(gbs / peak, 4)}
            ccl.ccl_comm_destroy(h)
            del ins, outs
    torch.cuda.empty_cache()
    return rows


def run_rs_ag(args, ins, outs, sptr, stream, peak, n):
    """The same buffers as separate ReduceScatter (out[r] = chunk r) and
    AllGather (in place): GB/s over each one's algorithmic bytes."""
    import torch
    import reducescatter_reduction_gb300 as ccl

    chunk = n // P
    rows = {}
    rs = ccl.ccl_comm_create(P, [t.data_ptr() for t in ins])
    ccl.ccl_comm_set_outputs(rs, [outs[r].data_ptr() + r * chunk * S for r in range(P)])
    ag = ccl.ccl_comm_create(P, [t.data_ptr() for t in outs])
    cases = (("reduce_scatter", lambda: ccl.ccl_reduce_scatter(rs, "sum", "bf16", n, "ring", sptr),
              (P + 1) * n * S, rs),
             ("all_gather_in_place", lambda: ccl.ccl_all_gather(ag, "bf16", n, sptr), P * n * S, ag))
    for name, call, nbytes, h in cases:
        for _ in range(5):
            call()
        torch.cuda.synchronize()
        iters = 200
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(iters):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / iters
        gbs = nbytes / (us * 1e-6) / 1e9
        rows[name] = {"us": round(us, 2), "GBps": round(gbs, 1), "frac_of_hbm_peak": round(gbs / peak, 4),
                      "algorithmic_bytes": nbytes, "launch": ccl.ccl_comm_last_launch(h)}
    ccl.ccl_comm_destroy(rs)
    ccl.ccl_comm_destroy(ag)
    return rows


def run_collective_only(args, dist):
    """Profiling mode: the ReduceScatter or the in-place AllGather of the
    rs_ag rows alone (same buffers, launch shape and bytes), so that ncu can
    capture that kernel on a small case."""
    import torch
    import __graft_entry__
    import reducescatter_reduction_gb300 as ccl
    __graft_entry__.build()
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    n = args.n - args.n % P
    chunk = n // P
    ins = [torch.randn(n, device=dev, dtype=torch.float32).to(torch.bfloat16) for _ in range(P)]
    outs = [torch.empty_like(t) for t in ins]
    if args.collective == "rs":
        h = ccl.ccl_comm_create(P, [t.data_ptr() for t in ins])
        ccl.ccl_comm_set_outputs(h, [outs[r].data_ptr() + r * chunk * S for r in range(P)])
        call = lambda s: ccl.ccl_reduce_scatter(h, "sum", "bf16", n, "ring", s)
        nbytes = (P + 1) * n * S
    else:
        h = ccl.ccl_comm_create(P, [t.data_ptr() for t in outs])
        call = lambda s: ccl.ccl_all_gather(h, "bf16", n, s)
        nbytes = P * n * S
    s = torch.cuda.current_stream()
    for _ in range(args.warmup):
        call(s.cuda_stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(args.steps):
        call(s.cuda_stream)
    e1.record(s)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / max(1, args.steps)
    ccl.ccl_comm_check(h)
    print(json.dumps({"mode": args.collective, "n_per_rank": n, "us_per_call": round(us, 2),
                      "GBps": round(nbytes / (us * 1e-6) / 1e9, 1), "algorithmic_bytes": nbytes,
                      "launch": ccl.ccl_comm_last_launch(h)}), flush=True)
    ccl.ccl_comm_destroy(h)
    return 0


def calibrate(dev):
    """Per-call device time of the p=8 bf16 AllReduce for the ld/st and TMA
    variants at several SM budgets over 16 KiB .. 256 MiB per rank (CUDA-graph
    replay below 8 MiB, events above), and a least-squares fit of
    t = alpha + bytes / B (bytes = 2 p n s) on relative error."""
    import numpy as np
    import torch
    import reducescatter_reduction_gb300 as ccl

    sizes = [1 << k for k in range(13, 28, 2)]              # bf16 elements per rank
    big = [(torch.randn(sizes[-1], device=dev)).to(torch.bfloat16) for _ in range(P)]
    outs = [torch.empty_like(t) for t in big]
    table = []
    for variant in ("ldst", "tma"):
        for budget in (0, 8, 16, 32, 76):
            ts = []
            for n in sizes:
                h = ccl.ccl_comm_create(P, [t.data_ptr() for t in big])
                ccl.ccl_comm_set_outputs(h, [t.data_ptr() for t in outs])
                ccl.ccl_set_launch(h, budget, variant, 0)
                s = torch.cuda.current_stream()
                ccl.ccl_allreduce(h, "sum", "bf16", n, "ring", s.cuda_stream)
                torch.cuda.synchronize()
                calls = 100 if n * S * P < (64 << 20) else 5
                side = torch.cuda.Stream()
                side.wait_stream(s)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.stream(side):
                    with torch.cuda.graph(g, stream=side):
                        cs = torch.cuda.current_stream().cuda_stream
                        for _ in range(calls):
                            ccl.ccl_allreduce(h, "sum", "bf16", n, "ring", cs)
                s.wait_stream(side)
                g.replay()
                torch.cuda.synchronize()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(3):
                    g.replay()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e-3 / (3 * calls))
                ccl.ccl_comm_destroy(h)
            x = np.array([2.0 * P * n * S for n in sizes])
            t = np.array(ts)
            # minimise sum ((alpha + x/B - t) / t)^2: linear in (alpha, 1/B)
            A = np.stack([1.0 / t, x / t], axis=1)
            coef, *_ = np.linalg.lstsq(A, np.ones_like(t), rcond=None)
            alpha, inv_b = float(coef[0]), float(coef[1])
            pred = alpha + x * inv_b
            table.append({"variant": variant, "sm_budget": budget, "alpha_us": round(alpha * 1e6, 3),
                          "B_GBps": round(1.0 / inv_b / 1e9, 1),
                          "max_rel_residual": round(float(np.max(np.abs(pred - t) / t)), 3),
                          "points_us": [round(v * 1e6, 2) for v in ts]})
    return {"sizes_bytes_per_rank": [n * S for n in sizes], "fits": table}


def run_rmsnorm(dev, peak):
    """AllReduce fused with the residual merge and RMSNorm at TP=8 (p=8 bf16,
    hidden 8192) at 1, 32, 256 and 4096 tokens, against the
    AllReduce alone and against the AllReduce followed by the same epilogue in
    torch on one rank's copy (a lower bound for the unfused path, which would
    also write p outputs).  Per-call device time from CUDA-graph replay."""
    import torch
    import reducescatter_reduction_gb300 as ccl

    p, hidden = 8, 8192
    rows_out = {}
    for tokens in (1, 32, 256, 4096):
        n = tokens * hidden
        ins = [(0.02 * torch.randn(n, device=dev)).to(torch.bfloat16) for _ in range(p)]
        outs = [torch.empty_like(t) for t in ins]
        res = torch.randn(n, device=dev).to(torch.bfloat16)
        res_out = torch.empty_like(res)
        gamma = torch.randn(hidden, device=dev).to(torch.bfloat16)
        h = ccl.ccl_comm_create(p, [t.data_ptr() for t in ins])
        ccl.ccl_comm_set_outputs(h, [t.data_ptr() for t in outs])

        def fused(s):
            ccl.ccl_allreduce_residual_rmsnorm(h, "bf16", tokens, hidden, res.data_ptr(), res_out.data_ptr(),
                                               gamma.data_ptr(), 1e-6, "ring", s)

        def ar_only(s):
            ccl.ccl_allreduce(h, "sum", "bf16", n, "ring", s)

        def unfused(s):
            ccl.ccl_allreduce(h, "sum", "bf16", n, "ring", s)
            y = outs[0].view(tokens, hidden)
            hh = (y.float() + res.view(tokens, hidden).float()).to(torch.bfloat16)
            hf = hh.float()
            o = hf * torch.rsqrt(hf.pow(2).mean(-1, keepdim=True) + 1e-6) * gamma.float()
            res_out.view(tokens, hidden).copy_(hh)
            outs[1].view(tokens, hidden).copy_(o.to(torch.bfloat16))

        calls = 50 if tokens == 1 else 10
        row = {}
        fused(torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        fused_launch = ccl.ccl_comm_last_launch(h)
        for name, fn in (("fused", fused), ("allreduce_only", ar_only), ("allreduce_then_torch_epilogue", unfused)):
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                fn(side.cuda_stream)                      # warm-up (kernel attributes, torch caches)
                side.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    cs = torch.cuda.current_stream().cuda_stream
                    for _ in range(calls):
                        fn(cs)
            torch.cuda.current_stream().wait_stream(side)
            g.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(5):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            row[name] = {"us": round(e0.elapsed_time(e1) * 1e3 / (5 * calls), 2)}
        nbytes = (2 * p + 2) * n * S + hidden * S
        row["fused"]["bytes"] = nbytes
        row["fused"]["GBps"] = round(nbytes / (row["fused"]["us"] * 1e-6) / 1e9, 1)
        row["fused"]["frac_of_hbm_peak"] = round(row["fused"]["GBps"] / peak, 4)
        row["launch"] = fused_launch
        rows_out[f"tokens_{tokens}"] = row
        ccl.ccl_comm_destroy(h)
        del ins, outs, res, res_out
        torch.cuda.empty_cache()
    return rows_out


def run_budgets(dev, sptr, stream, peak, p=16, n=16384 * 7168, variants=("ldst", "tma", "tma_bulkred"),
                budgets=(4, 8, 16, 32, 76, 0)):
    """At SM budgets from 4 SMs to the whole GPU, per variant (T-CCL's
    restricted-CTA-budget comparison).  Default: the MoE hidden-state
    AllReduce, p=16 bf16 [16384, 7168] per rank (224 MiB, 3.5 GiB in +
    3.5 GiB out), ring; also run at p=8, 32 MiB per rank."""
    import torch
    import reducescatter_reduction_gb300 as ccl

    nbytes = 2 * p * n * S
    ins = [torch.randn(n, device=dev, dtype=torch.float32).to(torch.bfloat16) for _ in range(p)]
    outs = [torch.empty_like(t) for t in ins]
    h = ccl.ccl_comm_create(p, [t.data_ptr() for t in ins])
    ccl.ccl_comm_set_outputs(h, [t.data_ptr() for t in outs])
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    rows = []
    for variant in variants:
        for budget in budgets:
            ccl.ccl_set_launch(h, budget, variant, 0)
            for _ in range(2):
                ccl.ccl_allreduce(h, "sum", "bf16", n, "ring", sptr)
            torch.cuda.synchronize()
            iters = 3 if budget and budget <= 16 else 10
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(iters):
                ccl.ccl_allreduce(h, "sum", "bf16", n, "ring", sptr)
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / iters
            gbs = nbytes / (ms * 1e-3) / 1e9
            used = budget or sms
            rows.append({"variant": variant, "sm_budget": budget or "all", "ms": round(ms, 3),
                         "GBps": round(gbs, 1), "GBps_per_SM": round(gbs / used, 2),
                         "frac_of_hbm_peak": round(gbs / peak, 4),
                         "launch": ccl.ccl_comm_last_launch(h)})
    ccl.ccl_comm_check(h)
    ccl.ccl_comm_destroy(h)
    del ins, outs
    torch.cuda.empty_cache()
    return rows


def graph_latency(comms, sets, n, sched, calls=200):
    """Per-call device time with the host out of the way: `calls` AllReduces
    (rotating buffer sets) captured in one CUDA graph and replayed."""
    import torch
    import reducescatter_reduction_gb300 as ccl

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            cs = torch.cuda.current_stream().cuda_stream
            for i in range(calls):
                ccl.ccl_allreduce(comms[i % sets], "sum", "bf16", n, sched, cs)
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (5 * calls)


def launch_floor(calls=200):
    """Per-launch time of an empty kernel (torch.cuda._sleep(0): one thread,
    no memory access) replayed the same way as graph_latency: the floor the
    small-message calls are measured against."""
    import torch

    if not hasattr(torch.cuda, "_sleep"):
        return None
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        torch.cuda._sleep(0)
        side.synchronize()
        with torch.cuda.graph(g, stream=side):
            for _ in range(calls):
                torch.cuda._sleep(0)
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return {"us_graph": round(e0.elapsed_time(e1) * 1e3 / (5 * calls), 3),
            "kernel": "empty kernel (torch.cuda._sleep(0)), ordinary launches, CUDA-graph replay"}


def run_sweep(dist, dev, sptr, stream, peak, l2, big_inputs):
    """GB/s vs message size, 1 KiB .. 256 MiB per rank, ring and all-pairs.
    Buffer sets rotate so that every timed call works on data that the
    previous calls did not leave in L2 (>= 4 x L2 across the sets)."""
    import torch
    import reducescatter_reduction_gb300 as ccl

    rows = []
    l2 = l2 or (126 << 20)
    for k in range(9, 28):
        n = 1 << k
        per_set = 2 * P * n * S
        sets = 1 if per_set >= 4 * l2 else min(64, max(3, math.ceil(4 * l2 / per_set)))
        comms, keep = [], []
        for i in range(sets):
            if n == big_inputs[0].numel() and i == 0:
                src = big_inputs
            else:
                src = [torch.randn(n, device=dev, dtype=torch.float32).to(torch.bfloat16) for _ in range(P)]
            dst = [torch.empty_like(t) for t in src]
            h = ccl.ccl_comm_create(P, [t.data_ptr() for t in src])
            ccl.ccl_comm_set_outputs(h, [t.data_ptr() for t in dst])
            comms.append(h)
            keep.append((src, dst))
        row = {"bytes_per_rank": n * S, "rotating_sets": sets}
        for sched in ("ring", "allpairs"):
            iters = max(20, min(2000, int(0.2 / max(per_set / 5e12, 5e-6))))
            for i in range(10):
                ccl.ccl_allreduce(comms[i % sets], "sum", "bf16", n, sched, sptr)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(iters):
                ccl.ccl_allreduce(comms[i % sets], "sum", "bf16", n, sched, sptr)
            e1.record(stream)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / iters
            gbs = per_set / (us * 1e-6) / 1e9
            row[sched] = {"us": round(us, 3), "GBps": round(gbs, 1),
                          "frac_of_hbm_peak": round(gbs / peak, 4) if per_set >= 4 * l2 else None}
            if n * S <= (4 << 20):
                row[sched]["us_graph"] = round(graph_latency(comms, sets, n, sched), 3)
        rows.append(row)
        for h in comms:
            ccl.ccl_comm_destroy(h)
        del keep
        torch.cuda.empty_cache()
    return rows


# ---------------------------------------------------------------------------
# CPU oracle (the baseline; also the --impl reference arm)
# ---------------------------------------------------------------------------

def _time_oracle(xs, reps=1):
    import oracle
    t = time.perf_counter()
    for _ in range(reps):
        oracle.allreduce(xs, "sum", "bf16", "ring")
    return (time.perf_counter() - t) / reps


def _host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _time_oracle_threads(parts):
    """Wall time of one oracle AllReduce per element of ``parts``, all run at
    once, each on its own thread (the oracle's ctypes calls release the GIL)."""
    import threading
    import oracle
    oracle.lib()
    ths = [threading.Thread(target=oracle.allreduce, args=(xs, "sum", "bf16", "ring")) for xs in parts]
    t = time.perf_counter()
    for th in ths:
        th.start()
    for th in ths:
        th.join()
    return time.perf_counter() - t


def _threaded_sample(host_slice, total, cores, single_rate, target_s):
    """Split the first ``total`` elements of each rank buffer into ``cores``
    disjoint slices, one oracle AllReduce per slice on its own thread; repeat
    until ~target_s of wall time.  Returns (GB/s, slice elements, reps, s)."""
    n_t = total // cores
    big = host_slice(n_t * cores)
    parts = [[x[i * n_t:(i + 1) * n_t] for x in big] for i in range(cores)]
    once = _time_oracle_threads(parts)
    reps = max(1, min(64, int(math.ceil(target_s / max(once, 1e-6)))))
    t = time.perf_counter()
    for _ in range(reps):
        _time_oracle_threads(parts)
    secs = time.perf_counter() - t
    return 2.0 * P * n_t * cores * S * reps / secs / 1e9, n_t, reps, secs


def _host_cpu() -> str:
    """The host CPU's model name (reported beside the oracle timings)."""
    import platform
    import subprocess
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine() or "unknown"


def cpu_baseline_from(ins):
    """Time the oracle, as it stands, on a slice of the benchmark's own inputs:
    single-threaded on ~10-15 s of work, and on every host core at once (one
    oracle call per core on disjoint slices) for a few seconds."""
    import numpy as np
    import torch

    def host_slice(n):
        return [t[:n].view(torch.int16).cpu().numpy().view(np.uint16).copy() for t in ins]

    probe_n = 1 << 20
    rate = probe_n / _time_oracle(host_slice(probe_n))   # elements per second per call
    n = probe_n
    while n * 2 <= ins[0].numel() and (n * 2) / rate <= 15.0:
        n *= 2
    secs = _time_oracle(host_slice(n))
    gbs1 = 2.0 * P * n * S / secs / 1e9
    single = {"value": round(gbs1, 4), "cores": 1, "seconds": round(secs, 3),
              "sample": f"first {n} elements (2^{int(math.log2(n))}) of each of the 8 rank buffers, "
                        "one ring AllReduce call on one thread"}
    cores = _host_cores()
    if cores < 2:
        return {"value": round(gbs1, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "cpu": _host_cpu(),
                "sample": single["sample"] + f", {secs:.2f} s", "seconds": round(secs, 3)}
    gbs, n_t, reps, tsecs = _threaded_sample(host_slice, ins[0].numel(), cores, rate, 4.0)
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "cpu": _host_cpu(),
            "sample": f"the 2^27-element rank buffers of the benchmark workload split into {cores} disjoint "
                      f"slices of {n_t} elements, one ring AllReduce per slice on its own thread, all at once, "
                      f"{reps} times ({tsecs:.2f} s wall)",
            "seconds": round(tsecs, 3), "single_thread": single}


def run_reference(args, dist: Dist):
    """The CPU oracle, timed on the host cores, on bounded samples of the
    workload: each step one oracle AllReduce of n_s elements per rank."""
    import numpy as np
    from reducescatter_reduction_gb300 import inputs

    if dist.rank != 0:
        return None
    probe = 1 << 18
    xs = inputs.sweep(probe, P)
    rate = probe / _time_oracle(xs, reps=3)
    cores = _host_cores()
    budget = 90.0 / max(1, args.steps + args.warmup)      # whole run within ~1.5 min
    n = probe                                             # elements per rank per thread
    while n * 2 * cores <= N and (n * 2) / rate <= budget:
        n *= 2
    while n > 512 and n / rate > budget:
        n //= 2
    full = inputs.sweep(n * cores, P)
    parts = [[x[i * n:(i + 1) * n] for x in full] for i in range(cores)]
    for _ in range(args.warmup):
        _time_oracle_threads(parts)
    secs = 0.0
    for _ in range(args.steps):
        secs += _time_oracle_threads(parts)
    gbs = 2.0 * P * n * cores * S * args.steps / secs / 1e9
    sample = (f"p=8 bf16 ring AllReduce: each step {cores} oracle calls at once, one per host core, each on its "
              f"own {n}-element (2^{int(math.log2(n))}) slice of every rank buffer of the 2^27-element workload")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(gbs, 4),
        "unit": "GB/s",
        "n_gpus": dist.world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(secs * 1e3 / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": sample, "p": P, "n_per_step": n * cores},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "cpu": _host_cpu(), "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_single(args, dist: Dist, p: int, n: int, mode: dict) -> int:
    """One bf16 sum AllReduce of p ranks of n elements (N(0,1) inputs, ring),
    with the chosen variant and SM budget: warm-up, then the timed steps; one
    JSON line.  The profiling modes (--moe-rows, --ranks) that the summaries
    in profiles/ name."""
    import torch
    import __graft_entry__
    import reducescatter_reduction_gb300 as ccl
    __graft_entry__.build()
    dev = torch.device("cuda", dist.local_rank)
    ins = [torch.randn(n, device=dev, dtype=torch.float32).to(torch.bfloat16) for _ in range(p)]
    outs = [torch.empty_like(t) for t in ins]
    h = ccl.ccl_comm_create(p, [t.data_ptr() for t in ins])
    ccl.ccl_comm_set_outputs(h, [t.data_ptr() for t in outs])
    ccl.ccl_set_launch(h, args.sm_budget, args.variant, 0)
    s = torch.cuda.current_stream()
    for _ in range(args.warmup):
        ccl.ccl_allreduce(h, "sum", "bf16", n, "ring", s.cuda_stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        ccl.ccl_allreduce(h, "sum", "bf16", n, "ring", s.cuda_stream)
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / max(1, args.steps)
    ccl.ccl_comm_check(h)
    print(json.dumps(dict(mode, variant=args.variant, sm_budget=args.sm_budget, us_per_call=round(us, 2),
                          GBps=round(2 * p * n * S / (us * 1e-6) / 1e9, 1),
                          launch=ccl.ccl_comm_last_launch(h))), flush=True)
    ccl.ccl_comm_destroy(h)
    return 0


def main(argv=None):
    args = parse_args(argv)
    dist = Dist()
    if args.rmsnorm_tokens:
        import torch
        import __graft_entry__
        import reducescatter_reduction_gb300 as ccl
        __graft_entry__.build()
        dev = torch.device("cuda", dist.local_rank)
        tokens, hidden, n = args.rmsnorm_tokens, 8192, args.rmsnorm_tokens * 8192
        ins = [(0.02 * torch.randn(n, device=dev)).to(torch.bfloat16) for _ in range(P)]
        outs = [torch.empty_like(t) for t in ins]
        res = torch.randn(n, device=dev).to(torch.bfloat16)
        res_out = torch.empty_like(res)
        gamma = torch.randn(hidden, device=dev).to(torch.bfloat16)
        h = ccl.ccl_comm_create(P, [t.data_ptr() for t in ins])
        ccl.ccl_comm_set_outputs(h, [t.data_ptr() for t in outs])
        s = torch.cuda.current_stream()
        for _ in range(args.warmup):
            ccl.ccl_allreduce_residual_rmsnorm(h, "bf16", tokens, hidden, res.data_ptr(), res_out.data_ptr(),
                                               gamma.data_ptr(), 1e-6, "ring", s.cuda_stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            ccl.ccl_allreduce_residual_rmsnorm(h, "bf16", tokens, hidden, res.data_ptr(), res_out.data_ptr(),
                                               gamma.data_ptr(), 1e-6, "ring", s.cuda_stream)
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / max(1, args.steps)
        print(json.dumps({"mode": "rmsnorm", "tokens": tokens, "us_per_call": round(us, 2),
                          "launch": ccl.ccl_comm_last_launch(h)}), flush=True)
        ccl.ccl_comm_destroy(h)
        return 0
    if args.moe_rows or args.ranks:
        # profiling modes: one AllReduce configuration, timed alone
        if args.moe_rows:
            p, n, mode = 16, args.moe_rows * 7168, {"mode": "moe", "rows": args.moe_rows}
        else:
            p = args.ranks
            n = args.n - args.n % (8 * p)          # whole 16-byte groups in every chunk
            mode = {"mode": "ranks", "p": p, "n": n}
        return run_single(args, dist, p, n, mode)
    if args.host_buffers:
        import torch
        import __graft_entry__
        import reducescatter_reduction_gb300 as ccl
        __graft_entry__.build()
        dev = torch.device("cuda", dist.local_rank)
        torch.cuda.set_device(dev)
        n = args.n
        ins = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True) for _ in range(P)]
        for t in ins:
            t.copy_(torch.randn(n, device=dev).to(torch.bfloat16))
        outs = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True) for _ in range(P)]
        h = ccl.ccl_comm_create(P, [t.data_ptr() for t in ins])
        ccl.ccl_comm_set_outputs(h, [t.data_ptr() for t in outs])
        ccl.ccl_set_launch(h, args.sm_budget, "ldst", 0)
        s = torch.cuda.current_stream()
        for _ in range(args.warmup):
            ccl.ccl_allreduce(h, "sum", "bf16", n, "ring", s.cuda_stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            ccl.ccl_allreduce(h, "sum", "bf16", n, "ring", s.cuda_stream)
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / max(1, args.steps)
        ccl.ccl_comm_check(h)
        print(json.dumps({"mode": "host_buffers", "n_per_rank": n, "sm_budget": args.sm_budget,
                          "us_per_call": round(us, 2), "GBps": round(2 * P * n * S / (us * 1e-6) / 1e9, 1),
                          "launch": ccl.ccl_comm_last_launch(h)}), flush=True)
        ccl.ccl_comm_destroy(h)
        return 0
    if args.collective:
        return run_collective_only(args, dist)
    if args.calibrate:
        import torch
        import __graft_entry__
        __graft_entry__.build()
        print(json.dumps(calibrate(torch.device("cuda", dist.local_rank))), flush=True)
        return 0
    if args.impl == "reference":
        res = run_reference(args, dist)
    else:
        res = run_ours(args, dist)
    if dist.rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
