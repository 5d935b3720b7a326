"""Measure the launch table that CCL_VARIANT_AUTO reads, and write it as
csrc/launch_table.inc (then rebuild the library).

T-CCL, section "Launch Configuration Tuning": configurations are profiled
offline and ranked per message size in a table that the runtime consults.
Here the configurations are the two fixed-order kernels, ld/st and TMA
(their results are identical bit for bit, so the choice changes only the
time), and the table holds the per-call device time of each at measured
points: rank count p, element size (2 or 4 bytes), SM budget (0 = every SM)
and bytes per rank.  The library interpolates between points; see
``ccl_launch_estimate`` in include/ccl.h.

What is timed: ccl_allreduce, sum, ring schedule, out of place, rank buffers
of random bits, through the C ABI.  Small calls (< 0.2 ms) are replayed
back to back from a CUDA graph, larger ones timed with CUDA events around
a loop; each point is the lower of two measurements.  A size sweep for one
configuration stops once a call takes longer than 4 ms (larger sizes are in
the bandwidth-bound regime, where the library extrapolates linearly), and
never asks for more than 4 GiB of inputs.

Usage (on the GPU the table is for):
    python -m reducescatter_reduction_gb300.calibrate [--quick] [--out PATH]
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import sys

_HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(_HERE, "csrc", "launch_table.inc")

P_POINTS = [2, 3, 4, 5, 8, 12, 16, 24, 32, 48, 64]
ELEM_BYTES = {2: "bf16", 4: "f32"}
BUDGETS = [4, 8, 16, 32, 76, 0]
SIZES = [16 << 10, 64 << 10, 256 << 10, 1 << 20, 4 << 20, 16 << 20, 64 << 20, 256 << 20]
MAX_INPUT_BYTES = 4 << 30
STOP_MS = 4.0


def _time_us(call, torch, stream):
    """Per-call device time (us): graph replay for short calls, events for long."""
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    call()
    e1.record(stream)
    torch.cuda.synchronize()
    one_ms = e0.elapsed_time(e1)
    best = float("inf")
    if one_ms < 0.2:
        k = 100
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(k):
                call()
        g.replay()
        torch.cuda.synchronize()
        for _ in range(2):
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) * 1e3 / k)
        del g
    else:
        k = max(3, min(50, int(10.0 / one_ms)))
        for _ in range(2):
            e0.record(stream)
            for _ in range(k):
                call()
            e1.record(stream)
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) * 1e3 / k)
    return best


def measure(quick=False, log=print, p_points=None, budgets=None, sizes=None):
    import torch
    import reducescatter_reduction_gb300 as ccl
    from reducescatter_reduction_gb300 import build

    build.build()
    ccl.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    props = torch.cuda.get_device_properties(dev)
    stream = torch.cuda.Stream(dev)
    p_points = p_points or ([2, 8, 16, 64] if quick else P_POINTS)
    budgets = budgets or ([8, 76, 0] if quick else BUDGETS)
    sizes = sizes or SIZES
    rows = []
    with torch.cuda.stream(stream):
        for p in p_points:
            max_rank_bytes = min(sizes[-1], MAX_INPUT_BYTES // p)
            ins = [torch.empty(max_rank_bytes, dtype=torch.uint8, device=dev).random_() for _ in range(p)]
            outs = [torch.empty(max_rank_bytes, dtype=torch.uint8, device=dev) for _ in range(p)]
            comm = ccl.ccl_comm_create(p, [t.data_ptr() for t in ins])
            ccl.ccl_comm_set_outputs(comm, [t.data_ptr() for t in outs])
            try:
                for es, dtype in ELEM_BYTES.items():
                    for budget in budgets:
                        stopped = {"ldst": False, "tma": False}
                        for nbytes in sizes:
                            if nbytes > max_rank_bytes:
                                break
                            n = nbytes // es
                            n -= n % (p * 16 // es)          # chunks of whole 16-byte groups: TMA can run
                            us = {}
                            for variant in ("ldst", "tma"):
                                if stopped[variant]:
                                    continue
                                ccl.ccl_set_launch(comm, budget, variant, 0)
                                call = lambda: ccl.ccl_allreduce(comm, "sum", dtype, n, "ring", stream.cuda_stream)
                                us[variant] = _time_us(call, torch, stream)
                                if us[variant] > STOP_MS * 1e3:
                                    stopped[variant] = True
                            ccl.ccl_comm_check(comm)
                            if "ldst" in us and "tma" in us:
                                rows.append({"p": p, "elem_bytes": es, "sm_budget": budget, "bytes_per_rank": n * es,
                                             "us_ldst": round(us["ldst"], 3), "us_tma": round(us["tma"], 3)})
                                log(json.dumps(rows[-1]))
                            if all(stopped.values()):
                                break
            finally:
                ccl.ccl_comm_destroy(comm)
                del ins, outs
                torch.cuda.empty_cache()
    return {"device": props.name, "sms": props.multi_processor_count,
            "when": datetime.datetime.now(datetime.timezone.utc).strftime("%Y-%m-%dT%H:%M:%SZ"),
            "rows": rows}


def render(table) -> str:
    """The C++ include the library compiles (see csrc/launch_table.cpp)."""
    lines = [
        "// Launch table for CCL_VARIANT_AUTO, written by reducescatter_reduction_gb300/calibrate.py -- do not",
        "// edit by hand; run the script on the GPU the table is for and rebuild.",
        f"// Measured on {table['device']} ({table['sms']} SMs), {table['when']}: per-call device time of",
        "// ccl_allreduce (sum, ring, out of place) for the ld/st and TMA kernels.",
        "// Columns: p, element bytes, SM budget (0 = every SM), bytes per rank, us ld/st, us TMA.",
        f"static const int kLaunchTableSms = {int(table['sms'])};",
        "static const LaunchPoint kLaunchTable[] = {",
    ]
    rows = sorted(table["rows"], key=lambda r: (r["p"], r["elem_bytes"], r["sm_budget"], r["bytes_per_rank"]))
    for r in rows:
        lines.append(f"    {{{r['p']}, {r['elem_bytes']}, {r['sm_budget']}, {r['bytes_per_rank']}ull, "
                     f"{r['us_ldst']:.3f}f, {r['us_tma']:.3f}f}},")
    lines.append("    {0, 0, 0, 0ull, 0.0f, 0.0f},  // end")
    lines.append("};")
    return "\n".join(lines) + "\n"


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--out", default=OUT)
    ap.add_argument("--json", default=None, help="also write the measured rows as JSON here")
    ap.add_argument("--quick", action="store_true", help="a few rank counts and budgets only (a trial run)")
    args = ap.parse_args(argv)
    table = measure(quick=args.quick, log=lambda s: print(s, file=sys.stderr, flush=True))
    with open(args.out, "w") as f:
        f.write(render(table))
    if args.json:
        with open(args.json, "w") as f:
            json.dump(table, f, indent=1)
    print(f"{len(table['rows'])} points -> {args.out}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
