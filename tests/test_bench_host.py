"""Host-side logic of bench.py that decides what its JSON line reports, on
the CPU: the measured HBM peak and its fallback, DRAM traffic taken from the
committed ncu summary only while it matches the kernel source, and the
clock-sample summary with its throttle reasons."""
import json
import os

import pytest

import bench

pytestmark = pytest.mark.cpu


def test_peak_is_the_measured_copy_bandwidth_else_the_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peak, src = bench.hbm_peak()
    assert peak == bench.FALLBACK_HBM_GBS and src.startswith("fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6755.8, "bf16_tflops": 1881.1}))
    peak, src = bench.hbm_peak()
    assert peak == 6755.8 and src.startswith("measured")


def test_traffic_only_while_the_record_matches_the_kernel_source(tmp_path, monkeypatch):
    rec = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(rec))
    traffic, why = bench.profiled_traffic()
    assert traffic is None and "missing" in why                   # no record
    rec.write_text(json.dumps({"kernel_source_sha256_16": bench.kernel_source_hash(),
                               "dram_bytes_per_launch": 4293472938, "how": "scaled from 32 MiB per rank"}))
    traffic, why = bench.profiled_traffic()
    assert traffic == 4293472938.0 and "dram__bytes_read.sum" in why and "scaled" in why
    rec.write_text(json.dumps({"kernel_source_sha256_16": "0000000000000000", "dram_bytes_per_launch": 1}))
    traffic, why = bench.profiled_traffic()
    assert traffic is None and "not reported" in why              # taken on another source


def test_committed_traffic_record_names_its_source_and_traffic():
    with open(bench.TRAFFIC_FILE) as f:
        rec = json.load(f)
    assert len(rec["kernel_source_sha256_16"]) == 16
    assert os.path.exists(os.path.join(bench.ROOT, rec["summary"]))
    algorithmic = 2 * bench.P * bench.N * bench.S
    assert rec["algorithmic_bytes_per_launch"] == algorithmic
    assert 0.99 < rec["dram_bytes_per_launch"] / algorithmic < 1.01


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_summary_median_and_reasons(tmp_path):
    path = tmp_path / "clocks.csv"
    path.write_text("2070, 2070, 900.1, 0x0000, Not Active, Not Active, Not Active, Not Active\n"
                    "1965, 2070, 1400.2, 0x0004, Not Active, Not Active, Not Active, Active\n"
                    "2070, 2070, 1100.0, 0x0000, Not Active, Not Active, Not Active, Not Active\n"
                    "[N/A], 2070, 0, 0, x, x, x, x\n")
    s = bench.ClockSampler(None)
    s.proc = _Done()
    s.file = open(path, "r+")
    out = s.stop()
    assert out == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "samples": 3, "reasons": ["sw_power_cap"]}
    assert not os.path.exists(path)


def test_workload_recipe_matches_the_benchmark():
    """The seeded workloads have the shapes the benchmark and the parity tests
    name: the p=8 bf16 sweep up to 2^27 elements (256 MiB) per rank, TP
    activations of hidden 8192 at 1/32/256/4096 tokens, the 64 Mi-element op
    coverage set, the p=16 [16384, 7168] MoE buffers; every workload its own
    seed."""
    from reducescatter_reduction_gb300 import inputs
    assert inputs.SWEEP_N[0] * 2 == 1024 and inputs.SWEEP_N[-1] == bench.N == 1 << 27
    assert bench.P == 8 and bench.S == inputs.ELEM_BYTES["bf16"]
    assert inputs.TP_HIDDEN == 8192 and inputs.TP_TOKENS == [1, 32, 256, 4096]
    assert inputs.COVERAGE_N == 64 * 1024 * 1024
    assert inputs.MOE_SHAPE == (16384, 7168)
    assert len(set(inputs.SEEDS.values())) == len(inputs.SEEDS)
    a = inputs.normal(1000, inputs.SEEDS["sweep"], 3, 1.0, "bf16")
    b = inputs.normal(1000, inputs.SEEDS["sweep"], 3, 1.0, "bf16")
    c = inputs.normal(1000, inputs.SEEDS["sweep"], 4, 1.0, "bf16")
    assert (a == b).all() and not (a == c).all()                  # seeded per (workload, rank)
