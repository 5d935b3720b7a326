"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, and its host logic (schedule builder, schedule validator, cost
model, argument checks that need no device) is right."""
import ctypes
import os
import re
import subprocess

import pytest

import oracle
import reducescatter_reduction_gb300 as ccl
from reducescatter_reduction_gb300 import build as ccl_build
from conftest import ROOT, golden_orders, read_golden

pytestmark = pytest.mark.cpu


@pytest.fixture(scope="module")
def lib():
    ccl_build.build()
    return ccl.load_library()


def header_symbols():
    text = open(os.path.join(ROOT, "include", "ccl.h")).read()
    return sorted(set(re.findall(r"CCL_API\s+[\w\s\*]*?\b(ccl_\w+)\s*\(", text)))


def test_header_symbols_listed_in_binding():
    assert header_symbols() == sorted(ccl.EXPORTS)


def test_library_exports_every_header_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", ccl.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for sym in header_symbols():
        assert sym in exported, sym
        assert hasattr(lib, sym)
    # nothing else leaks out of the C ABI
    assert {s for s in exported if s.startswith("ccl_")} == set(header_symbols())


def test_version(lib):
    assert ccl.ccl_version() == 10000


@pytest.mark.parametrize("fixture,p,sched", [
    ("ring_order_p3.txt", 3, "ring"),
    ("ring_order_p4.txt", 4, "ring"),
    ("ring_order_p8.txt", 8, "ring"),
    ("allpairs_order_p8.txt", 8, "allpairs"),
])
def test_schedule_orders_match_pages(lib, fixture, p, sched):
    _, order = ccl.ccl_schedule_build(p, 1000, sched)
    for c, want in golden_orders(fixture).items():
        assert order[c] == want


@pytest.mark.parametrize("p", [1, 2, 3, 7, 8, 16, 64])
@pytest.mark.parametrize("n", [0, 1, 5, 4096, 4099, 117440512])
@pytest.mark.parametrize("sched", ["ring", "allpairs"])
def test_schedule_table_matches_oracle(lib, p, n, sched):
    bounds, order = ccl.ccl_schedule_build(p, n, sched)
    for c in range(p):
        assert (bounds[c], bounds[c + 1]) == oracle.chunk_bounds(p, n, c)
        assert order[c] == oracle.chunk_order(p, sched, c)
    assert ccl.ccl_schedule_check(p, n, bounds, order) == ccl.CCL_OK


def test_schedule_check_rejects_bad_tables(lib):
    p, n = 4, 100
    bounds, order = ccl.ccl_schedule_build(p, n, "ring")
    bad = [row[:] for row in order]
    bad[2][1] = bad[2][0]                                  # rank repeated
    assert ccl.ccl_schedule_check(p, n, bounds, bad) == ccl.CCL_ERR_INVALID_ARG
    bad = [row[:] for row in order]
    bad[0][0] = 9                                          # rank out of range
    assert ccl.ccl_schedule_check(p, n, bounds, bad) == ccl.CCL_ERR_INVALID_ARG
    b2 = bounds[:]
    b2[-1] = n - 1                                         # does not cover [0, n)
    assert ccl.ccl_schedule_check(p, n, b2, order) == ccl.CCL_ERR_INVALID_ARG
    b2 = bounds[:]
    b2[1], b2[2] = b2[2], b2[1]                            # decreasing bounds
    assert ccl.ccl_schedule_check(p, n, b2, order) == ccl.CCL_ERR_INVALID_ARG
    assert "permutation" in ccl.ccl_last_error() or "bounds" in ccl.ccl_last_error()


def test_schedule_build_rejects(lib):
    for p, sched in [(0, "ring"), (65, "ring"), (4, "auto"), (4, "custom")]:
        with pytest.raises(ccl.CclError) as ei:
            ccl.ccl_schedule_build(p, 10, sched)
        assert ei.value.status == ccl.CCL_ERR_INVALID_ARG


def _page_params():
    g = {r[0]: r[1:] for r in read_golden("cost_model_example.txt")}
    return g, ccl.CostParams(float(g["alpha_us"][0]) * 1e-6, float(g["bw_GBps"][0]) * 1e9,
                             float(g["eff_ring"][0]), float(g["eff_allpairs"][0]))


def test_cost_model_worked_example(lib):
    g, prm = _page_params()
    p = int(g["p"][0])
    nb, want = int(g["speedup_allpairs_at_bytes"][0]), float(g["speedup_allpairs_at_bytes"][1])
    r = ccl.ccl_cost_estimate(p, nb, "ring", prm) / ccl.ccl_cost_estimate(p, nb, "allpairs", prm)
    assert round(r, 2) == want
    nb, want = int(g["speedup_ring_at_bytes"][0]), float(g["speedup_ring_at_bytes"][1])
    r = ccl.ccl_cost_estimate(p, nb, "allpairs", prm) / ccl.ccl_cost_estimate(p, nb, "ring", prm)
    assert round(r, 1) == want
    # NULL parameters are the page's assumptions
    assert ccl.ccl_cost_estimate(p, 12345, "ring") == ccl.ccl_cost_estimate(p, 12345, "ring", prm)


def test_cost_model_matches_oracle_and_selects(lib):
    g, prm = _page_params()
    p = 8
    for nb in [1 << k for k in range(10, 32)]:
        tr = oracle.time_ring(p, nb, prm.alpha_s, prm.bw_bytes_per_s, prm.eff_ring)
        ta = oracle.time_allpairs(p, nb, prm.alpha_s, prm.bw_bytes_per_s, prm.eff_allpairs)
        assert ccl.ccl_cost_estimate(p, nb, "ring", prm) == pytest.approx(tr, rel=1e-12)
        assert ccl.ccl_cost_estimate(p, nb, "allpairs", prm) == pytest.approx(ta, rel=1e-12)
        want = ccl.CCL_SCHED_ALLPAIRS if ta < tr else ccl.CCL_SCHED_RING
        assert ccl.ccl_select_schedule(p, nb, prm) == want
    xover = float(g["crossover_MiB"][0]) * 2 ** 20
    assert ccl.ccl_select_schedule(p, 0.9 * xover, prm) == ccl.CCL_SCHED_ALLPAIRS
    assert ccl.ccl_select_schedule(p, 1.1 * xover, prm) == ccl.CCL_SCHED_RING
    assert ccl.ccl_select_schedule(1, 1e6, prm) == ccl.CCL_SCHED_RING   # p=1: tie -> ring


def test_cost_model_bad_arguments(lib):
    assert ccl.ccl_cost_estimate(0, 100, "ring") < 0
    assert ccl.ccl_cost_estimate(8, -1, "ring") < 0
    assert ccl.ccl_cost_estimate(8, 100, "custom") < 0


def test_null_comm_is_rejected(lib):
    L = lib
    for st in (L.ccl_allreduce(None, 0, 0, 10, 0, None), L.ccl_reduce_scatter(None, 0, 0, 10, 0, None),
               L.ccl_all_gather(None, 0, 10, None), L.ccl_set_launch(None, 0, 0, 0),
               L.ccl_comm_set_outputs(None, None), L.ccl_comm_check(None)):
        assert st == ccl.CCL_ERR_INVALID_ARG
    assert L.ccl_comm_destroy(None) == ccl.CCL_OK
    assert ccl.ccl_comm_launch_count(None) == 0


def test_comm_create_argument_checks(lib):
    h = ctypes.c_void_p()
    ptrs = (ctypes.c_void_p * 2)(0x1000, 0)
    assert lib.ccl_comm_create(ctypes.byref(h), 2, ptrs) == ccl.CCL_ERR_INVALID_ARG   # NULL buffer
    assert "rank_ptrs[1]" in ccl.ccl_last_error()
    assert lib.ccl_comm_create(ctypes.byref(h), 0, ptrs) == ccl.CCL_ERR_INVALID_ARG
    assert lib.ccl_comm_create(ctypes.byref(h), 65, ptrs) == ccl.CCL_ERR_INVALID_ARG
    assert lib.ccl_comm_create(None, 2, ptrs) == ccl.CCL_ERR_INVALID_ARG
    assert lib.ccl_comm_create(ctypes.byref(h), 2, None) == ccl.CCL_ERR_INVALID_ARG


def test_comm_create_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    ptrs = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    assert lib.ccl_comm_create(ctypes.byref(h), 2, ptrs) == ccl.CCL_ERR_CUDA
    assert h.value is None


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(ccl, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        ccl.load_library(str(tmp_path / "libccl.so"))


def test_binding_refuses_pointer_lists_of_the_wrong_length():
    # the C side reads exactly p pointers; the binding checks the list first
    with pytest.raises(ccl.CclError) as ei:
        ccl.ccl_comm_create(3, [16, 32])
    assert ei.value.status == ccl.CCL_ERR_INVALID_ARG and "p = 3" in str(ei.value)
    with pytest.raises(ccl.CclError) as ei:
        ccl.ccl_allreduce_static(2, [16, 32], [16], "sum", "f32", 8)
    assert ei.value.status == ccl.CCL_ERR_INVALID_ARG
