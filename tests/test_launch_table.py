"""The measured launch table behind CCL_VARIANT_AUTO and its lookup,
ccl_launch_estimate, on the CPU (no GPU needed): the committed table covers
every rank count, element size and SM budget the calibration measures, and
the estimates are the table's own numbers at measured points, a power law
between neighbouring sizes, the smallest size's time below it and the line
through the two largest sizes above it, at the nearest measured rank count
and budget (T-CCL, section "Launch Configuration Tuning")."""
import math
import os
import re

import pytest

import reducescatter_reduction_gb300 as ccl
from reducescatter_reduction_gb300 import build as ccl_build
from reducescatter_reduction_gb300 import calibrate

pytestmark = pytest.mark.cpu

ROW = re.compile(r"\{(\d+), (\d+), (\d+), (\d+)ull, ([0-9.]+)f, ([0-9.]+)f\}")
DT = {2: "bf16", 4: "f32"}


@pytest.fixture(scope="module")
def table():
    ccl_build.build()
    ccl.load_library()
    text = open(os.path.join(ccl_build.CSRC, "launch_table.inc")).read()
    sms = int(re.search(r"kLaunchTableSms = (\d+);", text).group(1))
    rows = [tuple(int(v) for v in m.groups()[:4]) + (float(m.group(5)), float(m.group(6)))
            for m in ROW.finditer(text)]
    rows = [r for r in rows if r[0] != 0]
    return sms, rows


def key_rows(rows, p, es, b):
    return sorted((r for r in rows if r[:3] == (p, es, b)), key=lambda r: r[3])


def test_table_covers_every_measured_configuration(table):
    sms, rows = table
    assert rows, "the launch table is empty"
    assert rows == sorted(rows, key=lambda r: r[:4])
    for p in calibrate.P_POINTS:
        for es in calibrate.ELEM_BYTES:
            for b in calibrate.BUDGETS:
                pts = key_rows(rows, p, es, b)
                assert len(pts) >= 3, (p, es, b)
                assert pts[0][3] <= 16 << 10
                assert all(r[4] > 0 and r[5] > 0 for r in pts)
                # the size sweep reaches the bandwidth-bound regime: the last step
                # costs at least twice the step before it (4x the bytes)
                assert pts[-1][4] > 1.5 * pts[-2][4] or pts[-1][3] >= 64 << 20, (p, es, b)


def test_estimate_is_the_table_at_measured_points(table):
    sms, rows = table
    for p, es, b, nbytes, us_l, us_t in rows[:: max(1, len(rows) // 200)]:
        for variant, want in (("ldst", us_l), ("tma", us_t)):
            got = ccl.ccl_launch_estimate(p, DT[es], b, nbytes, variant)
            assert math.isclose(got, want, rel_tol=1e-6), (p, es, b, nbytes, variant)


def test_power_law_between_sizes_and_line_above(table):
    sms, rows = table
    p, es, b = 8, 2, 0
    pts = key_rows(rows, p, es, b)
    for lo, hi in zip(pts, pts[1:]):
        mid = int(math.sqrt(lo[3] * hi[3]))
        got = ccl.ccl_launch_estimate(p, "bf16", b, mid, "ldst")
        f = math.log(mid / lo[3]) / math.log(hi[3] / lo[3])
        want = math.exp(math.log(lo[4]) + f * (math.log(hi[4]) - math.log(lo[4])))
        assert math.isclose(got, want, rel_tol=1e-6)
        assert min(lo[4], hi[4]) <= got <= max(lo[4], hi[4])
    a, z = pts[-2], pts[-1]
    big = 4 * z[3]
    got = ccl.ccl_launch_estimate(p, "bf16", b, big, "tma")
    assert math.isclose(got, z[5] + (z[5] - a[5]) / (z[3] - a[3]) * (big - z[3]), rel_tol=1e-6)
    assert math.isclose(ccl.ccl_launch_estimate(p, "bf16", b, 1, "ldst"), pts[0][4], rel_tol=1e-6)


def test_nearest_rank_count_and_budget(table):
    sms, rows = table
    ps = sorted({r[0] for r in rows})
    nbytes = 1 << 20
    for p in range(1, 65):
        near = min(ps, key=lambda t: (abs(math.log2(t) - math.log2(p)), -t))
        assert math.isclose(ccl.ccl_launch_estimate(p, "f32", 0, nbytes, "ldst"),
                            ccl.ccl_launch_estimate(near, "f32", 0, nbytes, "ldst"), rel_tol=1e-9)
    # every SM: budget 0, the SM count, or more
    for b in (sms, sms + 10, 10 * sms):
        assert ccl.ccl_launch_estimate(8, "bf16", b, nbytes, "ldst") == ccl.ccl_launch_estimate(8, "bf16", 0, nbytes, "ldst")
    budgets = sorted({r[2] for r in rows if r[2] > 0})
    for b in range(1, sms):
        near = min(budgets + [sms], key=lambda t: (abs(math.log2(t) - math.log2(b)), -t))
        want = ccl.ccl_launch_estimate(8, "bf16", 0 if near == sms else near, nbytes, "tma")
        assert ccl.ccl_launch_estimate(8, "bf16", b, nbytes, "tma") == want, b
    # fp16 shares the 2-byte rows, int32 the 4-byte rows
    assert ccl.ccl_launch_estimate(8, "f16", 0, nbytes, "ldst") == ccl.ccl_launch_estimate(8, "bf16", 0, nbytes, "ldst")
    assert ccl.ccl_launch_estimate(8, "i32", 0, nbytes, "ldst") == ccl.ccl_launch_estimate(8, "f32", 0, nbytes, "ldst")


def test_estimate_errors():
    ccl_build.build()
    for args in ((0, "bf16", 0, 1024, "ldst"), (65, "bf16", 0, 1024, "ldst"), (8, "bf16", -1, 1024, "ldst"),
                 (8, "bf16", 0, 1024, "tma_bulkred"), (8, "bf16", 0, 1024, "auto")):
        with pytest.raises(ccl.CclError) as ei:
            ccl.ccl_launch_estimate(*args)
        assert ei.value.status == ccl.CCL_ERR_INVALID_ARG


def test_render_round_trips():
    rows = [{"p": 8, "elem_bytes": 2, "sm_budget": 0, "bytes_per_rank": 16384, "us_ldst": 2.15, "us_tma": 3.6},
            {"p": 2, "elem_bytes": 4, "sm_budget": 8, "bytes_per_rank": 1 << 20, "us_ldst": 12.5, "us_tma": 13.25}]
    text = calibrate.render({"device": "GPU", "sms": 152, "when": "now", "rows": rows})
    got = [m.groups() for m in ROW.finditer(text)]
    assert got[0] == ("2", "4", "8", str(1 << 20), "12.500", "13.250")        # sorted by p first
    assert got[1] == ("8", "2", "0", "16384", "2.150", "3.600")
    assert got[-1] == ("0", "0", "0", "0", "0.0", "0.0")                      # the end marker


@pytest.mark.gpu
def test_calibration_script_measures_and_renders_a_table():
    """The script that writes the launch table runs on the GPU (a reduced grid)
    and its rendering parses back into the rows it measured."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    table = calibrate.measure(p_points=[2, 8], budgets=[8, 0], sizes=[16 << 10, 1 << 20], log=lambda s: None)
    rows = table["rows"]
    assert {(r["p"], r["elem_bytes"], r["sm_budget"]) for r in rows} == {
        (p, es, b) for p in (2, 8) for es in (2, 4) for b in (8, 0)}
    assert all(r["us_ldst"] > 0 and r["us_tma"] > 0 for r in rows)
    assert table["sms"] == torch.cuda.get_device_properties(0).multi_processor_count
    parsed = [m.groups() for m in ROW.finditer(calibrate.render(table))]
    assert len(parsed) == len(rows) + 1                                    # rows and the end marker
