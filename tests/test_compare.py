"""GPU tests of the comparison executors: the ring run hop by hop (partials
in the element type, NCCL's ring numerics) against the oracle's stepwise
ring, and one-phase all-pairs against the fused oracle -- bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import reducescatter_reduction_gb300 as ccl
from reducescatter_reduction_gb300 import inputs
from ccl_testutil import bits_equal, ensure_built
from test_parity import gen, run_collective

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ensure_built()


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "prod", "min", "max", "avg"])
def test_ring_stepwise_matches_oracle(dtype, op):
    s = inputs.ELEM_BYTES[dtype]
    for p in (1, 2, 3, 8, 16):
        for n in (p * (16 // s) * 1000, p * 1001 + 3):          # 16-byte groups / element path
            xs = gen(dtype, op, p, n, seed=110 + p)
            want = oracle.allreduce_ring_stepwise(xs, op, dtype)
            for inplace in (False, True):
                res, desc = run_collective(xs, "ar", op, dtype, "ring", variant="ring_stepwise", inplace=inplace)
                if p > 1:
                    assert "allreduce_ring_stepwise" in desc
                for r in range(p):
                    assert bits_equal(res.host(r), want[r]), (p, n, inplace, r)


def test_ring_stepwise_differs_from_fused_only_in_rounding():
    """bf16: per-hop rounding changes bits somewhere, within (p-1) roundings."""
    p, n = 8, 8 * 4096
    xs = gen("bf16", "sum", p, n, seed=120)
    step, _ = run_collective(xs, "ar", "sum", "bf16", "ring", variant="ring_stepwise")
    fused, _ = run_collective(xs, "ar", "sum", "bf16", "ring", variant="ldst")
    a = torch.from_numpy(step.host(0).view(np.int16).copy()).view(torch.bfloat16).double()
    b = torch.from_numpy(fused.host(0).view(np.int16).copy()).view(torch.bfloat16).double()
    assert not torch.equal(a, b)
    absum = sum(torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).double().abs() for x in xs)
    assert bool(((a - b).abs() <= 2 * p * 2.0 ** -8 * absum).all())


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "max", "avg"])
@pytest.mark.parametrize("sched", ["ring", "allpairs"])
def test_one_phase_matches_fused_oracle(dtype, op, sched):
    s = inputs.ELEM_BYTES[dtype]
    for p in (1, 2, 5, 8, 16):
        for n in (p * (16 // s) * 700, p * 333 + 1):
            xs = gen(dtype, op, p, n, seed=130 + p)
            res, desc = run_collective(xs, "ar", op, dtype, sched, variant="one_phase")
            assert "allreduce_one_phase" in desc
            want = oracle.allreduce(xs, op, dtype, sched)
            for r in range(p):
                assert bits_equal(res.host(r), want[r]), (p, n, r)


def test_comparison_executor_statuses():
    xs = gen("f32", "sum", 4, 4 * 64, seed=140)
    for variant, coll, sched, inplace in (("ring_stepwise", "ar", "allpairs", False),
                                          ("ring_stepwise", "rs", "ring", False),
                                          ("one_phase", "ag", "ring", False),
                                          ("one_phase", "ar", "ring", True)):
        with pytest.raises(ccl.CclError) as ei:
            run_collective(xs, coll, "sum", "f32", sched, variant=variant, inplace=inplace)
        assert ei.value.status == ccl.CCL_ERR_UNSUPPORTED, (variant, coll)
