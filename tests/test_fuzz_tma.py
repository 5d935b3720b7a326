"""Seeded random cases through the TMA kernels, checked bit for bit against
the oracle on order-revealing inputs: the narrow kernel (a tile of every rank
per stage, p <= 13) and the wide one (ranks through the stages eight or four
at a time), explicit tile sizes (some refused as too large for the shared
memory, which must fail cleanly), SM budgets on both sides of the small-grid
threshold (32), rank counts on both sides of the narrow/wide switch (13/14)
and of 32/33, AllReduce in and out of place and ReduceScatter."""
import numpy as np
import pytest
import torch

import oracle
import reducescatter_reduction_gb300 as ccl
from reducescatter_reduction_gb300 import inputs
from ccl_testutil import Comm, RankBuffers, bits_equal, ensure_built, stream_ptr
from test_parity import gen

pytestmark = pytest.mark.gpu

PS = [2, 3, 4, 5, 6, 7, 8, 9, 12, 13, 14, 15, 16, 17, 20, 24, 31, 32, 33, 40, 48, 63, 64]
BUDGETS = [0, 0, 1, 2, 3, 5, 8, 16, 31, 32, 33, 76]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ensure_built()


def draw(rng):
    p = int(rng.choice(PS))
    dtype = str(rng.choice(["f32", "f16", "bf16", "i32"]))
    op = str(rng.choice(["sum", "prod", "min", "max", "avg"]))
    coll = str(rng.choice(["ar", "ar", "rs"]))
    sched = str(rng.choice(["ring", "allpairs"]))
    budget = int(rng.choice(BUDGETS))
    tile = 0
    if rng.random() < 0.4:
        tile = int(rng.integers(1, 33)) * 1024
        if rng.random() < 0.3:
            tile -= 16 * int(rng.integers(1, 4))          # multiples of 16 that are not of 1 KiB
    per16 = 16 // inputs.ELEM_BYTES[dtype]
    n = p * per16 * int(rng.integers(1, 2500))
    inplace = coll == "ar" and bool(rng.integers(0, 2))
    return dict(p=p, dtype=dtype, op=op, coll=coll, sched=sched, budget=budget, tile=tile, n=n, inplace=inplace)


def rank_inputs(case, seed):
    p, n, dtype, op = case["p"], case["n"], case["dtype"], case["op"]
    if dtype != "i32" and op in ("sum", "avg"):
        return [inputs.cancel(n, seed, r, p, dtype) for r in range(p)]
    if dtype != "i32" and op == "prod":
        return [inputs.prod_inexact(n, seed, r, dtype) for r in range(p)]
    if dtype != "i32":
        return [inputs.signed_zero(n, r, p, dtype) for r in range(p)]
    return gen(dtype, op, p, n, seed=seed)


@pytest.mark.parametrize("seed", range(8))
def test_random_tma_cases_match_oracle(seed):
    rng = np.random.default_rng([4242, seed])
    for k in range(12):
        case = draw(rng)
        p, n, dtype, op, coll, sched = (case[key] for key in ("p", "n", "dtype", "op", "coll", "sched"))
        xs = rank_inputs(case, 7000 + 100 * seed + k)
        storage = inputs.STORAGE[dtype]
        ins = RankBuffers(xs, n, storage)
        outs = None if case["inplace"] else RankBuffers(None, n // p if coll == "rs" else n, storage, p=p)
        with Comm(ins, outs) as cm:
            ccl.ccl_set_launch(cm.h, case["budget"], "tma", case["tile"])
            try:
                if coll == "ar":
                    ccl.ccl_allreduce(cm.h, op, dtype, n, sched, stream_ptr())
                else:
                    ccl.ccl_reduce_scatter(cm.h, op, dtype, n, sched, stream_ptr())
            except ccl.CclError as e:
                # only an explicit tile whose stages do not fit may be refused, and nothing runs
                assert case["tile"] and e.status == ccl.CCL_ERR_INVALID_ARG, (case, e)
                continue
            torch.cuda.synchronize()
            ccl.ccl_comm_check(cm.h)
            desc = ccl.ccl_comm_last_launch(cm.h)
        assert "_tma" in desc, (case, desc)
        res = ins if case["inplace"] else outs
        want = oracle.allreduce(xs, op, dtype, sched) if coll == "ar" else oracle.reduce_scatter(xs, op, dtype, sched)
        for r in range(p):
            assert bits_equal(res.host(r), want[r]), (case, r, desc)
        assert ins.guards_intact() and (outs is None or outs.guards_intact())
