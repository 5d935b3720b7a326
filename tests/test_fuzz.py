"""Seeded random cases across the whole launch surface, checked bit for bit
against the oracle: rank count, element type, op, collective, schedule,
variant, SM budget, message size (ragged chunks and tails included), in
place or out of place, and misaligned pointers.  Each case is small enough
for the oracle to finish at once; the draw is fixed by the seed, so a
failure names a reproducible case."""
import numpy as np
import pytest
import torch

import oracle
from reducescatter_reduction_gb300 import inputs
from ccl_testutil import bits_equal, ensure_built
from test_parity import gen, run_collective

pytestmark = pytest.mark.gpu

DTYPES = ["f32", "f16", "bf16", "i32"]
OPS = ["sum", "prod", "min", "max", "avg"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ensure_built()


def draw(rng):
    """One valid case.  The TMA variant needs 16-byte aligned pointers and
    chunk boundaries and has no AllGather; the comparison executors run
    AllReduce only, and the one-phase executor out of place only."""
    p = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 9, 16, 17, 31, 64], p=[.04, .12, .08, .1, .06, .06, .16, .06, .12, .06, .06, .08]))
    dtype = str(rng.choice(DTYPES))
    op = str(rng.choice(OPS))
    s = inputs.ELEM_BYTES[dtype]
    per16 = 16 // s
    variant = str(rng.choice(["ldst", "ldst", "tma", "auto", "ring_stepwise", "one_phase"]))
    if variant in ("ring_stepwise", "one_phase"):
        coll = "ar"
    elif variant == "tma":
        coll = str(rng.choice(["ar", "ar", "rs"]))         # AllGather has no TMA variant
    else:
        coll = str(rng.choice(["ar", "ar", "rs", "ag"]))
    sched = "ring" if variant == "ring_stepwise" else str(rng.choice(["ring", "allpairs"]))
    budget = int(rng.choice([0, 0, 1, 2, 5, 16]))
    if variant == "tma":
        n = p * per16 * int(rng.integers(1, 2500))
        offset = 0
    else:
        per_rank = int(rng.integers(0, 40000))
        n = p * per_rank if coll != "ar" else per_rank * p + int(rng.integers(0, p))
        offset = int(rng.choice([0, 0, 0, s]))
    inplace = bool(rng.integers(0, 2)) and variant != "one_phase" and coll != "rs"
    if coll == "ag":
        op = "sum"                      # ignored by AllGather; keeps gen() simple
    return dict(p=p, dtype=dtype, op=op, coll=coll, sched=sched, variant=variant, budget=budget, n=n,
                offset=offset, inplace=inplace)


def expected(case, xs):
    op, dtype, sched = case["op"], case["dtype"], case["sched"]
    if case["coll"] == "ag":
        return oracle.all_gather(xs, dtype)
    if case["coll"] == "rs":
        return oracle.reduce_scatter(xs, op, dtype, sched)
    if case["variant"] == "ring_stepwise":
        return oracle.allreduce_ring_stepwise(xs, op, dtype)
    return oracle.allreduce(xs, op, dtype, sched)


@pytest.mark.parametrize("seed", range(16))
def test_random_cases_match_oracle(seed):
    rng = np.random.default_rng([2024, seed])
    for k in range(16):
        case = draw(rng)
        xs = gen(case["dtype"], case["op"], case["p"], case["n"], seed=1000 * seed + k)
        if case["n"] == 0:
            xs = [np.zeros(0, dtype=x.dtype) for x in xs]
        res, desc = run_collective(xs, case["coll"], case["op"], case["dtype"], case["sched"],
                                   inplace=case["inplace"], offset=case["offset"], budget=case["budget"],
                                   variant=case["variant"], n=case["n"])
        if case["n"] == 0:
            continue
        want = expected(case, xs)
        for r in range(case["p"]):
            assert bits_equal(res.host(r), want[r]), (case, r, desc)
