"""GPU parity on inputs whose bits depend on the rank order and on where the
result is rounded, through every kernel instantiation.

On N(0,1) inputs the fp32 sum of p <= 16 bf16 or fp16 values is almost always
exact, so a kernel that folded a chunk in the wrong rank order would still
match the oracle there.  These tests use the order-revealing recipes of
``inputs`` (``cancel`` for sum and avg, ``signed_zero`` for the first rank of
min and max, ``prod_inexact`` and ``prod_overflow`` for prod); the CPU tests in
test_probe_inputs.py show, by planting wrong orders and per-hop rounding in
the oracle, that each of those mistakes changes the bits on these inputs.

Every fixed-order path is compared with the oracle bit for bit, under the
ring, all-pairs and explicit (custom table) schedules: the ld/st kernel for
the p-specialised instantiations (p = 2, 3, 4, 8, 16), the generic one
(5, 6, 13, 17, 33, 64) and its other register shapes (fp32 at p = 5/6, fp16/bf16
min/max at p = 8), the SM-budget persistent kernel (with and without its
work counter), the TMA kernel (narrow, and wide from 14 ranks; static split
and tile counter), ReduceScatter through each, the allocation-free entry
point, the one-phase executor, the stepwise ring (against its own oracle)
and the fused residual + RMSNorm (its merged residual h).  The ring's order
is the one "Inside NCCL AllReduce" prints in "The ring, exactly as the kernel
runs it"; all-pairs folds rank 0 first ("MSCCL, in depth").
"""
import math

import numpy as np
import pytest
import torch

import oracle
import reducescatter_reduction_gb300 as ccl
from reducescatter_reduction_gb300 import inputs
from ccl_testutil import Comm, RankBuffers, bits_equal, ensure_built, sample_indices, stream_ptr

pytestmark = pytest.mark.gpu

FLOATS = ["f32", "f16", "bf16"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ensure_built()


# ---------------------------------------------------------------------------
# sizes and inputs
# ---------------------------------------------------------------------------

WIDE_FROM = 14          # the TMA kernel brings the ranks through its stages eight at a time from here


def tile_elems(p, dtype):
    """Elements per TMA tile at the library's largest default tile for p (the
    one a small SM budget takes; on every SM the tile is the same or half)."""
    s = inputs.ELEM_BYTES[dtype]
    t = 24576 if p <= 3 else 12288 if p <= 6 else 16384 if p >= WIDE_FROM else 8192
    return t // s


def chunk_len(p, dtype):
    """Elements per chunk: several TMA tiles plus a short last one (chunks stay
    16-byte multiples), and at least 66 tiles in all, so that a one-SM budget
    turns on the TMA tile counter."""
    tiles = max(2 if p >= WIDE_FROM else 3, math.ceil(66 / p))
    return tiles * tile_elems(p, dtype) + 24


def recipe(kind, p, n, dtype, seed):
    if kind == "cancel":
        return [inputs.cancel(n, seed, r, p, dtype) for r in range(p)]
    if kind == "zero":
        return [inputs.signed_zero(n, r, p, dtype) for r in range(p)]
    if kind == "prod_inexact":
        return [inputs.prod_inexact(n, seed, r, dtype) for r in range(p)]
    if kind == "prod_overflow":
        return [inputs.prod_overflow(n, seed, r, p, dtype) for r in range(p)]
    raise ValueError(kind)


def table_for(p, sched):
    if sched == "custom":
        rng = np.random.default_rng(500 + p)
        return [list(int(v) for v in rng.permutation(p)) for _ in range(p)]
    return [oracle.chunk_order(p, sched, c) for c in range(p)]


# ---------------------------------------------------------------------------
# one call through the C ABI
# ---------------------------------------------------------------------------

def run(xs, coll, op, dtype, sched, table, variant="ldst", budget=0, n=None):
    """Runs one collective on fresh device buffers; returns (outputs, launch description)."""
    p = len(xs)
    n = xs[0].size if n is None else n
    storage = inputs.STORAGE[dtype]
    ins = RankBuffers(xs, n, storage)
    out_n = n // p if coll == "rs" else n
    outs = RankBuffers(None, out_n, storage, p=p)
    if variant == "static":
        ccl.ccl_allreduce_static(p, ins.ptrs(), outs.ptrs(), op, dtype, n, sched, stream_ptr())
        torch.cuda.synchronize()
        desc = "static"
    else:
        with Comm(ins, outs) as cm:
            ccl.ccl_set_launch(cm.h, budget, variant, 0)
            if sched == "custom":
                ccl.ccl_comm_set_schedule(cm.h, table)
            if coll == "ar":
                ccl.ccl_allreduce(cm.h, op, dtype, n, sched, stream_ptr())
            else:
                ccl.ccl_reduce_scatter(cm.h, op, dtype, n, sched, stream_ptr())
            torch.cuda.synchronize()
            ccl.ccl_comm_check(cm.h)
            desc = ccl.ccl_comm_last_launch(cm.h)
    assert ins.guards_intact() and outs.guards_intact(), "write outside the buffers"
    return outs, desc


def check_ar(outs, want, p):
    assert bits_equal(outs.host(0), want[0])
    assert outs.identical_across_ranks()


def check_rs(outs, want_ar, p, n):
    for r in range(p):
        b, e = oracle.chunk_bounds(p, n, r)
        assert bits_equal(outs.host(r), want_ar[0][b:e]), f"rank {r}"


def budget_threads(p):
    return 1024 if p in (2, 3, 4, 8) else 512


PATHS_AR = ["ldst", "ldst_budget", "tma", "tma_budget", "static", "one_phase"]


def run_paths(xs, op, dtype, sched, table, paths=PATHS_AR, rs=True):
    """Every AllReduce path in ``paths`` (and ReduceScatter through the ld/st
    and TMA kernels) against one oracle result."""
    p, n = len(xs), xs[0].size
    want = oracle.allreduce_orders(xs, op, dtype, table)
    for path in paths:
        if path == "static" and sched == "custom":
            continue
        variant = {"ldst_budget": "ldst", "tma_budget": "tma"}.get(path, path)
        budget = 1 if path.endswith("_budget") else 0
        outs, desc = run(xs, "ar", op, dtype, sched, table, variant=variant, budget=budget)
        if path == "ldst":
            assert "allreduce_ldst" in desc and "vec=1" in desc, desc
        elif path == "ldst_budget":
            assert "allreduce_ldst" in desc and f"block={budget_threads(p)}" in desc and "grid=1 " in desc, desc
        elif path.startswith("tma"):
            assert "allreduce_tma" in desc, desc
            if path == "tma_budget":
                assert "counter=1" in desc, desc
        try:
            check_ar(outs, want, p)
        except AssertionError as e:
            raise AssertionError(f"{path}: {desc}") from e
    if rs:
        for variant in ("ldst", "tma"):
            outs, desc = run(xs, "rs", op, dtype, sched, table, variant=variant)
            assert "reduce_scatter" in desc, desc
            try:
                check_rs(outs, want, p, n)
            except AssertionError as e:
                raise AssertionError(f"reduce_scatter {variant}: {desc}") from e


P_ALL = [2, 3, 4, 5, 6, 8, 13, 16, 17, 33, 64]


# ---------------------------------------------------------------------------
# sum and avg: the cancelling pair
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("p", P_ALL)
@pytest.mark.parametrize("dtype", FLOATS)
@pytest.mark.parametrize("sched", ["ring", "allpairs", "custom"])
def test_sum_order_every_path(p, dtype, sched):
    n = p * chunk_len(p, dtype)
    xs = recipe("cancel", p, n, dtype, seed=100 + p)
    run_paths(xs, "sum", dtype, sched, table_for(p, sched))


@pytest.mark.parametrize("p", [3, 5, 6, 8, 16, 33])
@pytest.mark.parametrize("dtype", FLOATS)
@pytest.mark.parametrize("sched", ["ring", "allpairs"])
def test_avg_order_every_path(p, dtype, sched):
    n = p * chunk_len(p, dtype)
    xs = recipe("cancel", p, n, dtype, seed=200 + p)
    run_paths(xs, "avg", dtype, sched, table_for(p, sched))


@pytest.mark.parametrize("p", [3, 8, 17])
@pytest.mark.parametrize("dtype", FLOATS)
def test_sum_order_ragged_chunks(p, dtype):
    """Chunks that are not 16-byte multiples: groups straddling a chunk
    boundary are folded element by element, each in its own chunk's order."""
    n = p * 3000 + p // 2 + 1
    xs = recipe("cancel", p, n, dtype, seed=300 + p)
    for sched in ("ring", "allpairs"):
        want = oracle.allreduce_orders(xs, "sum", dtype, table_for(p, sched))
        for budget in (0, 1):
            outs, desc = run(xs, "ar", "sum", dtype, sched, None, variant="ldst", budget=budget)
            check_ar(outs, want, p)


# ---------------------------------------------------------------------------
# min and max: the first rank of every chunk's order
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("p", P_ALL)
@pytest.mark.parametrize("dtype", FLOATS)
@pytest.mark.parametrize("op", ["min", "max"])
def test_first_rank_every_path(p, dtype, op):
    n = p * chunk_len(p, dtype)
    xs = recipe("zero", p, n, dtype, seed=0)
    for sched in ("ring", "allpairs", "custom"):
        run_paths(xs, op, dtype, sched, table_for(p, sched), rs=(sched != "allpairs"))


# ---------------------------------------------------------------------------
# prod: rounding of the partial product, and the order through fp32 overflow
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("p", [2, 3, 4, 5, 8, 16, 17, 64])
@pytest.mark.parametrize("dtype", FLOATS)
def test_prod_inexact_every_path(p, dtype):
    n = p * chunk_len(p, dtype)
    xs = recipe("prod_inexact", p, n, dtype, seed=400 + p)
    for sched in ("ring", "custom"):
        run_paths(xs, "prod", dtype, sched, table_for(p, sched), rs=(sched == "ring"))


@pytest.mark.parametrize("p", [3, 5, 8, 16, 33])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("sched", ["ring", "allpairs", "custom"])
def test_prod_overflow_order_every_path(p, dtype, sched):
    n = p * max(chunk_len(p, dtype), 8192)
    xs = recipe("prod_overflow", p, n, dtype, seed=500 + p)
    run_paths(xs, "prod", dtype, sched, table_for(p, sched), rs=False)


# ---------------------------------------------------------------------------
# the budget kernel's work counter, the TMA tile counter on the whole GPU,
# and the benchmark's own size (sampled)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("p", [2, 3, 8, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_budget_work_counter_keeps_the_order(p, dtype):
    """Large enough that the one-SM persistent kernel's warps take blocks from
    the work counter."""
    groups = (1 << 18) if budget_threads(p) == 1024 else (1 << 17)
    n = p * (groups * (16 // inputs.ELEM_BYTES[dtype]) // p + 64)
    xs = recipe("cancel", p, n, dtype, seed=600 + p)
    want = oracle.allreduce(xs, "sum", dtype, "ring")
    outs, desc = run(xs, "ar", "sum", dtype, "ring", None, variant="ldst", budget=1)
    assert "counter=1" in desc, desc
    check_ar(outs, want, p)
    outs, desc = run(xs, "rs", "sum", dtype, "ring", None, variant="ldst", budget=1)
    check_rs(outs, want, p, n)


def test_benchmark_size_order_sampled():
    """p=8 bf16 at 128 MiB per rank, both kernels on every SM (the TMA kernel
    with its tile counter), cancel inputs, sampled against the oracle."""
    p, dtype, n = 8, "bf16", 1 << 26
    xs = inputs.cancel_ranks(n, 700, p, dtype)
    idx = sample_indices(p, n, count=200000, seed=7)
    for sched in ("ring", "allpairs"):
        want = oracle.allreduce_at(xs, idx, "sum", dtype, sched)
        for variant in ("ldst", "tma"):
            outs, desc = run(xs, "ar", "sum", dtype, sched, None, variant=variant)
            if variant == "tma":
                assert "counter=1" in desc, desc
            for r in (0, 3, 7):
                assert bits_equal(outs.at(r, idx), want), (sched, variant, r)
        other = oracle.allreduce_at(xs, idx, "sum", dtype, "allpairs" if sched == "ring" else "ring")
        assert np.mean(want != other) > 0.3          # the inputs do reveal the order at this size


# ---------------------------------------------------------------------------
# comparison executors and the fused epilogue
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("p", [3, 8, 16])
@pytest.mark.parametrize("dtype", FLOATS)
@pytest.mark.parametrize("kind,op", [("cancel", "sum"), ("prod_inexact", "prod"), ("cancel", "avg")])
def test_stepwise_ring_against_its_oracle(p, dtype, kind, op):
    n = p * 2048 + 8 * p
    xs = recipe(kind, p, n, dtype, seed=800 + p)
    want = oracle.allreduce_ring_stepwise(xs, op, dtype)
    outs, desc = run(xs, "ar", op, dtype, "ring", None, variant="ring_stepwise")
    assert "ring_stepwise" in desc
    check_ar(outs, want, p)


def _ulp(vals, dtype):
    mant = {"f32": 23, "f16": 10, "bf16": 7}[dtype]
    tiny = {"f32": 2.0 ** -126, "f16": 2.0 ** -14, "bf16": 2.0 ** -126}[dtype]
    return 2.0 ** (np.floor(np.log2(np.maximum(np.abs(vals), tiny))) - mant)


def _decode(arr, dtype):
    if dtype == "f32":
        return arr.astype(np.float64)
    if dtype == "f16":
        return arr.view(np.float16).astype(np.float64)
    return torch.from_numpy(arr.view(np.int16).copy()).view(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("p", [3, 8, 16])
@pytest.mark.parametrize("dtype", FLOATS)
@pytest.mark.parametrize("rows", [1, 160, 320])
def test_fused_rmsnorm_merge_keeps_the_order(p, dtype, rows):
    """The merged residual h = round(y + residual) carries the AllReduce's
    bits; with the cancel inputs it depends on every position of the order.
    rows 1 / 160 / 320 take the cluster, 1024-thread and 256-thread shapes."""
    hidden = 1024
    n = rows * hidden
    xs = recipe("cancel", p, n, dtype, seed=900 + p)
    res = inputs.normal(n, 901, 0, 0.5, dtype)
    gamma = inputs.normal(hidden, 902, 0, 1.0, dtype)
    storage = inputs.STORAGE[dtype]
    for sched in ("ring", "allpairs"):
        want_out, want_h = oracle.allreduce_residual_rmsnorm(xs, res, gamma, rows, hidden, dtype, sched, 1e-6)
        ins = RankBuffers(xs, n, storage)
        outs = RankBuffers(None, n, storage, p=p)
        r_in = RankBuffers([res], n, storage)
        r_out = RankBuffers(None, n, storage, p=1)
        g = RankBuffers([gamma], hidden, storage)
        with Comm(ins, outs) as cm:
            ccl.ccl_allreduce_residual_rmsnorm(cm.h, dtype, rows, hidden, r_in.ptr(0), r_out.ptr(0), g.ptr(0),
                                               1e-6, sched, stream_ptr())
            torch.cuda.synchronize()
        assert bits_equal(r_out.host(0), want_h), sched
        got, want = _decode(outs.host(0), dtype), _decode(want_out, dtype)
        if dtype == "f32":
            assert np.all(np.abs(got - want) <= 1e-5 * np.abs(want) + 1e-30)
        else:
            assert np.all(np.abs(got - want) <= _ulp(want, dtype))
        assert outs.identical_across_ranks()
        for b in (ins, outs, r_in, r_out, g):
            assert b.guards_intact()
