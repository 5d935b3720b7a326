"""GPU tests of the TMA variant (bulk copies through shared-memory stages):
bit-identical to the oracle in every op/dtype/schedule, independent of the
tile size and the SM budget, explicit statuses for layouts it cannot take,
and the bounded-wait timeout path (without faulting or hanging the GPU)."""
import numpy as np
import pytest
import torch

import oracle
import reducescatter_reduction_gb300 as ccl
from reducescatter_reduction_gb300 import inputs
from ccl_testutil import Comm, RankBuffers, bits_equal, ensure_built, stream_ptr
from test_parity import gen, run_collective

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ensure_built()


def tma_sizes(p, dtype):
    """Chunk sizes that are multiples of 16 bytes and make several tiles per
    chunk with a short last tile (16 bytes past a whole number of tiles)."""
    s = inputs.ELEM_BYTES[dtype]
    per16 = 16 // s
    return [p * per16, p * (3 * 8192 // s + per16), p * (64 * 1024 // s + 5 * per16)]


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "prod", "min", "max", "avg"])
@pytest.mark.parametrize("sched", ["ring", "allpairs"])
def test_tma_allreduce_matches_oracle(dtype, op, sched):
    for p in (2, 3, 8, 16):
        for n in tma_sizes(p, dtype):
            xs = gen(dtype, op, p, n, seed=31 + p)
            res, desc = run_collective(xs, "ar", op, dtype, sched, variant="tma")
            assert "allreduce_tma" in desc and "variant=tma" in desc
            want = oracle.allreduce(xs, op, dtype, sched)
            for r in range(p):
                assert bits_equal(res.host(r), want[r]), (p, n, r)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "max", "avg"])
def test_tma_reduce_scatter_matches_oracle(dtype, op):
    for p in (2, 5, 8, 16):
        n = tma_sizes(p, dtype)[1]
        xs = gen(dtype, op, p, n, seed=37)
        res, desc = run_collective(xs, "rs", op, dtype, "ring", variant="tma")
        assert "reduce_scatter_tma" in desc
        want = oracle.reduce_scatter(xs, op, dtype, "ring")
        for r in range(p):
            assert bits_equal(res.host(r), want[r]), (p, r)


@pytest.mark.parametrize("p", [8, 16])
def test_tma_in_place_and_budgets_equal_ldst(p):
    """In place, at SM budgets 1, 4, 16 and all, and at several tile sizes,
    the TMA variant gives the ld/st kernel's bits."""
    n = p * (1 << 20)
    xs = gen("bf16", "sum", p, n, seed=41)
    ref, _ = run_collective(xs, "ar", "sum", "bf16", "ring", variant="ldst")
    for budget, tile in ((0, 0), (1, 0), (4, 2048), (16, 4096), (0, 1024)):
        storage = inputs.STORAGE["bf16"]
        ins = RankBuffers(xs, n, storage)
        with Comm(ins) as cm:                      # in place
            ccl.ccl_set_launch(cm.h, budget, "tma", tile)
            ccl.ccl_allreduce(cm.h, "sum", "bf16", n, "ring", stream_ptr())
            torch.cuda.synchronize()
            desc = ccl.ccl_comm_last_launch(cm.h)
            ccl.ccl_comm_check(cm.h)
        grid = int(desc.split("grid=")[1].split()[0])
        if budget:
            assert grid <= budget
        for r in range(p):
            assert torch.equal(ins.views[r], ref.views[0]), (budget, tile, r)
        assert ins.guards_intact()


@pytest.mark.parametrize("p", [8, 16])
def test_tma_tile_counter_starts_at_zero_for_every_launch(p):
    """On messages with many tiles per CTA the TMA kernel hands out tiles
    from a counter in the communicator's status block, and the last CTA of a
    launch returns it to zero.  Four launches in a row on one stream (counter
    on 3 SMs, on 2 SMs, the static split on every SM, the counter on 3 SMs
    again), each after its outputs were zeroed on the same stream and with no
    host synchronisation in between: a launch that started from a stale
    counter would leave zero tiles behind.  p = 16 runs the wide kernel,
    which on these small grids takes four tiles per visit and asks for its
    next grab ahead (one grab per CTA is never taken)."""
    n = p * (3 * 8192 + 40)                        # ragged last tile in every chunk
    xs = gen("f32", "sum", p, n, seed=47)
    ref, _ = run_collective(xs, "ar", "sum", "f32", "ring", variant="ldst")
    ins = RankBuffers(xs, n, np.float32)
    outs = RankBuffers(None, n, np.float32, p=p)
    with Comm(ins, outs) as cm:
        for budget, tile in ((3, 2048), (2, 1024), (0, 0), (3, 2048)):
            for v in outs.views:
                v.zero_()
            ccl.ccl_set_launch(cm.h, budget, "tma", tile)
            ccl.ccl_allreduce(cm.h, "sum", "f32", n, "ring", stream_ptr())
            if budget:
                assert "counter=1" in ccl.ccl_comm_last_launch(cm.h)
        torch.cuda.synchronize()
        ccl.ccl_comm_check(cm.h)
    for r in range(p):
        assert torch.equal(outs.views[r], ref.views[0]), r
    assert outs.guards_intact()


@pytest.mark.parametrize("dtype,op", [("bf16", "sum"), ("f32", "avg"), ("i32", "prod"), ("f16", "max")])
def test_tma_wide_ranks_match_oracle(dtype, op):
    """From 14 ranks: the wide kernel brings a tile's ranks through the
    stages eight at a time and keeps the partial in registers across them;
    bits equal the oracle for AllReduce and ReduceScatter, with a short last
    tile, a last batch of fewer than eight ranks, several tile sizes and SM
    budgets."""
    s = inputs.ELEM_BYTES[dtype]
    per16 = 16 // s
    # four ranks of a 16 KB tile per stage: the default on small grids (budgets 2 and 7), forced on every SM by
    # the tile size (40, 16384, 0), and a 12 KB tile (24, 12288, 5); eight ranks of 8 KB or less otherwise
    for p, tile, budget in ((14, 0, 0), (16, 0, 2), (24, 4096, 0), (24, 12288, 5), (33, 0, 0), (40, 4096, 3),
                            (40, 16384, 0), (64, 1024, 0), (64, 0, 7)):
        n = p * (3 * 8192 // s + 5 * per16)
        xs = gen(dtype, op, p, n, seed=150 + p)
        storage = inputs.STORAGE[dtype]
        ins = RankBuffers(xs, n, storage)
        outs = RankBuffers(None, n, storage, p=p)
        with Comm(ins, outs) as cm:
            ccl.ccl_set_launch(cm.h, budget, "tma", tile)
            ccl.ccl_allreduce(cm.h, op, dtype, n, "ring", stream_ptr())
            torch.cuda.synchronize()
            desc = ccl.ccl_comm_last_launch(cm.h)
            ccl.ccl_comm_check(cm.h)
        assert "allreduce_tma_wide" in desc, desc
        if budget:
            assert int(desc.split("grid=")[1].split()[0]) <= budget
        want = oracle.allreduce(xs, op, dtype, "ring")
        for r in range(p):
            assert bits_equal(outs.host(r), want[r]), (p, tile, budget, r)
        assert ins.guards_intact() and outs.guards_intact()
        rs, desc = run_collective(xs, "rs", op, dtype, "allpairs", variant="tma")
        assert "reduce_scatter_tma_wide" in desc
        want = oracle.reduce_scatter(xs, op, dtype, "allpairs")
        for r in range(p):
            assert bits_equal(rs.host(r), want[r]), (p, r)


def test_tma_wide_bounded_wait_times_out_and_context_survives():
    p, n = 40, 40 * (1 << 13)
    xs = gen("bf16", "sum", p, n, seed=160)
    storage = inputs.STORAGE["bf16"]
    ins = RankBuffers(xs, n, storage)
    outs = RankBuffers(None, n, storage, p=p)
    with Comm(ins, outs) as cm:
        ccl.ccl_set_launch(cm.h, 1, "tma", 2048)
        ccl.ccl_comm_set_debug(cm.h, 20_000_000, 1)
        ccl.ccl_allreduce(cm.h, "sum", "bf16", n, "ring", stream_ptr())
        with pytest.raises(ccl.CclError) as ei:
            ccl.ccl_comm_check(cm.h)
        assert ei.value.status == ccl.CCL_ERR_TIMEOUT
        ccl.ccl_comm_set_debug(cm.h, 0, 0)
        ccl.ccl_allreduce(cm.h, "sum", "bf16", n, "ring", stream_ptr())
        ccl.ccl_comm_check(cm.h)
    want = oracle.allreduce(xs, "sum", "bf16", "ring")
    for r in range(p):
        assert bits_equal(outs.host(r), want[r])


def test_tma_statuses():
    p = 4
    xs = gen("bf16", "sum", p, 4 * 1001, seed=43)          # chunk 1001 elements: not 16-byte aligned
    ins = RankBuffers(xs, xs[0].size, np.uint16)
    outs = RankBuffers(None, xs[0].size, np.uint16, p=p)
    with Comm(ins, outs) as cm:
        ccl.ccl_set_launch(cm.h, 0, "tma", 0)
        with pytest.raises(ccl.CclError) as ei:
            ccl.ccl_allreduce(cm.h, "sum", "bf16", xs[0].size, "ring", stream_ptr())
        assert ei.value.status == ccl.CCL_ERR_UNSUPPORTED
        with pytest.raises(ccl.CclError) as ei:
            ccl.ccl_all_gather(cm.h, "bf16", xs[0].size - 4, stream_ptr())
        assert ei.value.status == ccl.CCL_ERR_UNSUPPORTED
        ccl.ccl_set_launch(cm.h, 0, "tma_bulkred", 0)
        with pytest.raises(ccl.CclError) as ei:                   # a product has no bulk reduction
            ccl.ccl_allreduce(cm.h, "prod", "bf16", 4 * 1000, "ring", stream_ptr())
        assert ei.value.status == ccl.CCL_ERR_UNSUPPORTED
    p = 64
    xs = gen("bf16", "sum", p, p * 64, seed=44)
    ins = RankBuffers(xs, xs[0].size, np.uint16)
    with Comm(ins) as cm:
        ccl.ccl_set_launch(cm.h, 0, "tma", 32768)                # 65 tiles of 32 KiB cannot fit twice
        with pytest.raises(ccl.CclError) as ei:
            ccl.ccl_allreduce(cm.h, "sum", "bf16", xs[0].size, "ring", stream_ptr())
        assert ei.value.status == ccl.CCL_ERR_INVALID_ARG
    torch.cuda.synchronize()


@pytest.mark.parametrize("p,budget,tile", [(8, 1, 4096), (16, 1, 4096), (8, 0, 0), (5, 3, 0), (16, 0, 0)])
def test_tma_bounded_wait_times_out_and_context_survives(p, budget, tile):
    """The producer withholds a tile (a wait nothing will satisfy); the
    consumers' wait gives up after 20 ms, the kernel records it and returns,
    ccl_comm_check reports CCL_ERR_TIMEOUT once, and the same communicator
    then runs correctly.  p = 5 and 8 run the narrow kernel (a tile of every
    rank per stage), p = 16 the wide one (eight ranks per stage); one CTA or
    many."""
    n = p * (1 << 16)
    xs = gen("bf16", "sum", p, n, seed=45)
    storage = inputs.STORAGE["bf16"]
    ins = RankBuffers(xs, n, storage)
    outs = RankBuffers(None, n, storage, p=p)
    with Comm(ins, outs) as cm:
        ccl.ccl_set_launch(cm.h, budget, "tma", tile)
        ccl.ccl_comm_set_debug(cm.h, 20_000_000, 1)
        ccl.ccl_allreduce(cm.h, "sum", "bf16", n, "ring", stream_ptr())
        with pytest.raises(ccl.CclError) as ei:
            ccl.ccl_comm_check(cm.h)
        assert ei.value.status == ccl.CCL_ERR_TIMEOUT
        assert "gave up" in str(ei.value)
        ccl.ccl_comm_check(cm.h)                                 # reported once, then cleared
        ccl.ccl_comm_set_debug(cm.h, 0, 0)
        ccl.ccl_allreduce(cm.h, "sum", "bf16", n, "ring", stream_ptr())
        ccl.ccl_comm_check(cm.h)
    want = oracle.allreduce(xs, "sum", "bf16", "ring")
    for r in range(p):
        assert bits_equal(outs.host(r), want[r])
    assert ins.guards_intact() and outs.guards_intact()


def test_debug_hook_arguments():
    xs = gen("f32", "sum", 2, 64, seed=46)
    ins = RankBuffers(xs, 64, np.float32)
    with Comm(ins) as cm:
        for bad in ((-1, 0), (0, 3), (0, -1)):
            with pytest.raises(ccl.CclError) as ei:
                ccl.ccl_comm_set_debug(cm.h, *bad)
            assert ei.value.status == ccl.CCL_ERR_INVALID_ARG


# ---------------------------------------------------------------------------
# bulk-reduce variant: reductions applied by the memory system
# ---------------------------------------------------------------------------

EPS_OUT = {"f32": 2.0 ** -23, "f16": 2.0 ** -10, "bf16": 2.0 ** -7}


def decode(arr, dtype):
    if dtype == "f32":
        return arr.astype(np.float64)
    if dtype == "f16":
        return arr.view(np.float16).astype(np.float64)
    return torch.from_numpy(arr.view(np.int16).copy()).view(torch.bfloat16).double().numpy()


def within_reassociation_bound(got, xs, dtype):
    """|y - exact| <= 2 p eps_out sum_k |x_k| per element (exact in fp64)."""
    p = len(xs)
    xf = np.stack([decode(x, dtype) for x in xs])
    exact = xf.sum(axis=0)
    bound = 2 * p * EPS_OUT[dtype] * np.abs(xf).sum(axis=0)
    err = np.abs(decode(got, dtype) - exact)
    return bool(np.all(err <= bound)), float(np.max(err / np.maximum(bound, 1e-300)))


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("p", [2, 8, 16])
def test_bulkred_allreduce_sum_within_bound(dtype, p):
    n = tma_sizes(p, dtype)[2]
    xs = gen(dtype, "sum", p, n, seed=80 + p)
    res, desc = run_collective(xs, "ar", "sum", dtype, "ring", variant="tma_bulkred")
    assert "allreduce_tma_bulkred" in desc
    ok, worst = within_reassociation_bound(res.host(0), xs, dtype)
    assert ok, worst
    assert res.identical_across_ranks()


@pytest.mark.parametrize("dtype,op", [("i32", "sum"), ("i32", "min"), ("i32", "max"),
                                      ("f16", "min"), ("f16", "max"), ("bf16", "min"), ("bf16", "max")])
def test_bulkred_exact_ops_match_oracle(dtype, op):
    """Integer sums and min/max are exact in any order: bit-identical."""
    for p in (4, 8, 16):
        n = tma_sizes(p, dtype)[1]
        xs = gen(dtype, op, p, n, seed=90 + p)
        res, _ = run_collective(xs, "ar", op, dtype, "ring", variant="tma_bulkred")
        want = oracle.allreduce(xs, op, dtype, "ring")
        for r in range(p):
            assert bits_equal(res.host(r), want[r]), (p, r)
        rs, desc = run_collective(xs, "rs", op, dtype, "allpairs", variant="tma_bulkred")
        assert "reduce_scatter_tma_bulkred" in desc
        want = oracle.reduce_scatter(xs, op, dtype, "allpairs")
        for r in range(p):
            assert bits_equal(rs.host(r), want[r]), (p, r)


@pytest.mark.parametrize("budget", [1, 4])
def test_bulkred_exact_ops_under_budget_match_oracle(budget):
    """Under an SM budget one CTA per SM runs several bulk-reduce pipes (up to
    four, each on its own tiles): int32 sum and bf16 max stay bit-identical to
    the oracle for every p, including a short last tile and more tiles than
    pipes x CTAs."""
    for dtype, op in (("i32", "sum"), ("bf16", "max")):
        for p in (2, 4, 8, 16, 17):
            n = tma_sizes(p, dtype)[2]
            xs = gen(dtype, op, p, n, seed=120 + p)
            res, desc = run_collective(xs, "ar", op, dtype, "ring", variant="tma_bulkred", budget=budget)
            assert int(desc.split("grid=")[1].split()[0]) <= budget, desc
            want = oracle.allreduce(xs, op, dtype, "ring")
            for r in range(p):
                assert bits_equal(res.host(r), want[r]), (dtype, p, r, desc)
            rs, desc = run_collective(xs, "rs", op, dtype, "allpairs", variant="tma_bulkred", budget=budget)
            want = oracle.reduce_scatter(xs, op, dtype, "allpairs")
            for r in range(p):
                assert bits_equal(rs.host(r), want[r]), (dtype, p, r, desc)


@pytest.mark.parametrize("p", [17, 24, 40, 64])
def test_bulkred_many_ranks(p):
    """Above 16 ranks the bulk-reduce stages hold eight ranks of a tile at a
    time: int32 sum and bf16 max stay bit-exact, bf16 sum within the bound,
    with a short last tile and a short last batch, on every SM and under a
    budget."""
    for dtype, op in (("i32", "sum"), ("bf16", "max"), ("bf16", "sum")):
        s = inputs.ELEM_BYTES[dtype]
        n = p * (3 * 4096 // s + 5 * (16 // s))
        xs = gen(dtype, op, p, n, seed=170 + p)
        for budget in (0, 3):
            res, desc = run_collective(xs, "ar", op, dtype, "ring", variant="tma_bulkred", budget=budget)
            if op == "sum" and dtype == "bf16":
                ok, worst = within_reassociation_bound(res.host(0), xs, dtype)
                assert ok, (p, budget, worst)
                assert res.identical_across_ranks()
            else:
                want = oracle.allreduce(xs, op, dtype, "ring")
                for r in range(p):
                    assert bits_equal(res.host(r), want[r]), (dtype, op, p, budget, r, desc)


def test_bulkred_reduce_scatter_in_place_and_budget():
    p, dtype = 8, "bf16"
    n = p * (1 << 18)
    xs = gen(dtype, "sum", p, n, seed=95)
    storage = inputs.STORAGE[dtype]
    ins = RankBuffers(xs, n, storage)
    chunk = n // p
    with Comm(ins, out_ptrs=[ins.ptr(r, r * chunk) for r in range(p)]) as cm:
        ccl.ccl_set_launch(cm.h, 8, "tma_bulkred", 0)
        ccl.ccl_reduce_scatter(cm.h, "sum", dtype, n, "ring", stream_ptr())
        torch.cuda.synchronize()
        desc = ccl.ccl_comm_last_launch(cm.h)
        ccl.ccl_comm_check(cm.h)
    assert int(desc.split("grid=")[1].split()[0]) <= 8
    for r in range(p):
        got = ins.host(r)[r * chunk:(r + 1) * chunk]
        ok, worst = within_reassociation_bound(got, [x[r * chunk:(r + 1) * chunk] for x in xs], dtype)
        assert ok, (r, worst)
    assert ins.guards_intact()


def test_bulkred_statuses():
    p = 8
    xs = gen("f32", "sum", p, p * 64, seed=96)
    ins = RankBuffers(xs, p * 64, np.float32)
    outs = RankBuffers(None, p * 64, np.float32, p=p)
    with Comm(ins, outs) as cm:
        ccl.ccl_set_launch(cm.h, 0, "tma_bulkred", 0)
        for op, dtype in (("prod", "f32"), ("avg", "f32"), ("min", "f32"), ("max", "f32")):
            with pytest.raises(ccl.CclError) as ei:
                ccl.ccl_allreduce(cm.h, op, dtype, p * 64, "ring", stream_ptr())
            assert ei.value.status == ccl.CCL_ERR_UNSUPPORTED
        with pytest.raises(ccl.CclError) as ei:                   # n % p != 0
            ccl.ccl_allreduce(cm.h, "sum", "f32", p * 64 - 4, "ring", stream_ptr())
        assert ei.value.status == ccl.CCL_ERR_UNSUPPORTED
    torch.cuda.synchronize()
