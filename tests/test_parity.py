"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle
on the same seeded inputs.  Fixed-order results must be bit-identical
(every op, every dtype, both schedules).  Full-size workloads compare sampled
elements one by one with the oracle and check size-independent properties
(all ranks identical, schedule invariance of exact ops, invariance to the
launch shape)."""
import numpy as np
import pytest
import torch

import oracle
import reducescatter_reduction_gb300 as ccl
from reducescatter_reduction_gb300 import inputs
from ccl_testutil import (Comm, RankBuffers, bits_equal, ensure_built, sample_indices,
                          stream_ptr)
from conftest import read_golden

pytestmark = pytest.mark.gpu

DTYPES = ["f32", "f16", "bf16", "i32"]
OPS = ["sum", "prod", "min", "max", "avg"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ensure_built()


def gen(dtype, op, p, n, seed):
    """Seeded rank buffers for an op: small ints for prod (exact, no overflow
    to inf), uniform ints for int32, normals otherwise."""
    if dtype == "i32":
        if op == "prod":
            return [inputs.choice(n, seed, r, [-1, 1, 2], "i32") for r in range(p)]
        return [inputs.uniform_int(n, seed, r, -1000, 1000, "i32") for r in range(p)]
    if op == "prod":
        return [inputs.choice(n, seed, r, [-2, -1, 1, 2], dtype) for r in range(p)]
    return [inputs.normal(n, seed, r, 1.0, dtype) for r in range(p)]


def run_collective(xs, coll, op, dtype, sched="ring", inplace=False, offset=0, budget=0,
                   variant="ldst", n=None, in_device="cuda", out_device="cuda"):
    storage = inputs.STORAGE[dtype]
    p = len(xs)
    n = xs[0].size if n is None else n
    ins = RankBuffers(xs, n, storage, offset=offset, device=in_device)
    out_n = n // p if coll == "rs" else n
    outs = None if inplace else RankBuffers(None, out_n, storage, p=p, offset=offset, device=out_device)
    with Comm(ins, outs) as cm:
        ccl.ccl_set_launch(cm.h, budget, variant, 0)
        before = ccl.ccl_comm_launch_count(cm.h)
        if coll == "ar":
            ccl.ccl_allreduce(cm.h, op, dtype, n, sched, stream_ptr())
        elif coll == "rs":
            ccl.ccl_reduce_scatter(cm.h, op, dtype, n, sched, stream_ptr())
        else:
            ccl.ccl_all_gather(cm.h, dtype, n, stream_ptr())
        torch.cuda.synchronize()
        launched = ccl.ccl_comm_launch_count(cm.h) - before
        desc = ccl.ccl_comm_last_launch(cm.h)
    res = ins if inplace else outs
    assert ins.guards_intact(), "write outside the buffers"
    if outs is not None:
        assert outs.guards_intact(), "write outside the output buffers"
    if n:
        assert launched >= 1, "no kernel ran"
    return res, desc


# ---------------------------------------------------------------------------
# the worked example workload
# ---------------------------------------------------------------------------

def test_worked_example_workload():
    rows = {r[0]: [float(v) for v in r[1:]] for r in read_golden("worked_example.txt")}
    xs = inputs.worked()
    res, desc = run_collective(xs, "ar", "sum", "f32", "ring")
    want = oracle.allreduce(xs, "sum", "f32", "ring")
    for r in range(2):
        got = res.host(r)
        assert got[:4].tolist() == rows["result"]
        assert bits_equal(got, want[r])
    assert "allreduce_ldst" in desc and "schedule=ring" in desc and "vec=1" in desc


# ---------------------------------------------------------------------------
# small shapes: every op x dtype x schedule, many p and n (incl. empty and
# sizes that are not multiples of the 16-byte group or of p)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("sched", ["ring", "allpairs"])
def test_allreduce_small_exhaustive(dtype, op, sched):
    for p in (1, 2, 3, 8, 16, 17, 64):
        for n in (0, 1, 9, 65, 1027):
            xs = gen(dtype, op, p, n, seed=1000 + p)
            res, _ = run_collective(xs, "ar", op, dtype, sched)
            want = oracle.allreduce(xs, op, dtype, sched)
            for r in range(p):
                assert bits_equal(res.host(r), want[r]), (p, n, r)


# ---------------------------------------------------------------------------
# several grid sweeps, ragged tails, chunk boundaries off the 16-byte grid
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("p,dtype,op,sched", [
    (8, "bf16", "sum", "ring"), (8, "bf16", "avg", "allpairs"), (16, "bf16", "sum", "ring"),
    (5, "f32", "sum", "ring"), (4, "f16", "max", "ring"), (8, "i32", "prod", "allpairs"),
    (3, "f32", "min", "allpairs"), (2, "bf16", "prod", "ring"), (24, "f16", "avg", "ring"),
    (16, "i32", "avg", "ring"),
])
def test_allreduce_multi_sweep_ragged(p, dtype, op, sched):
    n = 3 * (1 << 20) + 13
    xs = gen(dtype, op, p, n, seed=7)
    res, desc = run_collective(xs, "ar", op, dtype, sched)
    want = oracle.allreduce(xs, op, dtype, sched)
    for r in range(p):
        assert bits_equal(res.host(r), want[r]), r
    assert "vec=1" in desc


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("p,budget", [(8, 0), (8, 2), (5, 0), (16, 2)])
def test_allreduce_in_place(dtype, p, budget):
    """In place (outputs are the inputs): the launch takes the instantiation
    that loads without ld.global.nc (inplace=1); float inputs reveal the
    accumulation order (inputs.cancel)."""
    n = p * (1 << 15) + 5
    if dtype == "i32":
        xs = gen(dtype, "sum", p, n, seed=8)
    else:
        xs = [inputs.cancel(n, 8, r, p, dtype) for r in range(p)]
    for sched in ("ring", "allpairs"):
        res, desc = run_collective(xs, "ar", "sum", dtype, sched, inplace=True, budget=budget)
        assert "inplace=1" in desc and "allreduce_ldst" in desc, desc
        want = oracle.allreduce(xs, "sum", dtype, sched)
        for r in range(p):
            assert bits_equal(res.host(r), want[r])
    _, desc = run_collective(xs, "ar", "sum", dtype, "ring", budget=budget)
    assert "inplace=0" in desc, desc


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("coll", ["ar", "rs", "ag"])
def test_misaligned_pointers_take_elementwise_path(dtype, coll):
    p, n = 4, 4 * 1000
    s = inputs.ELEM_BYTES[dtype]
    xs = gen(dtype, "sum", p, n, seed=9)
    res, desc = run_collective(xs, coll, "sum", dtype, "allpairs", offset=s)
    assert "vec=0" in desc
    if coll == "ar":
        want = oracle.allreduce(xs, "sum", dtype, "allpairs")
    elif coll == "rs":
        want = oracle.reduce_scatter(xs, "sum", dtype, "allpairs")
    else:
        want = oracle.all_gather(xs, dtype)
    for r in range(p):
        assert bits_equal(res.host(r), want[r])


# ---------------------------------------------------------------------------
# ReduceScatter and AllGather
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", OPS)
def test_reduce_scatter(dtype, op):
    for p, n, sched in ((2, 2 * 4099, "ring"), (3, 3 * 1000, "allpairs"), (8, 8 * 65536, "ring"),
                        (16, 16 * 513, "allpairs"), (1, 77, "ring")):
        xs = gen(dtype, op, p, n, seed=11)
        res, _ = run_collective(xs, "rs", op, dtype, sched)
        want = oracle.reduce_scatter(xs, op, dtype, sched)
        for r in range(p):
            assert bits_equal(res.host(r), want[r]), (p, r)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_reduce_scatter_in_place_nccl_convention(dtype):
    """In place as NCCL defines it: rank r's output is chunk r of its own
    input buffer."""
    p, n = 8, 8 * 40000
    xs = [inputs.cancel(n, 12, r, p, dtype) for r in range(p)]
    storage = inputs.STORAGE[dtype]
    ins = RankBuffers(xs, n, storage)
    with Comm(ins, out_ptrs=[ins.ptr(r, r * (n // p)) for r in range(p)]) as cm:
        ccl.ccl_reduce_scatter(cm.h, "sum", dtype, n, "ring", stream_ptr())
        torch.cuda.synchronize()
        assert "inplace=1" in ccl.ccl_comm_last_launch(cm.h)
    want = oracle.reduce_scatter(xs, "sum", dtype, "ring")
    for r in range(p):
        got = ins.host(r)[r * (n // p):(r + 1) * (n // p)]
        assert bits_equal(got, want[r])
    assert ins.guards_intact()


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("inplace", [False, True])
@pytest.mark.parametrize("budget", [0, 3])
def test_all_gather(dtype, inplace, budget):
    """Budget 3: the persistent kernel (several units per thread per round)
    wherever the message needs more than three small CTAs."""
    for p, n in ((2, 2 * 4099), (3, 3 * 1000), (8, 8 * 65536), (16, 16 * 513), (5, 5 * 8)):
        xs = gen(dtype, "sum", p, n, seed=13)
        res, _ = run_collective(xs, "ag", None, dtype, inplace=inplace, budget=budget)
        want = oracle.all_gather(xs, dtype)
        for r in range(p):
            assert bits_equal(res.host(r), want[r]), (p, r)


@pytest.mark.parametrize("tokens", inputs.TP_TOKENS)
def test_tp_activation_allreduce_equals_rs_then_ag(tokens):
    """Tensor-parallel activations [tokens, 8192] at TP=8: AllReduce matches
    the oracle, and ReduceScatter (rank r gets [tokens, 1024]) followed by an
    in-place AllGather gives the same bits ("Inside NCCL AllReduce": all-reduce
    = reduce-scatter + all-gather)."""
    p, dtype = 8, "bf16"
    xs = inputs.tp(tokens, p)
    n = xs[0].size
    storage = inputs.STORAGE[dtype]
    ar, _ = run_collective(xs, "ar", "sum", dtype, "ring")
    if n <= 256 * 8192:
        want = oracle.allreduce(xs, "sum", dtype, "ring")
        for r in range(p):
            assert bits_equal(ar.host(r), want[r])
    else:
        idx = sample_indices(p, n)
        want = oracle.allreduce_at(xs, idx, "sum", dtype, "ring")
        for r in range(p):
            assert bits_equal(ar.at(r, idx), want)
    ins = RankBuffers(xs, n, storage)
    z = RankBuffers(None, n, storage, p=p)
    chunk = n // p
    with Comm(ins, out_ptrs=[z.ptr(r, r * chunk) for r in range(p)]) as cm:
        ccl.ccl_reduce_scatter(cm.h, "sum", dtype, n, "ring", stream_ptr())
    with Comm(z) as cm:                        # in place: out[r] == in[r]
        ccl.ccl_all_gather(cm.h, dtype, n, stream_ptr())
    torch.cuda.synchronize()
    for r in range(p):
        assert torch.equal(z.views[r], ar.views[r]), r
    assert z.guards_intact()


# ---------------------------------------------------------------------------
# custom schedules
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("p", [3, 8, 16, 20])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_custom_schedule(p, dtype):
    rng = np.random.default_rng(p)
    table = [list(rng.permutation(p)) for _ in range(p)]
    n = p * 10007 + 3
    xs = gen(dtype, "sum", p, n, seed=14)
    storage = inputs.STORAGE[dtype]
    ins = RankBuffers(xs, n, storage)
    outs = RankBuffers(None, n, storage, p=p)
    with Comm(ins, outs) as cm:
        ccl.ccl_comm_set_schedule(cm.h, table)
        ccl.ccl_allreduce(cm.h, "sum", dtype, n, "custom", stream_ptr())
        torch.cuda.synchronize()
        assert "schedule=custom" in ccl.ccl_comm_last_launch(cm.h)
    want = oracle.allreduce_orders(xs, "sum", dtype, table)
    for r in range(p):
        assert bits_equal(outs.host(r), want[r])


# ---------------------------------------------------------------------------
# schedule selection, launch accounting, streams
# ---------------------------------------------------------------------------

def test_auto_schedule_follows_cost_model(monkeypatch):
    p = 8
    for n, want in ((1 << 10, "allpairs"), (1 << 24, "ring")):
        xs = gen("bf16", "sum", p, n, seed=15)
        _, desc = run_collective(xs, "ar", "sum", "bf16", "auto")
        assert f"schedule={want}" in desc
        assert ccl.ccl_select_schedule(p, n * 2) == (ccl.CCL_SCHED_ALLPAIRS if want == "allpairs"
                                                     else ccl.CCL_SCHED_RING)
    monkeypatch.setenv("CCL_SCHEDULE", "ring")
    xs = gen("bf16", "sum", p, 1 << 10, seed=15)
    _, desc = run_collective(xs, "ar", "sum", "bf16", "auto")
    assert "schedule=ring" in desc


def test_environment_overrides_apply_only_to_open_choices(monkeypatch):
    """CCL_SCHEDULE, CCL_VARIANT and CCL_SM_BUDGET change a call only where
    the call or the communicator left the choice open (schedule auto, variant
    auto, SM budget 0); values outside their lists are refused, never ignored."""
    p, n = 8, 8 * (1 << 16)
    xs = gen("bf16", "sum", p, n, seed=17)
    want = oracle.allreduce(xs, "sum", "bf16", "allpairs")
    monkeypatch.setenv("CCL_VARIANT", "tma")
    monkeypatch.setenv("CCL_SM_BUDGET", "4")
    monkeypatch.setenv("CCL_SCHEDULE", "allpairs")
    res, desc = run_collective(xs, "ar", "sum", "bf16", "auto", variant="auto")
    assert "allreduce_tma" in desc and "sm_budget=4" in desc and "schedule=allpairs" in desc, desc
    assert bits_equal(res.host(0), want[0])
    # explicit arguments win
    res, desc = run_collective(xs, "ar", "sum", "bf16", "ring", variant="ldst", budget=8)
    assert "allreduce_ldst" in desc and "sm_budget=8" in desc and "schedule=ring" in desc, desc
    # AllGather has only the ld/st kernel: the variant override does not apply
    res, desc = run_collective(xs, "ag", "sum", "bf16", variant="auto")
    assert "all_gather_ldst" in desc and "sm_budget=4" in desc, desc
    for var, val in (("CCL_VARIANT", "fast"), ("CCL_SM_BUDGET", "-3"), ("CCL_SM_BUDGET", "4x"),
                     ("CCL_SCHEDULE", "tree")):
        monkeypatch.setenv(var, val)
        with pytest.raises(ccl.CclError) as ei:
            run_collective(xs, "ar", "sum", "bf16", "auto", variant="auto")
        assert ei.value.status == ccl.CCL_ERR_INVALID_ARG and var in str(ei.value)
        monkeypatch.setenv(var, {"CCL_VARIANT": "auto", "CCL_SM_BUDGET": "", "CCL_SCHEDULE": "auto"}[var])


def test_side_stream_and_launch_count():
    p, n, dtype = 8, 1 << 20, "bf16"
    xs = gen(dtype, "sum", p, n, seed=16)
    storage = inputs.STORAGE[dtype]
    ins = RankBuffers(xs, n, storage)
    outs = RankBuffers(None, n, storage, p=p)
    side = torch.cuda.Stream()
    torch.cuda.synchronize()
    with Comm(ins, outs) as cm:
        with torch.cuda.stream(side):
            for _ in range(3):
                ccl.ccl_allreduce(cm.h, "sum", dtype, n, "ring", side.cuda_stream)
        side.synchronize()
        assert ccl.ccl_comm_launch_count(cm.h) == 3
    want = oracle.allreduce(xs, "sum", dtype, "ring")
    assert bits_equal(outs.host(5), want[5])


# ---------------------------------------------------------------------------
# errors: explicit statuses, never a silent fallback
# ---------------------------------------------------------------------------

def test_argument_errors():
    p, n = 4, 4 * 256
    xs = gen("f32", "sum", p, n, seed=17)
    ins = RankBuffers(xs, n, np.float32)
    outs = RankBuffers(None, n, np.float32, p=p)
    with Comm(ins, outs) as cm:
        def status(fn, *a):
            try:
                fn(*a)
                return ccl.CCL_OK
            except ccl.CclError as e:
                return e.status
        s = stream_ptr()
        assert status(ccl.ccl_reduce_scatter, cm.h, "sum", "f32", n + 1, "ring", s) == ccl.CCL_ERR_INVALID_ARG
        assert status(ccl.ccl_all_gather, cm.h, "f32", n - 2, s) == ccl.CCL_ERR_INVALID_ARG
        assert status(ccl.ccl_allreduce, cm.h, 9, "f32", n, "ring", s) == ccl.CCL_ERR_INVALID_ARG
        assert status(ccl.ccl_allreduce, cm.h, "sum", 7, n, "ring", s) == ccl.CCL_ERR_INVALID_ARG
        assert status(ccl.ccl_allreduce, cm.h, "sum", "f32", n, 9, s) == ccl.CCL_ERR_INVALID_ARG
        assert status(ccl.ccl_allreduce, cm.h, "sum", "f32", n, "custom", s) == ccl.CCL_ERR_INVALID_ARG
        assert status(ccl.ccl_comm_set_schedule, cm.h, [[0, 1, 2, 2]] * 4) == ccl.CCL_ERR_INVALID_ARG
        assert status(ccl.ccl_set_launch, cm.h, -1, "ldst", 0) == ccl.CCL_ERR_INVALID_ARG
        assert status(ccl.ccl_set_launch, cm.h, 0, 9, 0) == ccl.CCL_ERR_INVALID_ARG
        assert status(ccl.ccl_set_launch, cm.h, 0, "tma", 100) == ccl.CCL_ERR_INVALID_ARG
        # overlapping outputs
        ccl.ccl_comm_set_outputs(cm.h, [outs.ptr(0), outs.ptr(0, 10), outs.ptr(2), outs.ptr(3)])
        assert status(ccl.ccl_allreduce, cm.h, "sum", "f32", n, "ring", s) == ccl.CCL_ERR_INVALID_ARG
        # an output overlapping another rank's input
        ccl.ccl_comm_set_outputs(cm.h, [ins.ptr(1), outs.ptr(1), outs.ptr(2), outs.ptr(3)])
        assert status(ccl.ccl_allreduce, cm.h, "sum", "f32", n, "ring", s) == ccl.CCL_ERR_INVALID_ARG
        # ReduceScatter written at offset 0 of its own (n-element) input overlaps chunk 0
        ccl.ccl_comm_set_outputs(cm.h, [ins.ptr(r) for r in range(p)])
        assert status(ccl.ccl_reduce_scatter, cm.h, "sum", "f32", n, "ring", s) == ccl.CCL_ERR_INVALID_ARG
        # n == 0 is a no-op
        ccl.ccl_comm_set_outputs(cm.h, None)
        count = ccl.ccl_comm_launch_count(cm.h)
        ccl.ccl_allreduce(cm.h, "sum", "f32", 0, "ring", s)
        assert ccl.ccl_comm_launch_count(cm.h) == count
        ccl.ccl_comm_check(cm.h)
    torch.cuda.synchronize()
    assert ins.guards_intact() and outs.guards_intact()
    for r in range(p):                         # nothing was written
        assert bits_equal(ins.host(r), xs[r])


# ---------------------------------------------------------------------------
# full-size workloads
# ---------------------------------------------------------------------------

def test_sweep_bf16_p8():
    """p=8 bf16 N(0,1), 1 KiB .. 256 MiB per rank, ring and all-pairs, in the
    launch shape the benchmark times (all SMs, ld/st): full comparison up to
    512 KiB per rank, sampled beyond; all ranks identical."""
    p = 8
    for n in inputs.SWEEP_N:
        xs = inputs.sweep(n, p)
        for sched in ("ring", "allpairs"):
            res, desc = run_collective(xs, "ar", "sum", "bf16", sched)
            assert "vec=1" in desc and f"schedule={sched}" in desc
            if n <= 1 << 18:
                want = oracle.allreduce(xs, "sum", "bf16", sched)
                for r in range(p):
                    assert bits_equal(res.host(r), want[r]), (n, sched)
            else:
                idx = sample_indices(p, n, count=50000, seed=n)
                want = oracle.allreduce_at(xs, idx, "sum", "bf16", sched)
                assert bits_equal(res.at(0, idx), want), (n, sched)
                assert bits_equal(res.at(p - 1, idx), want), (n, sched)
                assert res.identical_across_ranks(), (n, sched)
            del res
        del xs
        torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype,ops", [("i32", ["sum", "min", "max", "prod"]),
                                       ("f32", ["avg", "sum", "max"]),
                                       ("f16", ["avg", "sum", "max"])])
def test_op_coverage_64M(dtype, ops):
    """p=8, n = 64 Mi per rank: int32 results bit-exact and identical under
    both schedules; fp32/fp16 avg (1/p folded into the kernel), sum, max."""
    p, n = 8, inputs.COVERAGE_N
    idx = sample_indices(p, n, count=50000, seed=4)
    cache = {}
    for op in ops:
        key = op == "prod"
        if key not in cache:
            cache.clear()
            cache[key] = inputs.coverage(op, dtype, n=n, p=p)
        xs = cache[key]
        res, _ = run_collective(xs, "ar", op, dtype, "ring")
        want = oracle.allreduce_at(xs, idx, op, dtype, "ring")
        assert bits_equal(res.at(0, idx), want), op
        assert res.identical_across_ranks(), op
        if dtype == "i32" or op == "max":
            res2, _ = run_collective(xs, "ar", op, dtype, "allpairs")
            assert torch.equal(res.views[0], res2.views[0]), op
            del res2
        del res
        torch.cuda.empty_cache()


def test_moe_p16_sm_budgets():
    """p=16 bf16 [16384, 7168] per rank (224 MiB each), ring: sampled oracle
    comparison, and the same bits from the ld/st and TMA variants at SM
    budgets 4, 8, 16 and all; the bulk-reduce variant within its bound."""
    p, dtype = 16, "bf16"
    xs = inputs.moe(p)
    n = xs[0].size
    idx = sample_indices(p, n, count=50000, seed=5)
    want = oracle.allreduce_at(xs, idx, "sum", dtype, "ring")
    storage = inputs.STORAGE[dtype]
    ins = RankBuffers(xs, n, storage)
    xf = np.stack([x[idx.astype(np.int64)] for x in xs])
    xf = torch.from_numpy(xf.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    exact, bound = xf.sum(axis=0), 2 * p * 2.0 ** -7 * np.abs(xf).sum(axis=0)
    del xs
    ref = None
    for variant, budget in (("ldst", 0), ("ldst", 4), ("ldst", 8), ("ldst", 16),
                            ("tma", 0), ("tma", 4), ("tma", 8), ("tma", 16)):
        outs = RankBuffers(None, n, storage, p=p)
        with Comm(ins, outs) as cm:
            ccl.ccl_set_launch(cm.h, budget, variant, 0)
            ccl.ccl_allreduce(cm.h, "sum", dtype, n, "ring", stream_ptr())
            torch.cuda.synchronize()
            desc = ccl.ccl_comm_last_launch(cm.h)
        grid = int(desc.split("grid=")[1].split()[0])
        if budget:
            assert grid <= budget
        assert bits_equal(outs.at(0, idx), want)
        assert outs.identical_across_ranks()
        if ref is None:
            ref = outs.views[0].clone()
        else:
            assert torch.equal(outs.views[0], ref), budget
        assert outs.guards_intact()
        del outs
        torch.cuda.empty_cache()
    # the bulk-reduce variant lets the memory system order the adds: within the
    # reassociation bound at the sampled elements, identical on every rank
    for budget in (0, 16):
        outs = RankBuffers(None, n, storage, p=p)
        with Comm(ins, outs) as cm:
            ccl.ccl_set_launch(cm.h, budget, "tma_bulkred", 0)
            ccl.ccl_allreduce(cm.h, "sum", dtype, n, "ring", stream_ptr())
            torch.cuda.synchronize()
            ccl.ccl_comm_check(cm.h)
        got = torch.from_numpy(outs.at(0, idx).view(np.int16).copy()).view(torch.bfloat16).double().numpy()
        assert np.all(np.abs(got - exact) <= bound), budget
        assert outs.identical_across_ranks()
        del outs
        torch.cuda.empty_cache()


@pytest.mark.parametrize("variant", ["ldst", "tma"])
def test_cuda_graph_capture_and_replay(variant):
    """The collective calls only check arguments and enqueue kernels, so they
    can be captured in a CUDA graph; replays recompute from the current input
    contents."""
    p, n, dtype = 8, 8 * 65536, "bf16"
    xs = gen(dtype, "sum", p, n, seed=50)
    ys = gen(dtype, "sum", p, n, seed=51)
    storage = inputs.STORAGE[dtype]
    ins = RankBuffers(xs, n, storage)
    outs = RankBuffers(None, n, storage, p=p)
    rs_out = RankBuffers(None, n // p, storage, p=p)
    with Comm(ins, outs) as cm, Comm(ins, rs_out) as cm_rs:
        ccl.ccl_set_launch(cm.h, 0, variant, 0)
        ccl.ccl_set_launch(cm_rs.h, 0, variant, 0)
        ccl.ccl_allreduce(cm.h, "sum", dtype, n, "ring", stream_ptr())      # first use: kernel attributes
        ccl.ccl_reduce_scatter(cm_rs.h, "sum", dtype, n, "ring", stream_ptr())
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                s = torch.cuda.current_stream().cuda_stream
                ccl.ccl_allreduce(cm.h, "sum", dtype, n, "ring", s)
                ccl.ccl_reduce_scatter(cm_rs.h, "sum", dtype, n, "ring", s)
        torch.cuda.current_stream().wait_stream(side)
        for src in (xs, ys):
            for r in range(p):
                ins.views[r].copy_(torch.from_numpy(src[r].view(np.uint8)).to("cuda"))
            g.replay()
            torch.cuda.synchronize()
            want = oracle.allreduce(src, "sum", dtype, "ring")
            want_rs = oracle.reduce_scatter(src, "sum", dtype, "ring")
            for r in range(p):
                assert bits_equal(outs.host(r), want[r])
                assert bits_equal(rs_out.host(r), want_rs[r])
        ccl.ccl_comm_check(cm.h)


def _dependent_chain_oracle(xs):
    y = oracle.allreduce(xs, "sum", "f32", "ring")
    y[0] = y[0] * np.float32(2.0)
    y = oracle.allreduce(y, "max", "f32", "allpairs")
    y = oracle.allreduce(y, "sum", "f32", "ring")
    rs = oracle.reduce_scatter(y, "sum", "f32", "ring")
    chunk = len(rs[0])
    return y, [np.concatenate(rs) for _ in rs], chunk


@pytest.mark.parametrize("graph", [False, True])
def test_dependent_launch_chain(graph):
    """The ld/st, AllGather and fused kernels are launched as programmatic
    dependents: each may be scheduled while the kernel before it drains, and
    waits for that kernel's writes before touching memory.  A chain of
    collectives, each reading what the previous one wrote (with an ordinary
    torch kernel in between), issued back to back without synchronising,
    must give the oracle's chain bit for bit, on a stream and in a CUDA graph."""
    p, n = 8, 8 * 65536                                # one wave of CTAs: every CTA starts at once
    xs = gen("f32", "sum", p, n, seed=56)
    ins = RankBuffers(xs, n, np.float32)
    b = RankBuffers(None, n, np.float32, p=p)
    c = RankBuffers(None, n, np.float32, p=p)
    d = RankBuffers(None, n, np.float32, p=p)
    want_b, want_d, chunk = _dependent_chain_oracle(xs)
    with Comm(ins, b) as cm_ab, Comm(b, c) as cm_bc, Comm(c, b) as cm_cb, \
            Comm(b, out_ptrs=[d.ptr(r, r * (n // p)) for r in range(p)]) as cm_bd:
        ccl.ccl_set_launch(cm_cb.h, 3, "ldst", 0)                 # the persistent SM-budget kernel
        # the AllGather runs in place on D: its rank buffers are D itself
        ag = ccl.ccl_comm_create(p, d.ptrs())
        try:
            def chain(s):
                assert torch.cuda.current_stream().cuda_stream == s
                ccl.ccl_allreduce(cm_ab.h, "sum", "f32", n, "ring", s)
                b.views[0].view(torch.float32).mul_(2.0)            # torch's current stream is s
                ccl.ccl_allreduce(cm_bc.h, "max", "f32", n, "allpairs", s)
                ccl.ccl_allreduce(cm_cb.h, "sum", "f32", n, "ring", s)
                ccl.ccl_reduce_scatter(cm_bd.h, "sum", "f32", n, "ring", s)
                ccl.ccl_all_gather(ag, "f32", n, s)
            if graph:
                chain(stream_ptr())                                 # first use outside the capture
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                side = torch.cuda.Stream()
                side.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(side):
                    with torch.cuda.graph(g, stream=side):
                        chain(torch.cuda.current_stream().cuda_stream)
                torch.cuda.current_stream().wait_stream(side)
                for _ in range(2):
                    g.replay()
            else:
                for _ in range(2):
                    chain(stream_ptr())
            torch.cuda.synchronize()
        finally:
            ccl.ccl_comm_destroy(ag)
    for r in range(p):
        assert bits_equal(b.host(r), want_b[r]), r
        assert bits_equal(d.host(r), want_d[r]), r
    assert ins.guards_intact() and b.guards_intact() and c.guards_intact() and d.guards_intact()


def auto_expect(p, dtype, budget, nbytes):
    """The variant AUTO must take by the launch table's rule (include/ccl.h,
    ccl_launch_estimate): TMA exactly when its estimate is below 0.98 times
    the ld/st one (the layouts here all allow TMA)."""
    try:
        ldst = ccl.ccl_launch_estimate(p, dtype, budget, nbytes, "ldst")
        tma = ccl.ccl_launch_estimate(p, dtype, budget, nbytes, "tma")
    except ccl.CclError:
        return "ldst"
    return "tma" if tma < 0.98 * ldst else "ldst"


def test_budget_kernel_shapes():
    """Under a budget a large ld/st message runs one 512/1024-thread CTA per
    SM; a message that already fits in `budget` small CTAs keeps the regular
    kernel."""
    p, n = 16, 16 * 65536                                 # 2 MiB per rank: 131072 groups
    xs = gen("bf16", "sum", p, n, seed=52)
    _, desc = run_collective(xs, "ar", "sum", "bf16", "ring")
    assert "variant=ldst" in desc and "block=128" in desc
    _, desc = run_collective(xs, "ar", "sum", "bf16", "ring", budget=16)
    assert "variant=ldst" in desc and "grid=16 block=512" in desc
    small = gen("bf16", "sum", p, 16 * 64, seed=54)       # 2 KiB per rank: one 128-thread CTA
    res, desc = run_collective(small, "ar", "sum", "bf16", "ring", budget=16)
    assert "variant=ldst" in desc and "grid=1 block=128" in desc
    want = oracle.allreduce(small, "sum", "bf16", "ring")
    assert bits_equal(res.host(3), want[3])


@pytest.mark.parametrize("p,dtype,budget_frac,rank_bytes", [
    (8, "bf16", 0.5, 32 << 20), (8, "bf16", 0.5, 16 << 20), (8, "bf16", 0.0, 256 << 20), (8, "bf16", 32, 32 << 20),
    (2, "f32", 8, 4 << 20), (4, "bf16", 0.5, 64 << 20), (16, "bf16", 0.5, 64 << 20), (48, "bf16", 0.0, 68 << 20),
    (48, "bf16", 0.0, 8 << 20), (64, "f32", 0.0, 32 << 20), (3, "f32", 16, 1 << 20), (24, "bf16", 76, 16 << 20),
])
def test_auto_variant_follows_the_launch_table(p, dtype, budget_frac, rank_bytes):
    """AUTO takes the kernel the measured launch table estimates faster, and
    either kernel gives the ld/st kernel's bits.  budget_frac < 1 is a share
    of the device's SMs (0 = every SM), else an SM count."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    budget = int(budget_frac * sms) if budget_frac < 1 else int(budget_frac)
    s = inputs.ELEM_BYTES[dtype]
    grain = p * 16 // s                                   # 16-byte chunk boundaries: TMA may run
    n = (rank_bytes // s) // grain * grain
    want_variant = auto_expect(p, dtype, budget, n * s)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    ins = [torch.empty(n, dtype=tdt, device="cuda").normal_() for _ in range(p)]
    outs = [torch.empty_like(t) for t in ins]
    ref = [torch.empty_like(t) for t in ins]
    h = ccl.ccl_comm_create(p, [t.data_ptr() for t in ins])
    try:
        ccl.ccl_comm_set_outputs(h, [t.data_ptr() for t in outs])
        ccl.ccl_set_launch(h, budget, "auto", 0)
        ccl.ccl_allreduce(h, "sum", dtype, n, "ring", stream_ptr())
        desc = ccl.ccl_comm_last_launch(h)
        ccl.ccl_comm_set_outputs(h, [t.data_ptr() for t in ref])
        ccl.ccl_set_launch(h, budget, "ldst", 0)
        ccl.ccl_allreduce(h, "sum", dtype, n, "ring", stream_ptr())
        torch.cuda.synchronize()
        ccl.ccl_comm_check(h)
    finally:
        ccl.ccl_comm_destroy(h)
    assert f"variant={want_variant}" in desc, desc
    iv = torch.int16 if s == 2 else torch.int32
    assert all(torch.equal(a.view(iv), b.view(iv)) for a, b in zip(outs, ref))


def test_largest_buffers_64bit_indexing():
    """n = 2^31 + 64 bf16 per rank (4 GiB buffers, p=2): element indices pass
    2^31 and byte offsets pass 2^32.  ld/st, TMA and the allocation-free entry
    point agree with the oracle at sampled elements on both sides of 2^31 and
    of the chunk boundary n/2.  (With p=2 a sum is one fp32 addition, which is
    commutative, so the oracle on the sampled values alone is the reference.)"""
    p, n, dtype = 2, (1 << 31) + 64, "bf16"
    rng = np.random.default_rng(77)
    idx = np.unique(np.concatenate([rng.integers(0, n, 20000, dtype=np.int64),
                                    np.arange((1 << 31) - 64, n, dtype=np.int64),
                                    np.arange(0, 64, dtype=np.int64),
                                    np.arange(n // 2 - 16, n // 2 + 16, dtype=np.int64)]))
    didx = torch.from_numpy(idx).cuda()
    # seeded values at the sampled places, a constant elsewhere (cheap to build)
    bufs, xs_at = [], []
    for r in range(p):
        t = torch.full((n,), 0x3f80 + r, dtype=torch.int16, device="cuda")
        vals = inputs.normal(idx.size, 78, r, 1.0, dtype)
        t[didx] = torch.from_numpy(vals.view(np.int16)).cuda()
        bufs.append(t)
        xs_at.append(vals)
    want = oracle.allreduce(xs_at, "sum", dtype, "ring")[0]
    for variant in ("ldst", "tma"):
        out = [torch.empty_like(b) for b in bufs]
        h = ccl.ccl_comm_create(p, [b.data_ptr() for b in bufs])
        try:
            ccl.ccl_comm_set_outputs(h, [o.data_ptr() for o in out])
            ccl.ccl_set_launch(h, 0, variant, 0)
            ccl.ccl_allreduce(h, "sum", dtype, n, "ring", stream_ptr())
            torch.cuda.synchronize()
            ccl.ccl_comm_check(h)
        finally:
            ccl.ccl_comm_destroy(h)
        for r in range(p):
            got = out[r][didx].cpu().numpy().view(np.uint16)
            assert bits_equal(got, want), (variant, r)
        # an element outside the sample: 1.0 + 1.0078125 = 2.0078125, a bf16 tie -> 2.0 (0x4000)
        e_const = 1_000_000_007
        assert not np.isin(e_const, idx)
        for r in range(p):
            assert int(out[r][e_const].item()) == 0x4000
        del out
        torch.cuda.empty_cache()
    ccl.ccl_allreduce_static(p, [b.data_ptr() for b in bufs], [b.data_ptr() for b in bufs], "sum", dtype, n,
                             "ring", stream_ptr())
    torch.cuda.synchronize()
    for r in range(p):
        assert bits_equal(bufs[r][didx].cpu().numpy().view(np.uint16), want)
    del bufs
    torch.cuda.empty_cache()


def test_concurrent_communicators_on_separate_streams():
    """Several communicators (different p, dtypes, variants) enqueued on
    separate streams without synchronising in between: each result matches
    the oracle.  The library's only shared state is per-kernel launch
    attributes set once."""
    cases = [(8, "bf16", "sum", "ring", "ldst"), (16, "bf16", "sum", "allpairs", "tma"),
             (4, "f32", "max", "ring", "tma"), (3, "i32", "prod", "allpairs", "ldst")]
    runs = []
    for i, (p, dtype, op, sched, variant) in enumerate(cases):
        n = p * 8 * 4096
        xs = gen(dtype, op, p, n, seed=200 + i)
        storage = inputs.STORAGE[dtype]
        ins = RankBuffers(xs, n, storage)
        outs = RankBuffers(None, n, storage, p=p)
        h = ccl.ccl_comm_create(p, ins.ptrs())
        ccl.ccl_comm_set_outputs(h, outs.ptrs())
        ccl.ccl_set_launch(h, 0, variant, 0)
        runs.append((xs, ins, outs, h, torch.cuda.Stream(), p, dtype, op, sched))
    torch.cuda.synchronize()
    for _ in range(3):
        for xs, ins, outs, h, st, p, dtype, op, sched in runs:
            ccl.ccl_allreduce(h, op, dtype, xs[0].size, sched, st.cuda_stream)
    torch.cuda.synchronize()
    for xs, ins, outs, h, st, p, dtype, op, sched in runs:
        want = oracle.allreduce(xs, op, dtype, sched)
        for r in range(p):
            assert bits_equal(outs.host(r), want[r]), (p, dtype, op, r)
        ccl.ccl_comm_check(h)
        ccl.ccl_comm_destroy(h)


# ---------------------------------------------------------------------------
# min/max on IEEE special values (fp16/bf16 fold packed pairs in place)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("op", ["min", "max"])
@pytest.mark.parametrize("p,variant,budget", [(8, "ldst", 0), (3, "ldst", 0), (5, "ldst", 0), (8, "ldst", 4),
                                              (16, "ldst", 0), (8, "tma", 0), (5, "tma", 0), (40, "tma", 0)])
def test_min_max_special_values(dtype, op, p, variant, budget):
    """Signed zeros, subnormals, infinities and quiet NaNs of both signs,
    drawn so that ties are frequent: bit-identical to the oracle's
    compare-and-select (earlier operand wins ties; a NaN only if it comes
    first), AllReduce and ReduceScatter, both schedules."""
    n = p * 8 * 1500
    xs = [inputs.specials(n, 97, r, dtype) for r in range(p)]
    for sched in ("ring", "allpairs"):
        res, desc = run_collective(xs, "ar", op, dtype, sched, budget=budget, variant=variant)
        want = oracle.allreduce(xs, op, dtype, sched)
        for r in range(p):
            assert bits_equal(res.host(r), want[r]), (sched, r, desc)
        res, desc = run_collective(xs, "rs", op, dtype, sched, budget=budget, variant=variant)
        want = oracle.reduce_scatter(xs, op, dtype, sched)
        for r in range(p):
            assert bits_equal(res.host(r), want[r]), (sched, r, desc)
    if variant == "ldst":
        # ragged: a group straddling a chunk boundary and a sub-group tail
        m = n + 3
        ys = [inputs.specials(m, 98, r, dtype) for r in range(p)]
        res, desc = run_collective(ys, "ar", op, dtype, "ring", budget=budget, variant=variant)
        want = oracle.allreduce(ys, op, dtype, "ring")
        for r in range(p):
            assert bits_equal(res.host(r), want[r]), (r, desc)


# ---------------------------------------------------------------------------
# page-locked host buffers, addressed by the kernels directly (zero-copy)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("coll", ["ar", "rs", "ag"])
@pytest.mark.parametrize("where", [("pinned", "pinned"), ("pinned", "cuda"), ("cuda", "pinned")])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_host_buffers_zero_copy(coll, where, dtype):
    """Rank buffers in page-locked host memory: the ld/st kernels read and
    write them over the host link; bits equal the oracle's, and nothing is
    written outside the buffers."""
    p = 8
    n = p * 40000 + (3 if coll == "ar" else 0)
    op = "sum"
    xs = gen(dtype, op, p, n, seed=61)
    for inplace, budget in ((False, 0), (True, 0), (False, 8)):
        if inplace and (where[0] != where[1] or coll == "rs"):
            continue
        res, desc = run_collective(xs, coll, op, dtype, "ring", inplace=inplace, budget=budget,
                                   in_device=where[0], out_device=where[1])
        if coll == "ag":
            want = oracle.all_gather(xs, dtype)
        elif coll == "rs":
            want = oracle.reduce_scatter(xs, op, dtype, "ring")
        else:
            want = oracle.allreduce(xs, op, dtype, "ring")
        for r in range(p):
            assert bits_equal(res.host(r), want[r]), (coll, where, inplace, budget, r, desc)
