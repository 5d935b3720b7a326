"""ccl_allreduce_static: the AllReduce entry point for callers that may not
allocate device memory.

Such callers include a plug-in running inside an application that owns all
device memory (an inference server, a framework's memory pool), a process
whose memory budget is already committed, and a latency-critical path that
cannot afford cudaMalloc's implicit synchronisation.  The entry point needs
no communicator.  It keeps the only scratch its kernel uses, a 16-byte status
record, in a static device array of the library.

These tests call it through the C ABI and check that two calls in a row give
exactly the bits of the communicator entry point, ccl_allreduce, on the same
inputs (bit-exact, as every fixed-order test here). They also check that the
calls take no device memory. The file sorts last, so a run that stops at the
first failure has run every other test first.
"""
import numpy as np
import pytest
import torch

import reducescatter_reduction_gb300 as ccl
from reducescatter_reduction_gb300 import inputs
from ccl_testutil import Comm, RankBuffers, ensure_built, stream_ptr

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ensure_built()


CASES = [  # (dtype, op, schedule, p, n): every chunk a multiple of 16 bytes
    ("bf16", "sum", "ring", 8, 8 * (1 << 18)),
    ("f32", "avg", "allpairs", 16, 16 * 12288),
]


def _inputs(dtype, p, n, seed):
    return [inputs.normal(n, seed, r, 1.0, dtype) for r in range(p)]


def _reference(xs, dtype, op, sched):
    """The same AllReduce through the communicator API (ld/st kernel)."""
    n = xs[0].size
    storage = inputs.STORAGE[dtype]
    ins = RankBuffers(xs, n, storage)
    outs = RankBuffers(None, n, storage, p=len(xs))
    with Comm(ins, outs) as cm:
        ccl.ccl_allreduce(cm.h, op, dtype, n, sched, stream_ptr())
        torch.cuda.synchronize()
    return outs


def test_static_entry_matches_communicator_entry_on_two_calls():
    bufs = []
    for i, (dtype, op, sched, p, n) in enumerate(CASES):
        xs = _inputs(dtype, p, n, seed=60 + i)
        storage = inputs.STORAGE[dtype]
        bufs.append((xs, RankBuffers(xs, n, storage), RankBuffers(None, n, storage, p=p)))
    # two calls in a row, no synchronisation in between
    for (dtype, op, sched, p, n), (xs, ins, outs) in zip(CASES, bufs):
        ccl.ccl_allreduce_static(p, ins.ptrs(), outs.ptrs(), op, dtype, n, sched, stream_ptr())
    torch.cuda.synchronize()
    for (dtype, op, sched, p, n), (xs, ins, outs) in zip(CASES, bufs):
        ref = _reference(xs, dtype, op, sched)
        for r in range(p):
            assert torch.equal(outs.views[r], ref.views[r]), (dtype, op, r)
        assert outs.guards_intact() and ins.guards_intact()


def test_static_entry_allocates_nothing_and_keeps_working():
    dtype, op, sched, p, n = CASES[0]
    xs = _inputs(dtype, p, n, seed=70)
    storage = inputs.STORAGE[dtype]
    ins = RankBuffers(xs, n, storage)
    outs = RankBuffers(None, n, storage, p=p)
    ref = _reference(xs, dtype, op, sched)
    ccl.ccl_allreduce_static(p, ins.ptrs(), outs.ptrs(), op, dtype, n, sched, stream_ptr())
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        ccl.ccl_allreduce_static(p, ins.ptrs(), outs.ptrs(), op, dtype, n, sched, stream_ptr())
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before          # a device allocation would take at least a 2 MiB page
    for r in range(p):
        assert torch.equal(outs.views[r], ref.views[r])
    # in place
    ccl.ccl_allreduce_static(p, ins.ptrs(), ins.ptrs(), op, dtype, n, sched, stream_ptr())
    torch.cuda.synchronize()
    for r in range(p):
        assert torch.equal(ins.views[r], ref.views[r])


def test_static_entry_rejects_what_it_cannot_take():
    p, n = 4, 4 * 1001                        # chunks of 1001 bf16: not 16-byte aligned
    xs = _inputs("bf16", p, n, seed=71)
    ins = RankBuffers(xs, n, np.uint16)
    outs = RankBuffers(None, n, np.uint16, p=p)
    with pytest.raises(ccl.CclError) as ei:
        ccl.ccl_allreduce_static(p, ins.ptrs(), outs.ptrs(), "sum", "bf16", n, "ring", stream_ptr())
    assert ei.value.status == ccl.CCL_ERR_UNSUPPORTED
    with pytest.raises(ccl.CclError) as ei:       # outputs overlapping each other
        ccl.ccl_allreduce_static(p, ins.ptrs(), [outs.ptr(0)] * p, "sum", "bf16", n - 4, "ring", stream_ptr())
    assert ei.value.status == ccl.CCL_ERR_INVALID_ARG
    with pytest.raises(ccl.CclError) as ei:
        ccl.ccl_allreduce_static(65, (ins.ptrs() * 17)[:65], (outs.ptrs() * 17)[:65], "sum", "bf16", 0, "ring", stream_ptr())
    assert ei.value.status == ccl.CCL_ERR_INVALID_ARG
    with pytest.raises(ccl.CclError) as ei:
        ccl.ccl_allreduce_static(p, ins.ptrs(), outs.ptrs(), "sum", "bf16", n - 4, "custom", stream_ptr())
    assert ei.value.status == ccl.CCL_ERR_INVALID_ARG
