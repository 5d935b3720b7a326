"""ccl_allreduce_static: the AllReduce entry point for callers that may not
allocate device memory.

Such callers include a plug-in running inside an application that owns all
device memory and hands out only the buffers it manages (an inference
server, a framework's memory pool), a process whose memory budget is already
committed, and code that must not meet an out-of-memory failure once it runs.
The entry point needs no communicator.  It keeps the only scratch its kernel
uses, a 16-byte status record, in a static device array of the library.

These tests call it through the C ABI on inputs whose bits depend on every
chunk's rank order (inputs.cancel) and check two calls in a row bit for bit
against the CPU oracle, and against the communicator entry point,
ccl_allreduce, on the same inputs.  They also check that the calls take no
device memory, and that a bounded wait that runs out (made to, through the
test hook) is reported by the next call, which launches nothing, while the
call after it computes the right bits again.  The file sorts last, so a run
that stops at the first failure has run every other test first.
"""
import numpy as np
import pytest
import torch

import oracle
import reducescatter_reduction_gb300 as ccl
from reducescatter_reduction_gb300 import inputs
from ccl_testutil import Comm, RankBuffers, bits_equal, ensure_built, stream_ptr

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
    return [inputs.cancel(n, seed, r, p, dtype) for r in range(p)]


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
    # two calls in a row; each call waits for the work already queued on the
    # stream before it launches, so the two kernels run one after the other
    for (dtype, op, sched, p, n), (xs, ins, outs) in zip(CASES, bufs):
        ccl.ccl_allreduce_static(p, ins.ptrs(), outs.ptrs(), op, dtype, n, sched, stream_ptr())
    torch.cuda.synchronize()
    for (dtype, op, sched, p, n), (xs, ins, outs) in zip(CASES, bufs):
        want = oracle.allreduce(xs, op, dtype, sched)
        other = oracle.allreduce(xs, op, dtype, "allpairs" if sched == "ring" else "ring")
        assert not bits_equal(want[0], other[0])     # the inputs reveal the order
        for r in range(p):
            assert bits_equal(outs.host(r), want[r]), (dtype, op, r)
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
    want = oracle.allreduce(xs, op, dtype, sched)
    ccl.ccl_allreduce_static(p, ins.ptrs(), outs.ptrs(), op, dtype, n, sched, stream_ptr())
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        ccl.ccl_allreduce_static(p, ins.ptrs(), outs.ptrs(), op, dtype, n, sched, stream_ptr())
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before          # a device allocation would take at least a 2 MiB page
    for r in range(p):
        assert bits_equal(outs.host(r), want[r])
    # in place
    ccl.ccl_allreduce_static(p, ins.ptrs(), ins.ptrs(), op, dtype, n, sched, stream_ptr())
    torch.cuda.synchronize()
    for r in range(p):
        assert bits_equal(ins.host(r), want[r])


def test_static_entry_reports_a_wait_that_ran_out_on_the_next_call():
    """The producer withholds its second tile, so a consumer's wait (50 ms
    here) runs out: the kernel records it in the static array and returns.
    The next call reports CCL_ERR_TIMEOUT without launching; the one after
    that runs normally and gives the oracle's bits."""
    dtype, op, sched, p, n = CASES[0]
    xs = _inputs(dtype, p, n, seed=72)
    storage = inputs.STORAGE[dtype]
    ins = RankBuffers(xs, n, storage)
    outs = RankBuffers(None, n, storage, p=p)
    want = oracle.allreduce(xs, op, dtype, sched)
    try:
        ccl.ccl_allreduce_static_set_debug(50_000_000, 1)
        ccl.ccl_allreduce_static(p, ins.ptrs(), outs.ptrs(), op, dtype, n, sched, stream_ptr())
        torch.cuda.synchronize()                  # the kernel gave up and returned: the context is usable
    finally:
        ccl.ccl_allreduce_static_set_debug(0, 0)
    outs.views[0].zero_()
    torch.cuda.synchronize()
    with pytest.raises(ccl.CclError) as ei:
        ccl.ccl_allreduce_static(p, ins.ptrs(), outs.ptrs(), op, dtype, n, sched, stream_ptr())
    assert ei.value.status == ccl.CCL_ERR_TIMEOUT
    torch.cuda.synchronize()
    assert not bool(outs.views[0].any())          # that call launched nothing
    ccl.ccl_allreduce_static(p, ins.ptrs(), outs.ptrs(), op, dtype, n, sched, stream_ptr())
    torch.cuda.synchronize()
    for r in range(p):
        assert bits_equal(outs.host(r), want[r])
    assert outs.guards_intact() and ins.guards_intact()


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
    for bad in ((-1, 0), (0, 2), (0, -1)):
        with pytest.raises(ccl.CclError) as ei:
            ccl.ccl_allreduce_static_set_debug(*bad)
        assert ei.value.status == ccl.CCL_ERR_INVALID_ARG
