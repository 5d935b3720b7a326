"""The checked build's bounds record (include/ccl.h, ccl_bounds_checked):
every kernel tests the extent of each global access it computes against the
rank buffer it addresses, records the first violation in the communicator's
status block and skips the access; ccl_comm_check reports CCL_ERR_BOUNDS.
A violation is made on purpose with the debug hook (the TMA producer's check
of its second tile is made to fail; no access is made), on every variant of
the pipeline.  These tests run only against the checked library: the default
build has no checks (test_zy_checked_build.py runs them against it)."""
import pytest
import torch

import oracle
import reducescatter_reduction_gb300 as ccl
from reducescatter_reduction_gb300 import inputs
from ccl_testutil import Comm, RankBuffers, bits_equal, stream_ptr
from test_parity import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _checked():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ccl.load_library()
    if not ccl.ccl_bounds_checked():
        pytest.skip("the default build has no bounds checks (CCL_LIBRARY selects the checked build)")


@pytest.mark.parametrize("p,budget", [(8, 1), (8, 0), (16, 2), (40, 0)])
def test_bounds_violation_is_recorded_and_the_access_skipped(p, budget):
    n = p * (1 << 17)                     # enough tiles that CTAs reach a second stage
    xs = gen("bf16", "sum", p, n, seed=900 + p)
    storage = inputs.STORAGE["bf16"]
    ins = RankBuffers(xs, n, storage)
    outs = RankBuffers(None, n, storage, p=p)
    with Comm(ins, outs) as cm:
        ccl.ccl_set_launch(cm.h, budget, "tma", 0)
        ccl.ccl_comm_set_debug(cm.h, 20_000_000, 2)
        ccl.ccl_allreduce(cm.h, "sum", "bf16", n, "ring", stream_ptr())
        with pytest.raises(ccl.CclError) as ei:
            ccl.ccl_comm_check(cm.h)
        assert ei.value.status == ccl.CCL_ERR_BOUNDS
        assert "site 3" in str(ei.value)                      # the TMA producer's loads
        ccl.ccl_comm_check(cm.h)                               # reported once, then cleared
        ccl.ccl_comm_set_debug(cm.h, 0, 0)
        ccl.ccl_allreduce(cm.h, "sum", "bf16", n, "ring", stream_ptr())
        ccl.ccl_comm_check(cm.h)
    want = oracle.allreduce(xs, "sum", "bf16", "ring")
    for r in range(p):
        assert bits_equal(outs.host(r), want[r])
    assert ins.guards_intact() and outs.guards_intact()


def test_no_violation_on_every_collective_and_variant():
    """Every kernel family, each with a ragged tail: no record."""
    p, n = 8, 8 * 5000 + 3
    for dtype in ("bf16", "f32"):
        xs = gen(dtype, "sum", p, n, seed=910)
        storage = inputs.STORAGE[dtype]
        ins = RankBuffers(xs, n, storage)
        outs = RankBuffers(None, n, storage, p=p)
        with Comm(ins, outs) as cm:
            for variant, budget in (("ldst", 0), ("ldst", 3), ("ldst", 100)):
                ccl.ccl_set_launch(cm.h, budget, variant, 0)
                ccl.ccl_allreduce(cm.h, "sum", dtype, n, "ring", stream_ptr())
                ccl.ccl_comm_check(cm.h)
        m = p * 4000                                            # 16-byte chunks: TMA and AllGather
        xs = gen(dtype, "sum", p, m, seed=911)
        ins = RankBuffers(xs, m, storage)
        outs = RankBuffers(None, m, storage, p=p)
        with Comm(ins, outs) as cm:
            for variant, budget in (("tma", 0), ("tma", 3), ("tma_bulkred", 0), ("tma_bulkred", 2)):
                ccl.ccl_set_launch(cm.h, budget, variant, 0)
                ccl.ccl_allreduce(cm.h, "sum", dtype, m, "ring", stream_ptr())
                ccl.ccl_comm_check(cm.h)
                ccl.ccl_reduce_scatter(cm.h, "sum", dtype, m, "allpairs", stream_ptr())
                ccl.ccl_comm_check(cm.h)
        with Comm(ins) as cm:                                   # in-place AllGather
            for budget in (0, 3):
                ccl.ccl_set_launch(cm.h, budget, "ldst", 0)
                ccl.ccl_all_gather(cm.h, dtype, m, stream_ptr())
                ccl.ccl_comm_check(cm.h)
        assert ins.guards_intact()
    torch.cuda.synchronize()
