"""GPU tests of the AllReduce fused with the residual merge and RMSNorm:
the merged residual h bit-exact against the oracle, the normalised output
within one unit in the last place of the element type (fp32: 1e-5
relative), identical on every rank."""
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


def decode(arr, dtype):
    if dtype == "f32":
        return arr.astype(np.float64)
    if dtype == "f16":
        return arr.view(np.float16).astype(np.float64)
    return torch.from_numpy(arr.view(np.int16).copy()).view(torch.bfloat16).double().numpy()


def ulp(vals, dtype):
    """Spacing of the element type at |vals| (normal range)."""
    mant = {"f32": 23, "f16": 10, "bf16": 7}[dtype]
    tiny = {"f32": 2.0 ** -126, "f16": 2.0 ** -14, "bf16": 2.0 ** -126}[dtype]
    a = np.maximum(np.abs(vals), tiny)
    return 2.0 ** (np.floor(np.log2(a)) - mant)


def run_fused(xs, res, gamma, rows, hidden, dtype, sched="ring", eps=1e-6, inplace_res=False, inplace_out=False):
    storage = inputs.STORAGE[dtype]
    n = rows * hidden
    ins = RankBuffers(xs, n, storage)
    outs = None if inplace_out else RankBuffers(None, n, storage, p=len(xs))
    r_in = RankBuffers([res], n, storage)
    r_out = r_in if inplace_res else RankBuffers(None, n, storage, p=1)
    g = RankBuffers([gamma], hidden, storage)
    with Comm(ins, outs) as cm:
        ccl.ccl_allreduce_residual_rmsnorm(cm.h, dtype, rows, hidden, r_in.ptr(0), r_out.ptr(0), g.ptr(0),
                                           eps, sched, stream_ptr())
        torch.cuda.synchronize()
        desc = ccl.ccl_comm_last_launch(cm.h)
    res_bufs = ins if inplace_out else outs
    for b in (ins, r_in, r_out, g) + (() if outs is None else (outs,)):
        assert b.guards_intact()
    return res_bufs, r_out, desc


def check(res_bufs, r_out, xs, res, gamma, rows, hidden, dtype, sched, eps=1e-6):
    want_out, want_h = oracle.allreduce_residual_rmsnorm(xs, res, gamma, rows, hidden, dtype, sched, eps)
    assert bits_equal(r_out.host(0), want_h)
    got = decode(res_bufs.host(0), dtype)
    want = decode(want_out, dtype)
    if dtype == "f32":
        assert np.all(np.abs(got - want) <= 1e-5 * np.abs(want) + 1e-30)
    else:
        # the fp32 values differ by ~1e-6 relative, so one rounding to the
        # 16-bit type almost always agrees, and never by more than one ulp
        assert np.all(np.abs(got - want) <= ulp(want, dtype))
        assert np.mean(got == want) > 0.99
    assert res_bufs.identical_across_ranks()


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("tokens", [1, 32, 256])
def test_tp_activation_fused_rmsnorm(dtype, tokens):
    p, hidden = 8, inputs.TP_HIDDEN
    xs = inputs.tp(tokens, p, dtype=dtype)
    res = inputs.normal(tokens * hidden, 3, 100, 1.0, dtype)
    gamma = inputs.normal(hidden, 3, 200, 1.0, dtype)
    res_bufs, r_out, desc = run_fused(xs, res, gamma, tokens, hidden, dtype)
    assert "allreduce_residual_rmsnorm" in desc and "vec=1" in desc
    check(res_bufs, r_out, xs, res, gamma, tokens, hidden, dtype, "ring")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("p,rows,hidden,sched", [(3, 5, 1000, "allpairs"), (8, 7, 1023, "ring"),
                                                 (16, 2, 4096, "allpairs"), (2, 9, 64, "ring"),
                                                 (8, 200, 1023, "ring"), (8, 160, 12288, "allpairs"),
                                                 (3, 400, 1000, "allpairs"), (8, 350, 9216, "ring"),
                                                 (1, 7, 1000, "ring"), (1, 300, 8192, "allpairs")])
def test_fused_rmsnorm_shapes_and_in_place(dtype, p, rows, hidden, sched):
    """Rows below, between one and two times, and above twice the SM count
    take the three CTA shapes (128-thread clusters, 1024-thread CTAs,
    256-thread CTAs with four units per thread); hidden sizes that are not a
    multiple of 8 take the element path, and 12288 bf16 columns need a
    two-CTA cluster per row at 1024 threads."""
    n = rows * hidden
    xs = [inputs.normal(n, 5, r, 0.5, dtype) for r in range(p)]
    res = inputs.normal(n, 5, 100, 1.0, dtype)
    gamma = inputs.normal(hidden, 5, 200, 1.0, dtype)
    for inplace_res, inplace_out in ((False, False), (True, True)):
        res_bufs, r_out, _ = run_fused(xs, res, gamma, rows, hidden, dtype, sched,
                                       inplace_res=inplace_res, inplace_out=inplace_out)
        check(res_bufs, r_out, xs, res, gamma, rows, hidden, dtype, sched)


def test_fused_rmsnorm_prefill_4096_tokens():
    p, hidden, tokens, dtype = 8, inputs.TP_HIDDEN, 4096, "bf16"
    xs = inputs.tp(tokens, p)
    res = inputs.normal(tokens * hidden, 3, 100, 1.0, dtype)
    gamma = inputs.normal(hidden, 3, 200, 1.0, dtype)
    res_bufs, r_out, _ = run_fused(xs, res, gamma, tokens, hidden, dtype)
    check(res_bufs, r_out, xs, res, gamma, tokens, hidden, dtype, "ring")


def test_fused_rmsnorm_statuses():
    p, rows, hidden = 4, 2, 64
    xs = [inputs.normal(rows * hidden, 6, r, 1.0, "f32") for r in range(p)]
    ins = RankBuffers(xs, rows * hidden, np.float32)
    outs = RankBuffers(None, rows * hidden, np.float32, p=p)
    r = RankBuffers([xs[0]], rows * hidden, np.float32)
    g = RankBuffers([xs[0][:hidden].copy()], hidden, np.float32)
    with Comm(ins, outs) as cm:
        def status(*a):
            try:
                ccl.ccl_allreduce_residual_rmsnorm(cm.h, *a)
                return ccl.CCL_OK
            except ccl.CclError as e:
                return e.status
        s = stream_ptr()
        assert status("i32", rows, hidden, r.ptr(0), r.ptr(0), g.ptr(0), 1e-6, "ring", s) == ccl.CCL_ERR_UNSUPPORTED
        assert status("f32", rows, 0, r.ptr(0), r.ptr(0), g.ptr(0), 1e-6, "ring", s) == ccl.CCL_ERR_INVALID_ARG
        assert status("f32", rows, hidden, r.ptr(0), outs.ptr(1), g.ptr(0), 1e-6, "ring", s) == ccl.CCL_ERR_INVALID_ARG
        assert status("f32", rows, hidden, r.ptr(0), r.ptr(0, 1), g.ptr(0), 1e-6, "ring", s) == ccl.CCL_ERR_INVALID_ARG
        assert status("f32", rows, hidden, r.ptr(0), r.ptr(0), g.ptr(0), -1.0, "ring", s) == ccl.CCL_ERR_INVALID_ARG
        assert status("f32", rows, hidden, r.ptr(0), r.ptr(0), outs.ptr(0), 1e-6, "ring", s) == ccl.CCL_ERR_INVALID_ARG
        assert status("f32", 0, hidden, r.ptr(0), r.ptr(0), g.ptr(0), 1e-6, "ring", s) == ccl.CCL_OK
    torch.cuda.synchronize()


def test_fused_rmsnorm_exchange_wait_times_out_and_context_survives():
    """The CTAs of a row exchange their partial sums with a bounded wait.  With
    the stall hook the second CTA of each row withholds its sum: every wait of
    the row runs out (50 ms here), is recorded, and the CTAs finish after a
    second bounded wait;
    ccl_comm_check reports CCL_ERR_TIMEOUT, and the next call, with the hook
    off, gives the oracle's bits.  Nothing traps or faults."""
    p, rows, hidden, dtype = 8, 2, 8192, "bf16"   # decode shape: a cluster of CTAs per row
    n = rows * hidden
    xs = [inputs.cancel(n, 61, r, p, dtype) for r in range(p)]
    res = inputs.normal(n, 62, 0, 0.5, dtype)
    gamma = inputs.normal(hidden, 63, 0, 1.0, dtype)
    storage = inputs.STORAGE[dtype]
    ins = RankBuffers(xs, n, storage)
    outs = RankBuffers(None, n, storage, p=p)
    r_in = RankBuffers([res], n, storage)
    r_out = RankBuffers(None, n, storage, p=1)
    g = RankBuffers([gamma], hidden, storage)
    with Comm(ins, outs) as cm:
        ccl.ccl_comm_set_debug(cm.h, 50_000_000, 1)
        ccl.ccl_allreduce_residual_rmsnorm(cm.h, dtype, rows, hidden, r_in.ptr(0), r_out.ptr(0), g.ptr(0),
                                           1e-6, "ring", stream_ptr())
        torch.cuda.synchronize()
        with pytest.raises(ccl.CclError) as ei:
            ccl.ccl_comm_check(cm.h)
        assert ei.value.status == ccl.CCL_ERR_TIMEOUT
        ccl.ccl_comm_set_debug(cm.h, 0, 0)
        ccl.ccl_allreduce_residual_rmsnorm(cm.h, dtype, rows, hidden, r_in.ptr(0), r_out.ptr(0), g.ptr(0),
                                           1e-6, "ring", stream_ptr())
        torch.cuda.synchronize()
        ccl.ccl_comm_check(cm.h)
    check(outs, r_out, xs, res, gamma, rows, hidden, dtype, "ring")
    for b in (ins, outs, r_in, r_out, g):
        assert b.guards_intact()
