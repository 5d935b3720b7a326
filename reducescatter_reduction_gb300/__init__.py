"""Python binding of libccl.so, the C ABI in include/ccl.h.

AllReduce, ReduceScatter and AllGather over p rank buffers resident in one
GPU's memory, computed by hand-written sm_103a kernels.  Every function here
has the name of the C entry point it calls and only marshals arguments:
device pointers and streams are plain integers (``tensor.data_ptr()``,
``torch.cuda.current_stream().cuda_stream``); enum arguments accept the C
value or its name ("sum", "bf16", "ring", ...).  A non-OK status raises
:class:`CclError` carrying the status and ``ccl_last_error()``.

The library is built in-tree by :func:`reducescatter_reduction_gb300.build.build`;
calling any function before it exists raises ``RuntimeError`` (there is no
fallback implementation).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# CCL_LIBRARY names another build of this library to load instead (the
# checked build, libccl_checked.so, for tests)
LIB_PATH = os.environ.get("CCL_LIBRARY") or os.path.join(_HERE, "libccl.so")

CCL_OK, CCL_ERR_INVALID_ARG, CCL_ERR_UNSUPPORTED, CCL_ERR_CUDA, CCL_ERR_TIMEOUT, CCL_ERR_NOMEM, CCL_ERR_BOUNDS = range(7)
CCL_SUM, CCL_PROD, CCL_MIN, CCL_MAX, CCL_AVG = range(5)
CCL_F32, CCL_F16, CCL_BF16, CCL_I32 = range(4)
CCL_SCHED_AUTO, CCL_SCHED_RING, CCL_SCHED_ALLPAIRS, CCL_SCHED_CUSTOM = range(4)
(CCL_VARIANT_AUTO, CCL_VARIANT_LDST, CCL_VARIANT_TMA, CCL_VARIANT_TMA_BULKRED, CCL_VARIANT_RING_STEPWISE,
 CCL_VARIANT_ONE_PHASE) = range(6)
CCL_MAX_RANKS = 64

OPS = {"sum": CCL_SUM, "prod": CCL_PROD, "min": CCL_MIN, "max": CCL_MAX, "avg": CCL_AVG}
DTYPES = {"f32": CCL_F32, "f16": CCL_F16, "bf16": CCL_BF16, "i32": CCL_I32}
SCHEDULES = {"auto": CCL_SCHED_AUTO, "ring": CCL_SCHED_RING, "allpairs": CCL_SCHED_ALLPAIRS,
             "custom": CCL_SCHED_CUSTOM}
VARIANTS = {"auto": CCL_VARIANT_AUTO, "ldst": CCL_VARIANT_LDST, "tma": CCL_VARIANT_TMA,
            "tma_bulkred": CCL_VARIANT_TMA_BULKRED, "ring_stepwise": CCL_VARIANT_RING_STEPWISE,
            "one_phase": CCL_VARIANT_ONE_PHASE}
STATUS_NAMES = {CCL_OK: "CCL_OK", CCL_ERR_INVALID_ARG: "CCL_ERR_INVALID_ARG",
                CCL_ERR_UNSUPPORTED: "CCL_ERR_UNSUPPORTED", CCL_ERR_CUDA: "CCL_ERR_CUDA",
                CCL_ERR_TIMEOUT: "CCL_ERR_TIMEOUT", CCL_ERR_NOMEM: "CCL_ERR_NOMEM", CCL_ERR_BOUNDS: "CCL_ERR_BOUNDS"}

# Every symbol include/ccl.h declares.
EXPORTS = (
    "ccl_comm_create", "ccl_comm_set_outputs", "ccl_comm_set_schedule", "ccl_set_launch", "ccl_comm_set_debug",
    "ccl_comm_destroy", "ccl_comm_check", "ccl_allreduce", "ccl_reduce_scatter", "ccl_all_gather",
    "ccl_allreduce_static", "ccl_allreduce_static_set_debug", "ccl_allreduce_residual_rmsnorm",
    "ccl_schedule_build", "ccl_schedule_check", "ccl_cost_estimate", "ccl_select_schedule", "ccl_launch_estimate",
    "ccl_last_error", "ccl_comm_last_launch", "ccl_comm_launch_count", "ccl_version", "ccl_bounds_checked",
)


class CclError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class CostParams(ctypes.Structure):
    """ccl_cost_params_t."""
    _fields_ = [("alpha_s", ctypes.c_double), ("bw_bytes_per_s", ctypes.c_double),
                ("eff_ring", ctypes.c_double), ("eff_allpairs", ctypes.c_double)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libccl.so and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with reducescatter_reduction_gb300.build.build()")
    L = ctypes.CDLL(path)
    vp, i, sz, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint64
    pvp = ctypes.POINTER(ctypes.c_void_p)
    sigs = {
        "ccl_comm_create": (i, [ctypes.POINTER(vp), i, pvp]),
        "ccl_comm_set_outputs": (i, [vp, pvp]),
        "ccl_comm_set_schedule": (i, [vp, ctypes.POINTER(ctypes.c_uint8)]),
        "ccl_set_launch": (i, [vp, i, i, sz]),
        "ccl_comm_set_debug": (i, [vp, ctypes.c_longlong, i]),
        "ccl_comm_destroy": (i, [vp]),
        "ccl_comm_check": (i, [vp]),
        "ccl_allreduce": (i, [vp, i, i, sz, i, vp]),
        "ccl_reduce_scatter": (i, [vp, i, i, sz, i, vp]),
        "ccl_all_gather": (i, [vp, i, sz, vp]),
        "ccl_allreduce_static": (i, [i, pvp, pvp, i, i, sz, i, vp]),
        "ccl_allreduce_static_set_debug": (i, [ctypes.c_longlong, i]),
        "ccl_allreduce_residual_rmsnorm": (i, [vp, i, sz, sz, vp, vp, vp, ctypes.c_float, i, vp]),
        "ccl_schedule_build": (i, [i, u64, i, ctypes.POINTER(u64), ctypes.POINTER(ctypes.c_uint8)]),
        "ccl_schedule_check": (i, [i, u64, ctypes.POINTER(u64), ctypes.POINTER(ctypes.c_uint8)]),
        "ccl_cost_estimate": (ctypes.c_double, [i, ctypes.c_double, i, ctypes.POINTER(CostParams)]),
        "ccl_select_schedule": (i, [i, ctypes.c_double, ctypes.POINTER(CostParams)]),
        "ccl_launch_estimate": (i, [i, i, i, sz, i, ctypes.POINTER(ctypes.c_double)]),
        "ccl_last_error": (ctypes.c_char_p, []),
        "ccl_comm_last_launch": (i, [vp, ctypes.c_char_p, sz]),
        "ccl_comm_launch_count": (u64, [vp]),
        "ccl_version": (i, []),
        "ccl_bounds_checked": (i, []),
    }
    for name, (res, args) in sigs.items():
        f = getattr(L, name)
        f.restype, f.argtypes = res, args
    _lib = L
    return L


def _code(table, v):
    return table[v] if isinstance(v, str) else int(v)


def _check(status: int):
    if status != CCL_OK:
        raise CclError(status, ccl_last_error())


def _ptr_array(ptrs):
    return (ctypes.c_void_p * len(ptrs))(*[int(x) for x in ptrs])


def _params(params):
    if params is None:
        return None
    if isinstance(params, CostParams):
        return ctypes.byref(params)
    return ctypes.byref(CostParams(*params))


# --------------------------------------------------------------------------
# entry points
# --------------------------------------------------------------------------

def _want_len(ptrs, p: int, what: str):
    # the C side reads exactly p pointers: a shorter list would be read past its end
    if ptrs is not None and len(ptrs) != int(p):
        raise CclError(CCL_ERR_INVALID_ARG, f"{what} has {len(ptrs)} pointers, p = {int(p)}")


def ccl_comm_create(p: int, rank_ptrs) -> int:
    _want_len(rank_ptrs, p, "rank_ptrs")
    h = ctypes.c_void_p()
    _check(load_library().ccl_comm_create(ctypes.byref(h), int(p), _ptr_array(rank_ptrs)))
    return h.value


def ccl_comm_set_outputs(comm: int, out_ptrs=None) -> None:
    arr = None if out_ptrs is None else _ptr_array(out_ptrs)
    _check(load_library().ccl_comm_set_outputs(comm, arr))


def ccl_comm_set_schedule(comm: int, order) -> None:
    flat = [int(v) for row in order for v in (row if hasattr(row, "__len__") else [row])]
    arr = (ctypes.c_uint8 * len(flat))(*flat)
    _check(load_library().ccl_comm_set_schedule(comm, arr))


def ccl_set_launch(comm: int, sm_budget: int = 0, variant=CCL_VARIANT_AUTO,
                   pipeline_chunk_bytes: int = 0) -> None:
    _check(load_library().ccl_set_launch(comm, int(sm_budget), _code(VARIANTS, variant),
                                         int(pipeline_chunk_bytes)))


def ccl_comm_set_debug(comm: int, wait_limit_ns: int = 0, stall_test: int = 0) -> None:
    _check(load_library().ccl_comm_set_debug(comm, int(wait_limit_ns), int(stall_test)))


def ccl_comm_destroy(comm: int) -> None:
    _check(load_library().ccl_comm_destroy(comm))


def ccl_comm_check(comm: int) -> None:
    _check(load_library().ccl_comm_check(comm))


def ccl_allreduce(comm: int, op, dtype, n: int, schedule=CCL_SCHED_AUTO, stream: int = 0) -> None:
    _check(load_library().ccl_allreduce(comm, _code(OPS, op), _code(DTYPES, dtype), int(n),
                                        _code(SCHEDULES, schedule), stream or None))


def ccl_reduce_scatter(comm: int, op, dtype, n: int, schedule=CCL_SCHED_AUTO, stream: int = 0) -> None:
    _check(load_library().ccl_reduce_scatter(comm, _code(OPS, op), _code(DTYPES, dtype), int(n),
                                             _code(SCHEDULES, schedule), stream or None))


def ccl_all_gather(comm: int, dtype, n: int, stream: int = 0) -> None:
    _check(load_library().ccl_all_gather(comm, _code(DTYPES, dtype), int(n), stream or None))


def ccl_allreduce_static(p: int, in_ptrs, out_ptrs, op, dtype, n: int, schedule=CCL_SCHED_AUTO,
                         stream: int = 0) -> None:
    """The allocation-free AllReduce (see include/ccl.h): for callers that may
    not allocate device memory; needs no communicator."""
    _want_len(in_ptrs, p, "in_ptrs")
    _want_len(out_ptrs, p, "out_ptrs")
    _check(load_library().ccl_allreduce_static(int(p), _ptr_array(in_ptrs), _ptr_array(out_ptrs),
                                               _code(OPS, op), _code(DTYPES, dtype), int(n),
                                               _code(SCHEDULES, schedule), stream or None))


def ccl_allreduce_static_set_debug(wait_limit_ns: int = 0, stall_test: int = 0) -> None:
    _check(load_library().ccl_allreduce_static_set_debug(int(wait_limit_ns), int(stall_test)))


def ccl_allreduce_residual_rmsnorm(comm: int, dtype, rows: int, hidden: int, residual_in: int,
                                   residual_out: int, gamma: int, eps: float = 1e-6,
                                   schedule=CCL_SCHED_AUTO, stream: int = 0) -> None:
    _check(load_library().ccl_allreduce_residual_rmsnorm(comm, _code(DTYPES, dtype), int(rows), int(hidden),
                                                         residual_in, residual_out, gamma, float(eps),
                                                         _code(SCHEDULES, schedule), stream or None))


def ccl_schedule_build(p: int, n: int, schedule):
    """Returns (bounds: list of p+1 ints, order: list of p rows of p ranks)."""
    bounds = (ctypes.c_uint64 * (p + 1))()
    order = (ctypes.c_uint8 * (p * p))()
    _check(load_library().ccl_schedule_build(int(p), int(n), _code(SCHEDULES, schedule), bounds, order))
    return list(bounds), [list(order[c * p:(c + 1) * p]) for c in range(p)]


def ccl_schedule_check(p: int, n: int, bounds, order) -> int:
    """Returns the status (CCL_OK or CCL_ERR_INVALID_ARG); does not raise."""
    b = (ctypes.c_uint64 * len(bounds))(*[int(v) for v in bounds])
    flat = [int(v) for row in order for v in row]
    o = (ctypes.c_uint8 * len(flat))(*flat)
    return load_library().ccl_schedule_check(int(p), int(n), b, o)


def ccl_cost_estimate(p: int, nbytes: float, schedule, params=None) -> float:
    return load_library().ccl_cost_estimate(int(p), float(nbytes), _code(SCHEDULES, schedule),
                                            _params(params))


def ccl_select_schedule(p: int, nbytes: float, params=None) -> int:
    return load_library().ccl_select_schedule(int(p), float(nbytes), _params(params))


def ccl_launch_estimate(p: int, dtype, sm_budget: int, bytes_per_rank: int, variant) -> float:
    """The launch table's per-call time estimate (us) for the ld/st or TMA kernel."""
    us = ctypes.c_double()
    _check(load_library().ccl_launch_estimate(int(p), _code(DTYPES, dtype), int(sm_budget), int(bytes_per_rank),
                                              _code(VARIANTS, variant), ctypes.byref(us)))
    return us.value


def ccl_last_error() -> str:
    msg = load_library().ccl_last_error()
    return msg.decode() if msg else ""


def ccl_comm_last_launch(comm: int) -> str:
    buf = ctypes.create_string_buffer(512)
    _check(load_library().ccl_comm_last_launch(comm, buf, len(buf)))
    return buf.value.decode()


def ccl_comm_launch_count(comm: int) -> int:
    return load_library().ccl_comm_launch_count(comm)


def ccl_version() -> int:
    return load_library().ccl_version()


def ccl_bounds_checked() -> bool:
    """True when the loaded library is the checked build (CCL_BOUNDS_CHECK)."""
    return bool(load_library().ccl_bounds_checked())
