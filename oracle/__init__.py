"""ORACLE -- test infrastructure, not part of the library.

A plain CPU restatement of AllReduce / ReduceScatter / AllGather over p rank
buffers (``oracle.c``), loaded through ctypes.  Only the test suite, the
package entry point's ``smoke()`` check and the benchmark's CPU-baseline /
reference leg may import this module.  It shares no code with the CUDA path
and never imports it.

Every function follows the pages' definitions (see the header of
``oracle.c``): "Inside NCCL AllReduce" (the all-reduce contract, the worked
example, the ring's per-chunk order from the three-GPU state table, the avg
rule) and "MSCCL, in depth" (the all-pairs schedule and the alpha-beta cost
model).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, F16, BF16, I32 = 0, 1, 2, 3
SUM, PROD, MIN, MAX, AVG = 0, 1, 2, 3, 4
RING, ALLPAIRS = 1, 2

DTYPES = {"f32": F32, "f16": F16, "bf16": BF16, "i32": I32}
OPS = {"sum": SUM, "prod": PROD, "min": MIN, "max": MAX, "avg": AVG}
SCHEDULES = {"ring": RING, "allpairs": ALLPAIRS}

# Storage of each dtype in numpy: fp16 and bf16 travel as raw uint16 bits.
NP_STORAGE = {F32: np.float32, F16: np.uint16, BF16: np.uint16, I32: np.int32}


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (plain gcc, no CUDA)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC",
                               "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        u64, i32, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p
        pp = ctypes.POINTER(ctypes.c_void_p)
        L.oracle_allreduce.argtypes = [i32, u64, i32, i32, i32, pp, pp]
        L.oracle_reduce_scatter.argtypes = [i32, u64, i32, i32, i32, pp, pp]
        L.oracle_all_gather.argtypes = [i32, u64, i32, pp, pp]
        L.oracle_allreduce_orders.argtypes = [i32, u64, i32, i32, ctypes.POINTER(ctypes.c_uint8), pp, pp]
        L.oracle_allreduce_ring_stepwise.argtypes = [i32, u64, i32, i32, pp, pp]
        L.oracle_allreduce_residual_rmsnorm.argtypes = [i32, u64, u64, i32, i32, pp, vp, vp,
                                                        ctypes.c_double, vp, vp]
        L.oracle_allreduce_at.argtypes = [i32, u64, i32, i32, i32, pp,
                                          ctypes.POINTER(u64), u64, vp]
        L.oracle_chunk_bounds.argtypes = [i32, u64, i32, ctypes.POINTER(u64), ctypes.POINTER(u64)]
        L.oracle_chunk_bounds.restype = None
        L.oracle_chunk_order.argtypes = [i32, i32, i32, ctypes.POINTER(i32)]
        L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        L.oracle_f32_to_bf16.restype = ctypes.c_uint16
        L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_f32.restype = ctypes.c_float
        L.oracle_f32_to_f16.argtypes = [ctypes.c_float]
        L.oracle_f32_to_f16.restype = ctypes.c_uint16
        L.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_f16_to_f32.restype = ctypes.c_float
        for f in ("oracle_time_ring", "oracle_time_allpairs"):
            getattr(L, f).argtypes = [i32, ctypes.c_double, ctypes.c_double,
                                      ctypes.c_double, ctypes.c_double]
            getattr(L, f).restype = ctypes.c_double
        _lib = L
    return _lib


def _code(table, v):
    return table[v] if isinstance(v, str) else int(v)


def _ptrs(arrs):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def _check_inputs(xs, dt):
    st = NP_STORAGE[dt]
    for a in xs:
        if a.dtype != st or not a.flags.c_contiguous:
            raise TypeError(f"oracle input must be contiguous {np.dtype(st)}")


def allreduce(xs, op, dtype, schedule="ring"):
    """AllReduce of the p arrays ``xs`` (raw storage, see NP_STORAGE).
    Returns p output arrays, one per rank."""
    dt, o, s = _code(DTYPES, dtype), _code(OPS, op), _code(SCHEDULES, schedule)
    _check_inputs(xs, dt)
    n = xs[0].size
    ys = [np.empty(n, dtype=NP_STORAGE[dt]) for _ in xs]
    rc = lib().oracle_allreduce(len(xs), n, dt, o, s, _ptrs(xs), _ptrs(ys))
    if rc:
        raise ValueError("oracle_allreduce rejected its arguments")
    return ys


def allreduce_orders(xs, op, dtype, order):
    """AllReduce with explicit per-chunk orders: order[c][k] is the k-th rank
    folded into chunk c."""
    dt, o = _code(DTYPES, dtype), _code(OPS, op)
    _check_inputs(xs, dt)
    p, n = len(xs), xs[0].size
    flat = [int(v) for row in order for v in row]
    if len(flat) != p * p:
        raise ValueError("order must be p rows of p ranks")
    arr = (ctypes.c_uint8 * (p * p))(*flat)
    ys = [np.empty(n, dtype=NP_STORAGE[dt]) for _ in xs]
    if lib().oracle_allreduce_orders(p, n, dt, o, arr, _ptrs(xs), _ptrs(ys)):
        raise ValueError("oracle_allreduce_orders rejected its arguments")
    return ys


def allreduce_ring_stepwise(xs, op, dtype):
    """The ring run hop by hop, partials held in the element type between hops."""
    dt, o = _code(DTYPES, dtype), _code(OPS, op)
    _check_inputs(xs, dt)
    n = xs[0].size
    ys = [np.empty(n, dtype=NP_STORAGE[dt]) for _ in xs]
    if lib().oracle_allreduce_ring_stepwise(len(xs), n, dt, o, _ptrs(xs), _ptrs(ys)):
        raise ValueError("oracle_allreduce_ring_stepwise rejected its arguments")
    return ys


def allreduce_residual_rmsnorm(xs, residual, gamma, rows, hidden, dtype, schedule="ring", eps=1e-6):
    """AllReduce (sum) + residual merge + RMSNorm; returns (out, residual_out)."""
    dt, s = _code(DTYPES, dtype), _code(SCHEDULES, schedule)
    _check_inputs(list(xs) + [residual, gamma], dt)
    out = np.empty(rows * hidden, dtype=NP_STORAGE[dt])
    res_out = np.empty(rows * hidden, dtype=NP_STORAGE[dt])
    if lib().oracle_allreduce_residual_rmsnorm(len(xs), rows, hidden, dt, s, _ptrs(xs),
                                               residual.ctypes.data, gamma.ctypes.data, float(eps),
                                               out.ctypes.data, res_out.ctypes.data):
        raise ValueError("oracle_allreduce_residual_rmsnorm rejected its arguments")
    return out, res_out


def reduce_scatter(xs, op, dtype, schedule="ring"):
    """ReduceScatter: rank r receives chunk r (n/p elements)."""
    dt, o, s = _code(DTYPES, dtype), _code(OPS, op), _code(SCHEDULES, schedule)
    _check_inputs(xs, dt)
    p, n = len(xs), xs[0].size
    if n % p:
        raise ValueError("reduce_scatter needs n % p == 0")
    ys = [np.empty(n // p, dtype=NP_STORAGE[dt]) for _ in xs]
    rc = lib().oracle_reduce_scatter(p, n, dt, o, s, _ptrs(xs), _ptrs(ys))
    if rc:
        raise ValueError("oracle_reduce_scatter rejected its arguments")
    return ys


def all_gather(xs, dtype):
    """AllGather: rank r contributes chunk r of its own n-element buffer;
    every rank receives all n elements."""
    dt = _code(DTYPES, dtype)
    _check_inputs(xs, dt)
    p, n = len(xs), xs[0].size
    if n % p:
        raise ValueError("all_gather needs n % p == 0")
    ys = [np.empty(n, dtype=NP_STORAGE[dt]) for _ in xs]
    rc = lib().oracle_all_gather(p, n, dt, _ptrs(xs), _ptrs(ys))
    if rc:
        raise ValueError("oracle_all_gather rejected its arguments")
    return ys


def allreduce_at(xs, idx, op, dtype, schedule="ring"):
    """AllReduce output at the element indices ``idx`` only."""
    dt, o, s = _code(DTYPES, dtype), _code(OPS, op), _code(SCHEDULES, schedule)
    _check_inputs(xs, dt)
    idx = np.ascontiguousarray(idx, dtype=np.uint64)
    out = np.empty(idx.size, dtype=NP_STORAGE[dt])
    rc = lib().oracle_allreduce_at(len(xs), xs[0].size, dt, o, s, _ptrs(xs),
                                   idx.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)),
                                   idx.size, out.ctypes.data)
    if rc:
        raise ValueError("oracle_allreduce_at rejected its arguments")
    return out


def chunk_bounds(p, n, c):
    b, e = ctypes.c_uint64(), ctypes.c_uint64()
    lib().oracle_chunk_bounds(p, n, c, ctypes.byref(b), ctypes.byref(e))
    return b.value, e.value


def chunk_order(p, schedule, c):
    arr = (ctypes.c_int * p)()
    if lib().oracle_chunk_order(p, _code(SCHEDULES, schedule), c, arr):
        raise ValueError("bad chunk_order arguments")
    return list(arr)


def f32_to_bf16(v):
    return lib().oracle_f32_to_bf16(float(v))


def bf16_to_f32(h):
    return lib().oracle_bf16_to_f32(int(h))


def f32_to_f16(v):
    return lib().oracle_f32_to_f16(float(v))


def f16_to_f32(h):
    return lib().oracle_f16_to_f32(int(h))


def time_ring(p, nbytes, alpha_s, bw, eff):
    return lib().oracle_time_ring(p, nbytes, alpha_s, bw, eff)


def time_allpairs(p, nbytes, alpha_s, bw, eff):
    return lib().oracle_time_allpairs(p, nbytes, alpha_s, bw, eff)
