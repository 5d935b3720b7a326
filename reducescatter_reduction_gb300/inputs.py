"""Seeded synthetic rank buffers for the collectives' workloads.

This module only draws random numbers and stores them in the element type; it
holds none of the reduction's arithmetic.  Both the CUDA path's tests/benchmark
and the CPU oracle's tests take their inputs from here.

Every rank r of a workload with seed s draws from ``numpy.random.default_rng([s, r])``.
Normals are drawn in float32 and stored as the element type with
round-to-nearest-even (numpy for fp16, torch's CPU cast for bf16).

Workloads (the shapes of the pages' measurements: nccl-tests style message
sweeps and tensor-parallel activations, see "MSCCL++" evaluation and T-CCL
section "Experimental Setup"):

============  =========================================================  ======
name          buffers                                                    seed
============  =========================================================  ======
worked        p=2, n=4096 fp32, uniform ints in [-8, 8]; elements 0..3   1
              of ranks 0/1 are the all-reduce worked example
sweep         p=8 bf16, n = 2^9 .. 2^27 per rank (1 KiB .. 256 MiB), N(0,1)  2
tp            p=8 bf16, [tokens, 8192], tokens in {1, 32, 256, 4096},    3
              N(0, 0.02)
coverage      p=8, n = 64 Mi; int32 uniform in [-1000, 1000] (prod: values  4
              from {-1, 1, 2}); fp32 / fp16 N(0, 1)
moe           p=16 bf16, [16384, 7168] per rank, N(0, 1)                 5
============  =========================================================  ======

Parity-only recipes whose results depend on the rank order of every chunk,
so that a test comparing bits also checks the order (N(0,1) at bf16 or fp16
hides it: the fp32 sum of a few such values is almost always exact):

- ``cancel``: at each element two ranks (the same draw for every rank) hold
  +B and -B, B a large number with a random significand; every other rank
  holds a small normal value.  Whether a small value still counts in the
  result depends on where it falls relative to the two large ones.
- ``signed_zero``: +0 everywhere except that rank e mod p holds -0 at element
  e; min and max keep whichever zero they meet first.
- ``prod_inexact``: random signs times uniform values in [0.75, 1.3), whose
  products are inexact in fp32 and in the element type.
- ``prod_overflow``: at each element two ranks hold about 2^100 and one
  holds about 2^-100, the rest values near 1; some orders take the fp32
  product past the largest finite value, others never.  bf16 and fp32 only.
"""
from __future__ import annotations

import numpy as np

# element storage: fp16 and bf16 are kept as raw 16-bit patterns
STORAGE = {"f32": np.float32, "f16": np.uint16, "bf16": np.uint16, "i32": np.int32}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "i32": 4}

SEEDS = {"worked": 1, "sweep": 2, "tp": 3, "coverage": 4, "moe": 5}

# The all-reduce worked example ("Inside NCCL AllReduce", "What all-reduce promises").
WORKED_A = [8.0, 0.0, 4.0, 2.0]
WORKED_B = [0.0, 4.0, 8.0, 6.0]

SWEEP_N = [1 << k for k in range(9, 28)]        # bf16 elements per rank: 1 KiB .. 256 MiB
TP_HIDDEN = 8192
TP_TOKENS = [1, 32, 256, 4096]
COVERAGE_N = 64 * 1024 * 1024
MOE_SHAPE = (16384, 7168)


def rng(seed: int, rank: int) -> np.random.Generator:
    return np.random.default_rng([seed, rank])


def store(vals_f32: np.ndarray, dtype: str) -> np.ndarray:
    """Store float32 values as the element type (RNE), returning raw storage."""
    vals_f32 = np.ascontiguousarray(vals_f32, dtype=np.float32)
    if dtype == "f32":
        return vals_f32
    if dtype == "f16":
        return vals_f32.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        import torch
        t = torch.from_numpy(vals_f32).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    if dtype == "i32":
        return vals_f32.astype(np.int32)
    raise ValueError(dtype)


def normal(n: int, seed: int, rank: int, sigma: float, dtype: str) -> np.ndarray:
    v = rng(seed, rank).standard_normal(n, dtype=np.float32)
    if sigma != 1.0:
        v *= np.float32(sigma)
    return store(v, dtype)


def uniform_int(n: int, seed: int, rank: int, lo: int, hi: int, dtype: str) -> np.ndarray:
    v = rng(seed, rank).integers(lo, hi + 1, size=n, dtype=np.int32)
    if dtype == "i32":
        return v
    return store(v.astype(np.float32), dtype)


def choice(n: int, seed: int, rank: int, values, dtype: str) -> np.ndarray:
    vals = np.asarray(values, dtype=np.int32)
    v = vals[rng(seed, rank).integers(0, len(vals), size=n)]
    if dtype == "i32":
        return v
    return store(v.astype(np.float32), dtype)


# IEEE special values of the 16-bit float types, as bit patterns: +0 and -0,
# the smallest and the largest subnormal, the smallest normal, 1 and the next
# value above it, the largest finite value, infinity, and the quiet NaN of the
# conversions' canonical form -- each with both signs.
SPECIAL_BITS = {
    "f16": [0x0000, 0x0001, 0x03FF, 0x0400, 0x3C00, 0x3C01, 0x7BFF, 0x7C00, 0x7E00],
    "bf16": [0x0000, 0x0001, 0x007F, 0x0080, 0x3F80, 0x3F81, 0x7F7F, 0x7F80, 0x7FC0],
}


def specials(n: int, seed: int, rank: int, dtype: str, nan: bool = True) -> np.ndarray:
    """Raw 16-bit patterns drawn uniformly from SPECIAL_BITS[dtype] and their
    negatives (NaN left out when ``nan`` is false).  Few distinct values, so
    ties (and +0 against -0) are frequent."""
    vals = [b for b in SPECIAL_BITS[dtype] if nan or b not in (0x7E00, 0x7FC0)]
    table = np.asarray(vals + [b | 0x8000 for b in vals], dtype=np.uint16)
    return table[rng(seed, rank).integers(0, len(table), size=n)]


def worked(p: int = 2, n: int = 4096):
    """Uniform ints in [-8, 8] as fp32; ranks 0 and 1 start with the worked example."""
    xs = [uniform_int(n, SEEDS["worked"], r, -8, 8, "f32") for r in range(p)]
    m = min(4, n)
    xs[0][:m] = np.asarray(WORKED_A[:m], dtype=np.float32)
    if p > 1:
        xs[1][:m] = np.asarray(WORKED_B[:m], dtype=np.float32)
    return xs


def sweep(n: int, p: int = 8, dtype: str = "bf16"):
    return [normal(n, SEEDS["sweep"], r, 1.0, dtype) for r in range(p)]


def tp(tokens: int, p: int = 8, hidden: int = TP_HIDDEN, dtype: str = "bf16"):
    return [normal(tokens * hidden, SEEDS["tp"], r, 0.02, dtype) for r in range(p)]


def coverage(op: str, dtype: str, n: int = COVERAGE_N, p: int = 8):
    s = SEEDS["coverage"]
    if dtype == "i32":
        if op == "prod":
            return [choice(n, s, r, [-1, 1, 2], "i32") for r in range(p)]
        return [uniform_int(n, s, r, -1000, 1000, "i32") for r in range(p)]
    return [normal(n, s, r, 1.0, dtype) for r in range(p)]


def moe(p: int = 16, shape=MOE_SHAPE, dtype: str = "bf16"):
    n = shape[0] * shape[1]
    return [normal(n, SEEDS["moe"], r, 1.0, dtype) for r in range(p)]


# ---------------------------------------------------------------------------
# order-revealing parity inputs (see the module docstring)
# ---------------------------------------------------------------------------

_LAYOUT_RANK = 1 << 20   # the stream shared by every rank of a workload (element placement)


def _two_ranks(n: int, seed: int, p: int):
    """Per element, two distinct ranks j != m, drawn from the shared stream."""
    g = rng(seed, _LAYOUT_RANK)
    j = g.integers(0, p, size=n)
    m = (j + 1 + g.integers(0, max(p - 1, 1), size=n)) % p
    return g, j, m


def cancel(n: int, seed: int, rank: int, p: int, dtype: str) -> np.ndarray:
    big_exp, small_scale = (14, 0.25) if dtype == "f16" else (24, 1.0)
    g, j, m = _two_ranks(n, seed, p)
    big = (1.0 + g.random(n, dtype=np.float32)) * np.float32(2.0 ** big_exp)
    v = rng(seed, rank).standard_normal(n, dtype=np.float32) * np.float32(small_scale)
    v = np.where(j == rank, big, np.where(m == rank, -big, v)).astype(np.float32)
    return store(v, dtype)


def cancel_ranks(n: int, seed: int, p: int, dtype: str):
    """All p ranks of ``cancel`` at once (the same arrays, the layout drawn once)."""
    big_exp, small_scale = (14, 0.25) if dtype == "f16" else (24, 1.0)
    g, j, m = _two_ranks(n, seed, p)
    big = (1.0 + g.random(n, dtype=np.float32)) * np.float32(2.0 ** big_exp)
    out = []
    for r in range(p):
        v = rng(seed, r).standard_normal(n, dtype=np.float32) * np.float32(small_scale)
        v[j == r] = big[j == r]
        v[m == r] = -big[m == r]
        out.append(store(v, dtype))
    return out


def signed_zero(n: int, rank: int, p: int, dtype: str) -> np.ndarray:
    v = np.zeros(n, dtype=np.float32)
    v[(np.arange(n) % p) == rank] = -0.0
    return store(v, dtype)


def prod_inexact(n: int, seed: int, rank: int, dtype: str) -> np.ndarray:
    g = rng(seed, rank)
    mag = np.float32(0.75) + np.float32(0.55) * g.random(n, dtype=np.float32)
    sign = np.where(g.random(n) < 0.5, np.float32(-1.0), np.float32(1.0))
    return store((mag * sign).astype(np.float32), dtype)


def prod_overflow(n: int, seed: int, rank: int, p: int, dtype: str) -> np.ndarray:
    if dtype not in ("f32", "bf16"):
        raise ValueError("prod_overflow needs the fp32 exponent range (f32 or bf16)")
    g, j, m = _two_ranks(n, seed, p)
    i = (m + 1 + g.integers(0, max(p - 2, 1), size=n)) % p   # a third rank: i != m
    i = np.where(i == j, (i + 1) % p, i)                       # ... and i != j when p > 2
    big = (1.0 + g.random(n, dtype=np.float32)) * np.float32(2.0 ** 100)
    tiny = (1.0 + g.random(n, dtype=np.float32)) * np.float32(2.0 ** -100)
    v = prod_inexact(n, seed, rank, "f32")
    v = np.where((j == rank) | (m == rank), big, np.where(i == rank, tiny, v)).astype(np.float32)
    return store(v, dtype)
