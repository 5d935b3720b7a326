"""Pins for the CPU oracle, against facts that do not come from the oracle.

Each test checks the oracle against something the pages or the mathematics fix:
the all-reduce worked example, the ring's per-chunk order read off the pages'
state tables, closed forms, exact integer arithmetic, an fp64 error bound,
library conversions (numpy fp16, torch bf16), and the collectives' invariants.
"""
import itertools
import math

import numpy as np
import pytest

import oracle
from reducescatter_reduction_gb300 import inputs
from conftest import golden_orders, read_golden

pytestmark = pytest.mark.cpu


def f32(vals):
    return np.asarray(vals, dtype=np.float32)


def to_storage(vals, dtype):
    return inputs.store(np.asarray(vals, dtype=np.float32), dtype)


def as_float(arr, dtype):
    """Decode raw storage to float64 with library routines (numpy / torch)."""
    if dtype == "f32":
        return arr.astype(np.float64)
    if dtype == "f16":
        return arr.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        import torch
        return torch.from_numpy(arr.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    return arr.astype(np.float64)


# ---------------------------------------------------------------------------
# worked example
# ---------------------------------------------------------------------------

def test_worked_example_two_ranks():
    rows = {r[0]: [float(v) for v in r[1:]] for r in read_golden("worked_example.txt")}
    xs = [f32(rows["rank0"]), f32(rows["rank1"])]
    for sched in ("ring", "allpairs"):
        ys = oracle.allreduce(xs, "sum", "f32", sched)
        for y in ys:
            assert y.tolist() == rows["result"]


def test_worked_example_inside_workload():
    rows = {r[0]: [float(v) for v in r[1:]] for r in read_golden("worked_example.txt")}
    xs = inputs.worked()
    assert xs[0][:4].tolist() == rows["rank0"] and xs[1][:4].tolist() == rows["rank1"]
    ys = oracle.allreduce(xs, "sum", "f32", "ring")
    assert ys[0][:4].tolist() == rows["result"]
    assert np.array_equal(ys[0], ys[1])
    # integer-valued fp32 with |partial| <= 16: every fp32 sum is exact
    exact = xs[0].astype(np.int64) + xs[1].astype(np.int64)
    assert np.array_equal(ys[0].astype(np.int64), exact)


# ---------------------------------------------------------------------------
# accumulation order, observed through the numbers
# ---------------------------------------------------------------------------

def _triple_probe(p, dtype):
    """Element e of chunk c probes one ordered triple (i, j, m): rank j holds
    +B, rank m holds -B, rank i holds a small s, the rest 0.  In an fp32 fold
    the small value survives only if it is added after both +B and -B have
    cancelled: s next to B is absorbed (B + s rounds back to B)."""
    if dtype == "f16":
        # fp32 spacing is 2^-8 just above 2^15 and 2^-9 just below it, so both
        # 2^15 + 2^-10 and 2^15 - 2^-10 round back to 2^15
        big, small = 2.0 ** 15, 2.0 ** -10
    else:
        big, small = 2.0 ** 30, 1.0            # fp32 spacing: 128 above 2^30, 64 below
    triples = list(itertools.permutations(range(p), 3))
    T = len(triples)
    n = p * T
    vals = np.zeros((p, n), dtype=np.float32)
    for c in range(p):
        for t, (i, j, m) in enumerate(triples):
            e = c * T + t
            vals[j, e], vals[m, e], vals[i, e] = big, -big, small
    return triples, n, [to_storage(v, dtype) for v in vals]


def _survives(order, i, j, m):
    pos = {r: k for k, r in enumerate(order)}
    return pos[i] > pos[j] and pos[i] > pos[m]


@pytest.mark.parametrize("fixture,p,sched", [
    ("ring_order_p3.txt", 3, "ring"),
    ("ring_order_p4.txt", 4, "ring"),
    ("ring_order_p8.txt", 8, "ring"),
    ("allpairs_order_p8.txt", 8, "allpairs"),
])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("op", ["sum", "avg"])
def test_order_pin_sum(fixture, p, sched, dtype, op):
    expected = golden_orders(fixture)
    triples, n, xs = _triple_probe(p, dtype)
    T = len(triples)
    y = as_float(oracle.allreduce(xs, op, dtype, sched)[0], dtype)
    for c in range(p):
        got = y[c * T:(c + 1) * T] != 0
        want = np.array([_survives(expected[c], *t) for t in triples])
        assert np.array_equal(got, want), f"chunk {c}"


@pytest.mark.parametrize("fixture,p,sched", [
    ("ring_order_p3.txt", 3, "ring"),
    ("ring_order_p4.txt", 4, "ring"),
    ("ring_order_p8.txt", 8, "ring"),
    ("allpairs_order_p8.txt", 8, "allpairs"),
])
@pytest.mark.parametrize("op", ["min", "max"])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_order_pin_first_rank(fixture, p, sched, op, dtype):
    """+0 and -0 compare equal, so min/max keep whichever zero came first:
    the sign of the result names the first rank of the chunk's order (the
    position the sum probe cannot see, since x + y == y + x)."""
    expected = golden_orders(fixture)
    n = p * p
    vals = np.zeros((p, n), dtype=np.float32)
    for c in range(p):
        for j in range(p):
            vals[j, c * p + j] = -0.0
    xs = [to_storage(v, dtype) for v in vals]
    y = as_float(oracle.allreduce(xs, op, dtype, sched)[0], dtype)
    for c in range(p):
        for j in range(p):
            neg = math.copysign(1.0, y[c * p + j]) < 0
            assert neg == (expected[c][0] == j), (c, j)


@pytest.mark.parametrize("p", [3, 5, 8])
@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_order_pin_custom_tables(p, dtype):
    """The explicit-order entry folds each chunk in exactly the order given:
    random permutation tables, observed through the same absorption probe."""
    rng = np.random.default_rng(p)
    table = [list(rng.permutation(p)) for _ in range(p)]
    triples, n, xs = _triple_probe(p, dtype)
    T = len(triples)
    y = as_float(oracle.allreduce_orders(xs, "sum", dtype, table)[0], dtype)
    for c in range(p):
        got = y[c * T:(c + 1) * T] != 0
        want = np.array([_survives(table[c], *t) for t in triples])
        assert np.array_equal(got, want), f"chunk {c}"
    # first position, through the signed-zero probe
    vals = np.zeros((p, p * p), dtype=np.float32)
    for c in range(p):
        for j in range(p):
            vals[j, c * p + j] = -0.0
    y = as_float(oracle.allreduce_orders([to_storage(v, dtype) for v in vals], "min", dtype, table)[0], dtype)
    for c in range(p):
        for j in range(p):
            assert (math.copysign(1.0, y[c * p + j]) < 0) == (table[c][0] == j)


def test_custom_orders_reject_non_permutations():
    xs = [np.zeros(6, dtype=np.float32)] * 3
    with pytest.raises(ValueError):
        oracle.allreduce_orders(xs, "sum", "f32", [[0, 1, 2], [1, 1, 2], [2, 0, 1]])


def test_chunk_order_listing_matches_fixtures():
    for fixture, p, sched in [("ring_order_p3.txt", 3, "ring"), ("ring_order_p4.txt", 4, "ring"),
                              ("ring_order_p8.txt", 8, "ring"),
                              ("allpairs_order_p8.txt", 8, "allpairs")]:
        for c, order in golden_orders(fixture).items():
            assert oracle.chunk_order(p, sched, c) == order


# ---------------------------------------------------------------------------
# chunking
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("p", [1, 2, 3, 5, 8, 16, 64])
@pytest.mark.parametrize("n", [0, 1, 7, 64, 1000, 4096, 4097])
def test_chunk_bounds_partition(p, n):
    bounds = [oracle.chunk_bounds(p, n, c) for c in range(p)]
    assert bounds[0][0] == 0 and bounds[-1][1] == n
    for (b0, e0), (b1, e1) in zip(bounds, bounds[1:]):
        assert e0 == b1
    sizes = [e - b for b, e in bounds]
    assert max(sizes) - min(sizes) <= 1
    assert sizes == sorted(sizes, reverse=True)      # the larger chunks come first
    if n % p == 0:
        assert all(s == n // p for s in sizes)


# ---------------------------------------------------------------------------
# exact arithmetic: brute force against Python integers
# ---------------------------------------------------------------------------

def _wrap32(v):
    v &= 0xFFFFFFFF
    return v - (1 << 32) if v >= (1 << 31) else v


def _exact_int(vals, op, p):
    if op == "sum":
        return _wrap32(sum(vals))
    if op == "prod":
        return _wrap32(math.prod(vals))
    if op == "min":
        return min(vals)
    if op == "max":
        return max(vals)
    s = _wrap32(sum(vals))                           # avg: integer division toward zero
    q = abs(s) // p
    return q if s >= 0 else -q


@pytest.mark.parametrize("p", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("op", ["sum", "prod", "min", "max", "avg"])
@pytest.mark.parametrize("sched", ["ring", "allpairs"])
def test_int32_brute_force(p, op, sched):
    rng = np.random.default_rng(100 + p)
    for n in (0, 1, 2, 3, 17, 67):
        if op == "prod":
            xs = [rng.choice(np.array([-3, -1, 1, 2, 5], dtype=np.int32), n) for _ in range(p)]
        else:
            xs = [rng.integers(-(2 ** 31), 2 ** 31, n, dtype=np.int64).astype(np.int32)
                  for _ in range(p)]
        ys = oracle.allreduce(xs, op, "i32", sched)
        for e in range(n):
            want = _exact_int([int(x[e]) for x in xs], op, p)
            for y in ys:
                assert int(y[e]) == want


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("op", ["sum", "prod", "min", "max"])
@pytest.mark.parametrize("p", [1, 2, 3, 5, 8])
def test_float_small_integers_exact(dtype, op, p):
    """Small integers: every fp32 partial is exact, so the result is the exact
    integer whatever the order; a wrong operand or op shows up at once."""
    rng = np.random.default_rng(7 * p)
    n = 67
    lo, hi = (-3, 3) if op == "prod" else (-100, 100)
    ints = [rng.integers(lo, hi + 1, n) for _ in range(p)]
    xs = [to_storage(v, dtype) for v in ints]
    for sched in ("ring", "allpairs"):
        y = as_float(oracle.allreduce(xs, op, dtype, sched)[0], dtype)
        for e in range(n):
            vals = [int(v[e]) for v in ints]
            want = {"sum": sum, "prod": math.prod, "min": min, "max": max}[op](vals)
            # bf16 keeps 8 significant bits: the exact integer rounded once (RNE)
            want_f = float(as_float(to_storage([want], dtype), dtype)[0])
            assert y[e] == want_f, (e, vals)


def test_int32_wraparound():
    big = np.array([2 ** 31 - 1, -(2 ** 31), 65536], dtype=np.int32)
    xs = [big.copy(), big.copy()]
    y = oracle.allreduce(xs, "sum", "i32")[0]
    assert y.tolist() == [-2, 0, 131072]
    y = oracle.allreduce(xs, "prod", "i32")[0]
    assert y.tolist() == [1, 0, 0]                   # (2^31-1)^2 = 1 mod 2^32; 2^32 = 0


# ---------------------------------------------------------------------------
# error bound against an exact fp64 sum (math.fsum)
# ---------------------------------------------------------------------------

U_OUT = {"f32": 2.0 ** -24, "bf16": 2.0 ** -8, "f16": 2.0 ** -11}
SUB_ABS = {"f32": 2.0 ** -150, "bf16": 2.0 ** -134, "f16": 2.0 ** -25}


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("op", ["sum", "avg"])
@pytest.mark.parametrize("p", [2, 3, 8, 16])
def test_float_sum_error_bound(dtype, op, p):
    """Recursive fp32 summation of p terms errs by at most
    gamma_{p-1} * sum|x_k| (Higham, Accuracy and Stability of Numerical
    Algorithms, section 4.2); the one rounding to the output type adds at most
    u_out * |acc|.  A dropped or sign-flipped term breaks this at once."""
    n = 4096
    xs = [inputs.normal(n, 11, r, 1.0, dtype) for r in range(p)]
    xf = [as_float(x, dtype) for x in xs]
    u = 2.0 ** -24
    scale = float(np.float32(1.0) / np.float32(p)) if op == "avg" else 1.0
    for sched in ("ring", "allpairs"):
        y = as_float(oracle.allreduce(xs, op, dtype, sched)[0], dtype)
        for e in range(n):
            terms = [v[e] * scale for v in xf]
            exact = math.fsum(terms)
            absum = math.fsum(abs(t) for t in terms)
            gamma = (p - 1) * u / (1 - (p - 1) * u) + (u if op == "avg" else 0.0)
            d1 = gamma * absum
            bound = d1 + U_OUT[dtype] * (abs(exact) + d1) + SUB_ABS[dtype]
            assert abs(y[e] - exact) <= bound, (e, y[e], exact, bound)


def test_float_prod_relative_error():
    p, n = 8, 2048
    xs = [inputs.normal(n, 12, r, 1.0, "f32") for r in range(p)]
    y = oracle.allreduce(xs, "prod", "f32")[0].astype(np.float64)
    exact = np.prod(np.stack([x.astype(np.float64) for x in xs]), axis=0)
    rel = np.abs(y - exact) / np.abs(exact)
    assert np.all(rel <= (p - 1) * 2.0 ** -24 * 1.0001)


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("p", [1, 2, 4, 8, 16])
def test_constant_buffers(dtype, p):
    n = 100
    c = 1.5
    xs = [to_storage(np.full(n, c), dtype) for _ in range(p)]
    for sched in ("ring", "allpairs"):
        out = {op: as_float(oracle.allreduce(xs, op, dtype, sched)[0], dtype)
               for op in ("sum", "prod", "min", "max", "avg")}
        assert np.all(out["sum"] == p * c)
        assert np.all(out["min"] == c) and np.all(out["max"] == c)
        assert np.all(out["avg"] == c)               # p a power of two: 1/p is exact
        want_prod = float(as_float(to_storage([c ** p], dtype), dtype)[0])
        assert np.all(out["prod"] == want_prod)


def test_avg_identical_buffers_p3_within_rounding():
    x = inputs.normal(1000, 13, 0, 1.0, "f32")
    y = oracle.allreduce([x, x, x], "avg", "f32")[0].astype(np.float64)
    assert np.all(np.abs(y - x) <= 4 * 2.0 ** -24 * np.abs(x))


def test_int_constant_buffers():
    xs = [np.full(10, -7, dtype=np.int32) for _ in range(8)]
    assert np.all(oracle.allreduce(xs, "sum", "i32")[0] == -56)
    assert np.all(oracle.allreduce(xs, "avg", "i32")[0] == -7)
    assert np.all(oracle.allreduce(xs, "prod", "i32")[0] == (-7) ** 8)


# ---------------------------------------------------------------------------
# conversions against library routines
# ---------------------------------------------------------------------------

def test_f16_decode_all_patterns():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = pats.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_to_f32(h) for h in pats.tolist()], dtype=np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def _edge_f32():
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32)
    vals = list(bits.view(np.float32))
    # halfway cases and range ends
    for h in (0x3c00, 0x3c01, 0x7bff, 0x0001, 0x03ff, 0x0400):
        v = float(np.uint16(h).view(np.float16))
        nxt = float(np.uint16(h + 1).view(np.float16))
        vals += [np.float32((v + nxt) / 2), np.float32(v), np.float32(-v)]
    vals += [np.float32(65504), np.float32(65519.99), np.float32(65520), np.float32(1e-8),
             np.float32(2.0 ** -25), np.float32(3 * 2.0 ** -26), np.float32(0.0), np.float32(-0.0),
             np.float32(np.inf), np.float32(-np.inf), np.float32(3.4e38)]
    return np.array(vals, dtype=np.float32)


def test_f16_encode_matches_numpy():
    vals = _edge_f32()
    with np.errstate(over="ignore"):        # values above the fp16 range become +-Inf, as intended
        want = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_f16(v) for v in vals.tolist()], dtype=np.uint16)
    nan = np.isnan(vals)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all(np.isnan(got[nan].view(np.float16)))


def test_bf16_round_trip_matches_torch():
    import torch
    vals = _edge_f32()
    mid = np.array([0x3f808000, 0x3f818000, 0x7f7f8000, 0x00008000, 0x80018000],
                   dtype=np.uint32).view(np.float32)             # exact halfway patterns
    vals = np.concatenate([vals, mid])
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f32_to_bf16(v) for v in vals.tolist()], dtype=np.uint16)
    nan = np.isnan(vals)
    assert np.array_equal(got[~nan], want[~nan])
    pats = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    dec = torch.from_numpy(pats.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    got = np.array([oracle.bf16_to_f32(h) for h in pats.tolist()], dtype=np.float32)
    ok = ~np.isnan(dec)
    assert np.array_equal(got[ok].view(np.uint32), dec[ok].view(np.uint32))


# ---------------------------------------------------------------------------
# invariants of the collectives
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16", "i32"])
@pytest.mark.parametrize("op", ["sum", "prod", "min", "max", "avg"])
@pytest.mark.parametrize("sched", ["ring", "allpairs"])
def test_allgather_of_reducescatter_is_allreduce(dtype, op, sched):
    p, n = 8, 8 * 37
    if dtype == "i32":
        xs = [inputs.uniform_int(n, 21, r, -1000, 1000, "i32") for r in range(p)]
    else:
        xs = [inputs.normal(n, 21, r, 1.0, dtype) for r in range(p)]
    ar = oracle.allreduce(xs, op, dtype, sched)
    rs = oracle.reduce_scatter(xs, op, dtype, sched)
    # AllGather takes rank r's contribution at offset r*n/p of an n-element buffer
    staged = []
    for r in range(p):
        buf = np.zeros(n, dtype=rs[r].dtype)
        buf[r * n // p:(r + 1) * n // p] = rs[r]
        staged.append(buf)
    ag = oracle.all_gather(staged, dtype)
    for r in range(p):
        assert np.array_equal(ag[r].view(np.uint8), ar[r].view(np.uint8))
        assert np.array_equal(ar[r].view(np.uint8), ar[0].view(np.uint8))


def test_allgather_of_identical_buffers_is_identity():
    x = inputs.normal(64, 3, 0, 1.0, "bf16")
    ys = oracle.all_gather([x.copy() for _ in range(4)], "bf16")
    for y in ys:
        assert np.array_equal(y, x)


@pytest.mark.parametrize("op", ["sum", "prod", "min", "max", "avg"])
def test_int_invariant_under_permutation_and_schedule(op):
    p, n = 8, 999
    xs = inputs.coverage(op, "i32", n=n, p=p)
    base = oracle.allreduce(xs, op, "i32", "ring")[0]
    rng = np.random.default_rng(1)
    for _ in range(3):
        perm = rng.permutation(p)
        for sched in ("ring", "allpairs"):
            y = oracle.allreduce([xs[k] for k in perm], op, "i32", sched)[0]
            assert np.array_equal(y, base)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("op", ["min", "max"])
def test_minmax_invariant_under_schedule(dtype, op):
    xs = [inputs.normal(777, 9, r, 1.0, dtype) for r in range(8)]
    a = oracle.allreduce(xs, op, dtype, "ring")[0]
    b = oracle.allreduce(xs, op, dtype, "allpairs")[0]
    assert np.array_equal(a, b)


def test_schedules_differ_only_in_rounding():
    """Ring and all-pairs fold the same terms in different orders: the fp32
    results agree to within the fixed-order bound and do differ somewhere
    (reordering changes the bits: "MSCCL, in depth", "Failure modes").
    (bf16 inputs would not show it: p bf16 values sum exactly in fp32.)"""
    p, n = 8, 1 << 14
    xs = inputs.sweep(n, p, dtype="f32")
    a = oracle.allreduce(xs, "sum", "f32", "ring")[0].astype(np.float64)
    b = oracle.allreduce(xs, "sum", "f32", "allpairs")[0].astype(np.float64)
    absum = sum(np.abs(x.astype(np.float64)) for x in xs)
    assert np.all(np.abs(a - b) <= 2 * (p - 1) * 2.0 ** -24 * absum * 1.001)
    assert np.any(a != b)


@pytest.mark.parametrize("sched", ["ring", "allpairs"])
@pytest.mark.parametrize("p,n", [(5, 5003), (8, 8 * 1000), (3, 2)])
def test_sampled_matches_full(sched, p, n):
    """fp32 inputs, so that a wrong chunk (hence a wrong order) changes bits."""
    xs = [inputs.normal(n, 17, r, 1.0, "f32") for r in range(p)]
    full = oracle.allreduce(xs, "sum", "f32", sched)[0]
    edges = set()
    for c in range(p):
        b, e = oracle.chunk_bounds(p, n, c)
        edges |= {b, max(b, e - 1)}
    idx = np.array(sorted(i for i in edges if i < n) +
                   list(np.random.default_rng(0).integers(0, n, 500)), dtype=np.uint64)
    assert np.array_equal(oracle.allreduce_at(xs, idx, "sum", "f32", sched), full[idx])


def test_reject_bad_arguments():
    xs = [np.zeros(10, dtype=np.float32)] * 3
    with pytest.raises(ValueError):
        oracle.reduce_scatter(xs, "sum", "f32")      # 10 % 3 != 0
    with pytest.raises(ValueError):
        oracle.all_gather(xs, "f32")


def test_empty_buffers():
    xs = [np.zeros(0, dtype=np.uint16)] * 4
    for y in oracle.allreduce(xs, "sum", "bf16"):
        assert y.size == 0


# ---------------------------------------------------------------------------
# alpha-beta cost model
# ---------------------------------------------------------------------------

def test_cost_model_worked_example():
    g = {r[0]: r[1:] for r in read_golden("cost_model_example.txt")}
    p = int(g["p"][0])
    alpha = float(g["alpha_us"][0]) * 1e-6
    bw = float(g["bw_GBps"][0]) * 1e9
    e_ap, e_ring = float(g["eff_allpairs"][0]), float(g["eff_ring"][0])
    nb, want = int(g["speedup_allpairs_at_bytes"][0]), float(g["speedup_allpairs_at_bytes"][1])
    ratio = oracle.time_ring(p, nb, alpha, bw, e_ring) / oracle.time_allpairs(p, nb, alpha, bw, e_ap)
    assert round(ratio, 2) == want
    nb, want = int(g["speedup_ring_at_bytes"][0]), float(g["speedup_ring_at_bytes"][1])
    ratio = oracle.time_allpairs(p, nb, alpha, bw, e_ap) / oracle.time_ring(p, nb, alpha, bw, e_ring)
    assert round(ratio, 1) == want
    lo, hi = 1.0, 1e9                                 # crossover by bisection
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if oracle.time_allpairs(p, mid, alpha, bw, e_ap) < oracle.time_ring(p, mid, alpha, bw, e_ring):
            lo = mid
        else:
            hi = mid
    assert round(lo / 2 ** 20, 1) == float(g["crossover_MiB"][0])


# ---------------------------------------------------------------------------
# the ring run hop by hop (partials in the element type)
# ---------------------------------------------------------------------------

def test_ring_stepwise_worked_case():
    rows = {r[0]: [float(v) for v in r[1:]] for r in read_golden("ring_stepwise_bf16_p3.txt")}
    xs = [to_storage(rows[f"rank{k}"], "bf16") for k in range(3)]
    step = as_float(oracle.allreduce_ring_stepwise(xs, "sum", "bf16")[0], "bf16")
    fused = as_float(oracle.allreduce(xs, "sum", "bf16", "ring")[0], "bf16")
    assert step.tolist() == rows["stepwise"]
    assert fused.tolist() == rows["fused"]


@pytest.mark.parametrize("fixture,p", [("ring_order_p3.txt", 3), ("ring_order_p4.txt", 4),
                                       ("ring_order_p8.txt", 8)])
def test_ring_stepwise_order_pin(fixture, p):
    """fp32 partials are fp32 either way, so the absorption probe sees the
    page's ring order through the stepwise path too."""
    expected = golden_orders(fixture)
    triples, n, xs = _triple_probe(p, "f32")
    T = len(triples)
    y = oracle.allreduce_ring_stepwise(xs, "sum", "f32")[0]
    for c in range(p):
        got = y[c * T:(c + 1) * T] != 0
        want = np.array([_survives(expected[c], *t) for t in triples])
        assert np.array_equal(got, want), f"chunk {c}"


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("p", [2, 5, 8, 16])
def test_ring_stepwise_rounds_each_hop(dtype, p):
    """Each hop rounds once to the element type: the error stays within
    (p-1) roundings of |partial| <= sum|x| (u_out each) plus fp32 terms, and
    small-integer inputs (exact at every hop) give the exact sum."""
    n = 2048
    xs = [inputs.normal(n, 30, r, 1.0, dtype) for r in range(p)]
    xf = np.stack([as_float(x, dtype) for x in xs])
    y = as_float(oracle.allreduce_ring_stepwise(xs, "sum", dtype)[0], dtype)
    exact, absum = xf.sum(axis=0), np.abs(xf).sum(axis=0)
    assert np.all(np.abs(y - exact) <= (p - 1) * U_OUT[dtype] * absum * 1.001 + SUB_ABS[dtype] * p)
    ints = [to_storage(np.random.default_rng(r).integers(-8, 9, n), dtype) for r in range(p)]
    y = as_float(oracle.allreduce_ring_stepwise(ints, "sum", dtype)[0], dtype)
    assert np.array_equal(y, np.stack([as_float(x, dtype) for x in ints]).sum(axis=0))


@pytest.mark.parametrize("dtype", ["f32", "i32"])
@pytest.mark.parametrize("op", ["sum", "prod", "min", "max", "avg"])
def test_ring_stepwise_wide_types_match_fused(dtype, op):
    """fp32 and int32 partials lose nothing between hops: same bits as the
    fused ring fold (and the int32 closed forms)."""
    p, n = 8, 999
    xs = inputs.coverage(op, dtype, n=n, p=p) if dtype == "i32" else [
        inputs.normal(n, 31, r, 1.0, dtype) for r in range(p)]
    a = oracle.allreduce_ring_stepwise(xs, op, dtype)
    b = oracle.allreduce(xs, op, dtype, "ring")
    for r in range(p):
        assert np.array_equal(a[r].view(np.uint8), b[r].view(np.uint8))


# ---------------------------------------------------------------------------
# AllReduce + residual merge + RMSNorm
# ---------------------------------------------------------------------------

def _rms_case(p, rows, hidden, dtype, seed, sigma=0.02):
    xs = [inputs.normal(rows * hidden, seed, r, sigma, dtype) for r in range(p)]
    res = inputs.normal(rows * hidden, seed, 100, 1.0, dtype)
    gamma = inputs.normal(hidden, seed, 200, 1.0, dtype)
    return xs, res, gamma


def test_rmsnorm_closed_form_three_four():
    """A [3, 4] row (after the merge) has RMS 5/sqrt(2): out = [3, 4] * sqrt(2)/5."""
    xs = [to_storage([1.0, 2.0], "f32"), to_storage([2.0, 2.0], "f32")]   # sum = [3, 4]
    res = to_storage([0.0, 0.0], "f32")
    gamma = to_storage([1.0, 1.0], "f32")
    out, h = oracle.allreduce_residual_rmsnorm(xs, res, gamma, 1, 2, "f32", eps=0.0)
    assert h.tolist() == [3.0, 4.0]
    want = np.float32(np.array([3.0, 4.0]) * math.sqrt(2.0) / 5.0)
    assert np.array_equal(out, want)


def test_rmsnorm_mean_square_is_taken_over_the_stored_merge():
    """The norm reads h as stored (rounded to the element type), not the fp32
    merge before rounding.  Hand-checked bf16 row, eps = 0, gamma = 1:
    y = [2.75, 1.0625, 0.0625, -1.875], residual = [-0.0986328125,
    -0.2294921875, -0.21484375, -0.2412109375]; the fp32 merge is
    [2.6513671875, 0.8330078125, -0.15234375, -2.1162109375] and rounds to
    h = [2.65625, 0.83203125, -0.15234375, -2.109375] (bf16 steps 2^-6 in
    [2, 4), 2^-8 in [0.5, 1)).  mean(h^2) = 12.220611572265625 / 4, so
    h0 / rms = 1.51968..., 194.52 steps of 2^-7 -> 1.5234375.  Squaring the
    unrounded merge instead gives 194.50 steps -> 1.515625."""
    xs = [to_storage([2.75, 1.0625, 0.0625, -1.875], "bf16"), to_storage([0.0] * 4, "bf16")]
    res = to_storage([-0.0986328125, -0.2294921875, -0.21484375, -0.2412109375], "bf16")
    ones = to_storage([1.0] * 4, "bf16")
    out, h = oracle.allreduce_residual_rmsnorm(xs, res, ones, 1, 4, "bf16", eps=0.0)
    assert as_float(h, "bf16").tolist() == [2.65625, 0.83203125, -0.15234375, -2.109375]
    assert as_float(out, "bf16").tolist() == [1.5234375, 0.4765625, -0.0869140625, -1.203125]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_rmsnorm_constant_rows_give_sign_times_gamma(dtype):
    p, rows, hidden = 4, 3, 64
    vals = [0.5, -2.0, 1.0]
    xs = [to_storage(np.repeat([v / p for v in vals], hidden), dtype) for _ in range(p)]
    res = to_storage(np.zeros(rows * hidden), dtype)
    gamma = to_storage(np.linspace(-2, 2, hidden), dtype)
    out, h = oracle.allreduce_residual_rmsnorm(xs, res, gamma, rows, hidden, dtype, eps=0.0)
    g = as_float(gamma, dtype)
    o = as_float(out, dtype).reshape(rows, hidden)
    for i, v in enumerate(vals):
        assert np.array_equal(o[i], as_float(to_storage(np.sign(v) * g, dtype), dtype))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rmsnorm_invariants(dtype):
    """Unit gamma and eps = 0: every output row has mean square 1, and scaling
    the inputs and residual by a power of two leaves the output unchanged."""
    p, rows, hidden = 8, 4, 256
    xs, res, _ = _rms_case(p, rows, hidden, dtype, 40)
    ones = to_storage(np.ones(hidden), dtype)
    out, h = oracle.allreduce_residual_rmsnorm(xs, res, ones, rows, hidden, dtype, eps=0.0)
    o = as_float(out, dtype).reshape(rows, hidden)
    tol = 2e-6 if dtype == "f32" else 2e-2
    assert np.all(np.abs((o ** 2).mean(axis=1) - 1.0) < tol)
    xs2 = [to_storage(as_float(x, dtype) * 8.0, dtype) for x in xs]
    res2 = to_storage(as_float(res, dtype) * 8.0, dtype)
    out2, h2 = oracle.allreduce_residual_rmsnorm(xs2, res2, ones, rows, hidden, dtype, eps=0.0)
    assert np.array_equal(out2, out)
    assert np.array_equal(as_float(h2, dtype), as_float(h, dtype) * 8.0)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("sched", ["ring", "allpairs"])
def test_rmsnorm_merge_is_allreduce_plus_residual(dtype, sched):
    """h is the sum AllReduce, rounded, plus the residual, rounded once more."""
    p, rows, hidden = 8, 3, 128
    xs, res, gamma = _rms_case(p, rows, hidden, dtype, 41, sigma=1.0)
    _, h = oracle.allreduce_residual_rmsnorm(xs, res, gamma, rows, hidden, dtype, sched)
    y = as_float(oracle.allreduce(xs, "sum", dtype, sched)[0], dtype)
    want = to_storage(np.float32(y) + np.float32(as_float(res, dtype)), dtype)
    assert np.array_equal(h, want)


def test_rmsnorm_rejects():
    xs = [np.zeros(4, dtype=np.int32)] * 2
    with pytest.raises((ValueError, TypeError)):
        oracle.allreduce_residual_rmsnorm(xs, xs[0], xs[0][:2], 2, 2, "i32")


def test_rmsnorm_closed_form_with_eps():
    """eps enters under the square root: [3, 4] with eps = 0.5 has mean square
    12.5, so out = [3, 4] / sqrt(13)."""
    xs = [to_storage([3.0, 4.0], "f32")]
    res = to_storage([0.0, 0.0], "f32")
    gamma = to_storage([1.0, 1.0], "f32")
    out, _ = oracle.allreduce_residual_rmsnorm(xs, res, gamma, 1, 2, "f32", eps=0.5)
    assert np.array_equal(out, np.float32(np.array([3.0, 4.0]) / math.sqrt(13.0)))


@pytest.mark.parametrize("dtype,one,nan,ninf,sub", [("f16", 0x3C00, 0x7E00, 0xFC00, 0x0001),
                                                      ("bf16", 0x3F80, 0x7FC0, 0xFF80, 0x0001)])
def test_min_max_special_values_follow_compare_and_select(dtype, one, nan, ninf, sub):
    """min/max keep the earlier operand unless the later one compares
    strictly less (greater): +0 against -0 keeps whichever came first, a NaN
    stays only when it comes first, infinities and subnormals order as
    numbers.  All-pairs order folds rank 0 then rank 1."""
    pz, nz = 0x0000, 0x8000
    x0 = np.array([pz, nz, nan, one, ninf, sub, nz | sub, pz], dtype=np.uint16)
    x1 = np.array([nz, pz, one, nan, nz, pz, nz, nan | 0x8000], dtype=np.uint16)
    mn = oracle.allreduce([x0, x1], "min", dtype, "allpairs")[0]
    mx = oracle.allreduce([x0, x1], "max", dtype, "allpairs")[0]
    assert mn.tolist() == [pz, nz, nan, one, ninf, pz, nz | sub, pz]
    assert mx.tolist() == [pz, nz, nan, one, nz, sub, nz, pz]
    # ring order for p = 2: chunk 0 folds rank 1 then rank 0
    ring = oracle.allreduce([x0, x1], "min", dtype, "ring")[0]
    assert ring[:4].tolist() == [nz, pz, one, nan]


def test_special_value_table_holds_what_it_names():
    """The special-value generator's bit patterns decode (numpy for fp16,
    torch for bf16) to the values its table names, and draws cover both
    signs; nan=False leaves NaN out."""
    import torch
    f16 = np.array(inputs.SPECIAL_BITS["f16"], dtype=np.uint16).view(np.float16).astype(np.float64)
    assert f16[:7].tolist() == [0.0, 2.0 ** -24, 1023 * 2.0 ** -24, 2.0 ** -14, 1.0, 1.0 + 2.0 ** -10, 65504.0]
    assert np.isinf(f16[7]) and np.isnan(f16[8])
    bits = torch.tensor(np.array(inputs.SPECIAL_BITS["bf16"], dtype=np.uint16).view(np.int16))
    bf = bits.view(torch.bfloat16).double().numpy()
    assert bf[:7].tolist() == [0.0, 2.0 ** -133, 127 * 2.0 ** -133, 2.0 ** -126, 1.0, 1.0 + 2.0 ** -7,
                               (2.0 - 2.0 ** -7) * 2.0 ** 127]
    assert np.isinf(bf[7]) and np.isnan(bf[8])
    for dtype in ("f16", "bf16"):
        d = inputs.specials(4000, 5, 0, dtype)
        table = set(inputs.SPECIAL_BITS[dtype])
        assert set(d.tolist()) == table | {b | 0x8000 for b in table}
        d = inputs.specials(4000, 5, 0, dtype, nan=False)
        assert not any((b & 0x7FFF) in (0x7E00, 0x7FC0) for b in d.tolist())
