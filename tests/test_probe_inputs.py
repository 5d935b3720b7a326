"""The order-revealing parity inputs (inputs.cancel, signed_zero,
prod_inexact, prod_overflow) really reveal the order and the rounding.

The GPU tests in test_order_gpu.py compare the kernels with the oracle bit
for bit on these inputs.  That comparison checks the accumulation order only
if a wrong order would change the bits.  Here, on the CPU, mistakes are
planted in the oracle's order tables -- two neighbouring ranks of one chunk's
order swapped, or the first rank moved -- and in its rounding (the ring run
hop by hop, each partial rounded to the element type: the oracle's stepwise
function), and each must change the result on these inputs.  Sum is
commutative in its first two operands, so swaps start at position 1; the
first position is what the signed-zero input pins through min and max.
"""
import numpy as np
import pytest

import oracle
from reducescatter_reduction_gb300 import inputs

pytestmark = pytest.mark.cpu

FLOATS = ["f32", "f16", "bf16"]


def orders(p, sched, seed=0):
    if sched == "custom":
        rng = np.random.default_rng(1000 + p + seed)
        return [list(rng.permutation(p)) for _ in range(p)]
    return [oracle.chunk_order(p, sched, c) for c in range(p)]


def bits(a):
    return a.view(np.uint32 if a.dtype.itemsize == 4 else np.uint16)


def chunk(y, p, n, c):
    """Chunk c of a result, as raw bits (+0 and -0 differ)."""
    b, e = oracle.chunk_bounds(p, n, c)
    return bits(y[b:e])


def swaps_to_check(p, rng):
    """(chunk, position) pairs: all of them for small p, a sample above."""
    pairs = [(c, k) for c in range(p) for k in range(1, p - 1)]
    if len(pairs) <= 120:
        return pairs
    return [pairs[i] for i in rng.choice(len(pairs), 60, replace=False)]


@pytest.mark.parametrize("dtype", FLOATS)
@pytest.mark.parametrize("p,sched", [(3, "ring"), (4, "allpairs"), (5, "custom"), (8, "ring"),
                                     (8, "allpairs"), (16, "custom"), (17, "ring"), (33, "allpairs")])
@pytest.mark.parametrize("op", ["sum", "avg"])
def test_cancel_reveals_every_neighbour_swap(dtype, p, sched, op):
    n = p * 1024 + (p // 2)                      # ragged: chunk sizes differ by one
    xs = [inputs.cancel(n, 11, r, p, dtype) for r in range(p)]
    base_order = orders(p, sched)
    base = oracle.allreduce_orders(xs, op, dtype, base_order)[0]
    rng = np.random.default_rng(p)
    for c, k in swaps_to_check(p, rng):
        mo = [list(o) for o in base_order]
        mo[c][k], mo[c][k + 1] = mo[c][k + 1], mo[c][k]
        y = oracle.allreduce_orders(xs, op, dtype, mo)[0]
        diff = int(np.count_nonzero(chunk(y, p, n, c) != chunk(base, p, n, c)))
        assert diff >= 4, f"swap at chunk {c}, positions {k},{k + 1}: {diff} elements differ"
        # the swap touches chunk c only
        assert np.array_equal(np.delete(bits(y), np.arange(*oracle.chunk_bounds(p, n, c))),
                              np.delete(bits(base), np.arange(*oracle.chunk_bounds(p, n, c))))


@pytest.mark.parametrize("dtype", FLOATS)
@pytest.mark.parametrize("p,sched", [(2, "ring"), (3, "allpairs"), (8, "custom"), (17, "ring"), (64, "allpairs")])
@pytest.mark.parametrize("op", ["min", "max"])
def test_signed_zero_reveals_the_first_rank(dtype, p, sched, op):
    n = p * 64
    xs = [inputs.signed_zero(n, r, p, dtype) for r in range(p)]
    base_order = orders(p, sched)
    base = oracle.allreduce_orders(xs, op, dtype, base_order)[0]
    for c in range(p):
        mo = [list(o) for o in base_order]
        mo[c] = mo[c][1:] + mo[c][:1]            # a different first rank, same set
        y = oracle.allreduce_orders(xs, op, dtype, mo)[0]
        assert int(np.count_nonzero(chunk(y, p, n, c) != chunk(base, p, n, c))) >= 2


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("p", [3, 8, 16])
def test_prod_inexact_reveals_per_hop_rounding(dtype, p):
    """A kernel that rounded the partial product to the element type at every
    step would compute the stepwise ring's result; on these inputs that
    differs from the fused result in a large share of the elements."""
    n = p * 512
    xs = [inputs.prod_inexact(n, 12, r, dtype) for r in range(p)]
    fused = oracle.allreduce(xs, "prod", dtype, "ring")[0]
    stepwise = oracle.allreduce_ring_stepwise(xs, "prod", dtype)[0]
    assert np.mean(bits(fused) != bits(stepwise)) > 0.2


@pytest.mark.parametrize("p", [3, 8, 16])
def test_prod_inexact_reveals_the_order_in_fp32(p):
    n = p * 512
    xs = [inputs.prod_inexact(n, 12, r, "f32") for r in range(p)]
    ring = oracle.allreduce(xs, "prod", "f32", "ring")[0]
    pairs = oracle.allreduce(xs, "prod", "f32", "allpairs")[0]
    assert np.mean(bits(ring) != bits(pairs)) > 0.2


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("p,sched", [(3, "ring"), (5, "allpairs"), (8, "custom"), (16, "ring")])
def test_prod_overflow_reveals_every_neighbour_swap(dtype, p, sched):
    n = p * 8192          # a swap near the front of a 16-rank order moves only ~0.2 % of the elements
    xs = [inputs.prod_overflow(n, 13, r, p, dtype) for r in range(p)]
    base_order = orders(p, sched)
    base = oracle.allreduce_orders(xs, "prod", dtype, base_order)[0]
    for c, k in swaps_to_check(p, np.random.default_rng(p)):
        mo = [list(o) for o in base_order]
        mo[c][k], mo[c][k + 1] = mo[c][k + 1], mo[c][k]
        y = oracle.allreduce_orders(xs, "prod", dtype, mo)[0]
        assert int(np.count_nonzero(chunk(y, p, n, c) != chunk(base, p, n, c))) >= 2, (c, k)


def test_recipes_place_what_they_say():
    p, n = 6, 5000
    xs = np.stack([inputs.cancel(n, 3, r, p, "f32") for r in range(p)])
    big = np.abs(xs) >= 2.0 ** 24
    assert (big.sum(axis=0) == 2).all()                       # two large values per element
    cols = np.where(big.T)[1].reshape(n, 2)
    pair = xs[cols[:, 0], np.arange(n)] + xs[cols[:, 1], np.arange(n)]
    assert (pair == 0).all()                                  # +B and -B, the same B
    z = np.stack([inputs.signed_zero(n, r, p, "f32") for r in range(p)])
    assert (z == 0).all()
    assert (np.signbit(z).sum(axis=0) == 1).all() and (np.signbit(z)[np.arange(n) % p, np.arange(n)]).all()
    o = np.stack([inputs.prod_overflow(n, 3, r, p, "f32") for r in range(p)])
    assert ((np.abs(o) > 2.0 ** 99).sum(axis=0) == 2).all() and ((np.abs(o) < 2.0 ** -99).sum(axis=0) == 1).all()
    q = inputs.prod_inexact(n, 3, 0, "f32")
    assert ((np.abs(q) >= 0.75) & (np.abs(q) < 1.3)).all() and (q < 0).any() and (q > 0).any()
