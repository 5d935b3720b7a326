/*
 * ORACLE -- test infrastructure, not part of the library.
 *
 * A plain, slow, single-threaded CPU restatement of the collectives that the
 * CUDA library computes: AllReduce, ReduceScatter and AllGather over p
 * same-shaped "rank" buffers, with sum / prod / min / max / avg, following a
 * named chunk schedule (ring or all-pairs).  It shares no code, header, table
 * or constant with the CUDA path.  Only the test suite, the package entry
 * point's smoke check and the benchmark's CPU-baseline leg may load it.
 *
 * Sources (cited by page title and section):
 *  - "Inside NCCL AllReduce", section "What all-reduce promises": the
 *    contract (every rank ends with the identical element-wise combination of
 *    all p buffers), the worked example, and the avg rule (floats pre-scaled
 *    by 1/p as they are read; integers divided once at the end).
 *  - "Inside NCCL AllReduce", section "The ring, exactly as the kernel runs
 *    it": the buffer is cut into one chunk per rank; a chunk collects one
 *    more rank's contribution per hop and finishes at its owner.  The
 *    three-GPU state table (t1, t2) fixes the order: chunk a starts with a1,
 *    adds a2, and is completed by a0 on GPU 0.  So chunk c is accumulated in
 *    rank order (c+1) mod p, (c+2) mod p, ..., c.
 *  - "MSCCL, in depth", section "Writing an algorithm in MSCCLang": the
 *    all-pairs schedule scatters slice r of every rank to its owner r, which
 *    reduces it, then gathers.  The accumulation order used here for slice r
 *    is rank 0, 1, ..., p-1: the owner folds the contributions in rank order
 *    (a reading; the page fixes no order inside the owner's reduction).
 *  - T-CCL, section "Shard Ownership": P shards, one per rank, the owner
 *    produces the final value of its shard (ReduceScatter), which then goes
 *    to every rank (AllGather).
 *
 * Arithmetic (plain reading where the pages leave a step open):
 *  - fp16 / bf16 / fp32 inputs are widened exactly to fp32; every partial
 *    stays fp32 through all p-1 hops; the finished value is rounded once to
 *    the output type, round-to-nearest-even.
 *  - sum/avg: fp32 addition, no contraction.  avg: each contribution is
 *    multiplied by fl32(1/p) when read.  prod: fp32 multiplication.
 *  - min/max: acc = (v < acc) ? v : acc (resp. >): the earlier operand wins
 *    ties, so the schedule order fixes which of +0/-0 survives.
 *  - int32: sum and prod wrap modulo 2^32; avg is the wrapped sum divided by
 *    p with C division (truncation toward zero).  Parity unpinned for the
 *    rounding of that division when the sum is not a multiple of p: the
 *    pages fix no rounding, and the pins cover divisible sums only.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared -o liboracle.so oracle.c -lm
 */
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#include <math.h>

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_I32 = 3 };
enum { OR_SUM = 0, OR_PROD = 1, OR_MIN = 2, OR_MAX = 3, OR_AVG = 4 };
enum { OR_RING = 1, OR_ALLPAIRS = 2 };

/* ------------------------------------------------------------------------ */
/* IEEE-754 conversions, written from the format definitions.               */
/* ------------------------------------------------------------------------ */

static float bits_to_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bfloat16 is the top half of a binary32: widening appends 16 zero bits. */
float oracle_bf16_to_f32(uint16_t h) { return bits_to_f32((uint32_t)h << 16); }

/* binary32 -> bfloat16, round to nearest, ties to even.  The value keeps the
 * 8 exponent bits and the top 7 fraction bits; the dropped 16 bits decide the
 * rounding.  NaN stays NaN (quiet bit forced). */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u = f32_to_bits(f);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep = u >> 16;
    uint32_t dropped = u & 0xffffu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (keep & 1u)))
        keep += 1u; /* carries into the exponent; the largest finite rounds to inf */
    return (uint16_t)keep;
}

/* binary16 -> binary32: sign, 5 exponent bits (bias 15), 10 fraction bits. */
float oracle_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? (double)NAN : (double)INFINITY;
    else
        v = ldexp(1024.0 + (double)m, e - 25);     /* (1 + m/1024) * 2^(e-15) */
    return (float)(sign ? -v : v);
}

/* binary32 -> binary16, round to nearest, ties to even, from the definition:
 * find the spacing of binary16 numbers around |x|, round |x| / spacing to the
 * nearest even integer, and encode.  |x| >= 65520 (halfway between the
 * largest finite 65504 and 2^16) rounds to infinity. */
uint16_t oracle_f32_to_f16(float f)
{
    uint16_t sign = (f32_to_bits(f) >> 31) ? 0x8000u : 0u;
    if (isnan(f)) return (uint16_t)(sign | 0x7e00u);
    double a = fabs((double)f);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: spacing 2^-24, value = k * 2^-24, k in [0, 1024] */
        double k = nearbyint(ldexp(a, 24));        /* default mode: ties-to-even */
        return (uint16_t)(sign | (uint16_t)k);     /* k == 1024 is the smallest normal */
    }
    int ex;
    (void)frexp(a, &ex);                           /* a = fr * 2^ex, fr in [0.5, 1) */
    int e = ex - 1;                                /* a in [2^e, 2^(e+1)) */
    double k = nearbyint(ldexp(a, 10 - e));        /* significand * 2^10, in [1024, 2048] */
    if (k >= 2048.0) { k = 1024.0; e += 1; }
    if (e > 15) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)((int)k - 1024));
}

/* ------------------------------------------------------------------------ */
/* Schedule: chunk bounds and the accumulation order of each chunk.         */
/* ------------------------------------------------------------------------ */

/* Chunk c of an n-element buffer cut into p balanced pieces: the first n % p
 * chunks hold one extra element.  With n % p == 0 every chunk is n/p. */
void oracle_chunk_bounds(int p, uint64_t n, int c, uint64_t *begin, uint64_t *end)
{
    uint64_t q = n / (uint64_t)p, r = n % (uint64_t)p, uc = (uint64_t)c;
    *begin = uc * q + (uc < r ? uc : r);
    *end = *begin + q + (uc < r ? 1u : 0u);
}

/* Rank order in which chunk c collects contributions.
 * ring: starts at the rank after the owner and walks the ring, one rank per
 *       hop, so the owner c adds the last contribution.
 * all-pairs: the owner reduces what every rank sent it, rank 0 first. */
int oracle_chunk_order(int p, int schedule, int c, int *order)
{
    if (p < 1 || c < 0 || c >= p) return -1;
    for (int k = 0; k < p; ++k) {
        if (schedule == OR_RING) order[k] = (c + 1 + k) % p;
        else if (schedule == OR_ALLPAIRS) order[k] = k;
        else return -1;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* One output element.                                                      */
/* ------------------------------------------------------------------------ */

static float load_f(int dtype, const void *buf, uint64_t e)
{
    if (dtype == OR_F32) return ((const float *)buf)[e];
    if (dtype == OR_F16) return oracle_f16_to_f32(((const uint16_t *)buf)[e]);
    return oracle_bf16_to_f32(((const uint16_t *)buf)[e]);
}

static void store_f(int dtype, void *buf, uint64_t e, float v)
{
    if (dtype == OR_F32) ((float *)buf)[e] = v;
    else if (dtype == OR_F16) ((uint16_t *)buf)[e] = oracle_f32_to_f16(v);
    else ((uint16_t *)buf)[e] = oracle_f32_to_bf16(v);
}

/* The reduced value of element e, whose chunk has rank order `order`,
 * written to out[oe]. */
static void reduce_element(int p, int dtype, int op, const int *order,
                           const void *const *x, uint64_t e, void *out, uint64_t oe)
{
    if (dtype == OR_I32) {
        uint32_t acc = (uint32_t)((const int32_t *)x[order[0]])[e];
        for (int k = 1; k < p; ++k) {
            uint32_t v = (uint32_t)((const int32_t *)x[order[k]])[e];
            int32_t sa = (int32_t)acc, sv = (int32_t)v;
            switch (op) {
            case OR_SUM: case OR_AVG: acc = acc + v; break;
            case OR_PROD: acc = acc * v; break;
            case OR_MIN: acc = (sv < sa) ? v : acc; break;
            case OR_MAX: acc = (sv > sa) ? v : acc; break;
            }
        }
        int32_t res = (int32_t)acc;
        if (op == OR_AVG) res = res / p;            /* divided once, at the end */
        ((int32_t *)out)[oe] = res;
        return;
    }
    float scale = 1.0f / (float)p;                  /* fl32(1/p) */
    float acc = load_f(dtype, x[order[0]], e);
    if (op == OR_AVG) acc = acc * scale;            /* pre-scaled as it is read */
    for (int k = 1; k < p; ++k) {
        float v = load_f(dtype, x[order[k]], e);
        switch (op) {
        case OR_SUM: acc = acc + v; break;
        case OR_AVG: acc = acc + v * scale; break;
        case OR_PROD: acc = acc * v; break;
        case OR_MIN: acc = (v < acc) ? v : acc; break;
        case OR_MAX: acc = (v > acc) ? v : acc; break;
        }
    }
    store_f(dtype, out, oe, acc);
}

static int check_args(int p, int dtype, int op, int schedule)
{
    if (p < 1 || p > 64) return -1;
    if (dtype < OR_F32 || dtype > OR_I32) return -1;
    if (op < OR_SUM || op > OR_AVG) return -1;
    if (schedule != OR_RING && schedule != OR_ALLPAIRS) return -1;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Collectives.                                                             */
/* ------------------------------------------------------------------------ */

/* AllReduce with explicit per-chunk orders: order[c*p + k] is the k-th rank
 * folded into chunk c (each row a permutation of 0..p-1).  Every rank's
 * output y[k] receives all n elements. */
int oracle_allreduce_orders(int p, uint64_t n, int dtype, int op, const uint8_t *order,
                            const void *const *x, void *const *y)
{
    if (check_args(p, dtype, op, OR_RING)) return -1;
    size_t s = (dtype == OR_F32 || dtype == OR_I32) ? 4 : 2;
    int ord[64];
    for (int c = 0; c < p; ++c) {
        uint64_t seen = 0;
        for (int k = 0; k < p; ++k) {
            ord[k] = order[c * p + k];
            if (ord[k] >= p || ((seen >> ord[k]) & 1u)) return -1;
            seen |= (uint64_t)1 << ord[k];
        }
        uint64_t b, en;
        oracle_chunk_bounds(p, n, c, &b, &en);
        for (uint64_t e = b; e < en; ++e) {
            reduce_element(p, dtype, op, ord, x, e, y[0], e);
            for (int k = 1; k < p; ++k)             /* the finished chunk goes to every rank */
                memcpy((char *)y[k] + e * s, (const char *)y[0] + e * s, s);
        }
    }
    return 0;
}

/* AllReduce: every rank's output y[k] receives the full reduction, all n
 * elements; chunk c is reduced in its schedule order. */
int oracle_allreduce(int p, uint64_t n, int dtype, int op, int schedule,
                     const void *const *x, void *const *y)
{
    if (check_args(p, dtype, op, schedule)) return -1;
    uint8_t order[64 * 64];
    int row[64];
    for (int c = 0; c < p; ++c) {
        oracle_chunk_order(p, schedule, c, row);
        for (int k = 0; k < p; ++k) order[c * p + k] = (uint8_t)row[k];
    }
    return oracle_allreduce_orders(p, n, dtype, op, order, x, y);
}

/* AllReduce as the ring runs it hop by hop ("Inside NCCL AllReduce", "The
 * ring, exactly as the kernel runs it"): chunk c starts as rank (c+1)'s
 * contribution; at each of the p-1 reduce-scatter hops the next rank adds its
 * own contribution to the partial it received and passes it on.  Between hops
 * a partial lives in a rank buffer, so it is held in the element type: each
 * hop widens the received partial and the local contribution to fp32 (avg:
 * contributions pre-scaled by fl32(1/p) as read), applies the op once and
 * rounds the result back to the element type.  The finished chunk then
 * circulates unchanged (all-gather half).  int32 and fp32 give the same bits as
 * oracle_allreduce with the ring schedule; fp16/bf16 round at every hop. */
int oracle_allreduce_ring_stepwise(int p, uint64_t n, int dtype, int op, const void *const *x, void *const *y)
{
    if (check_args(p, dtype, op, OR_RING)) return -1;
    size_t s = (dtype == OR_F32 || dtype == OR_I32) ? 4 : 2;
    float scale = 1.0f / (float)p;
    for (int c = 0; c < p; ++c) {
        uint64_t b, en;
        oracle_chunk_bounds(p, n, c, &b, &en);
        for (uint64_t e = b; e < en; ++e) {
            int first = (c + 1) % p;
            unsigned char held[4];                    /* the partial, in the element type */
            if (dtype == OR_I32) {
                memcpy(held, (const char *)x[first] + e * s, 4);
            } else {
                float v = load_f(dtype, x[first], e);
                if (op == OR_AVG) v = v * scale;
                store_f(dtype, held, 0, v);
            }
            for (int hop = 1; hop < p; ++hop) {
                int d = (c + 1 + hop) % p;
                if (dtype == OR_I32) {
                    uint32_t acc, v;
                    memcpy(&acc, held, 4);
                    v = ((const uint32_t *)x[d])[e];
                    int32_t sa = (int32_t)acc, sv = (int32_t)v;
                    switch (op) {
                    case OR_SUM: case OR_AVG: acc = acc + v; break;
                    case OR_PROD: acc = acc * v; break;
                    case OR_MIN: acc = (sv < sa) ? v : acc; break;
                    case OR_MAX: acc = (sv > sa) ? v : acc; break;
                    }
                    memcpy(held, &acc, 4);
                } else {
                    float acc = load_f(dtype, held, 0);
                    float v = load_f(dtype, x[d], e);
                    switch (op) {
                    case OR_SUM: acc = acc + v; break;
                    case OR_AVG: acc = acc + v * scale; break;
                    case OR_PROD: acc = acc * v; break;
                    case OR_MIN: acc = (v < acc) ? v : acc; break;
                    case OR_MAX: acc = (v > acc) ? v : acc; break;
                    }
                    store_f(dtype, held, 0, acc);
                }
            }
            if (dtype == OR_I32 && op == OR_AVG) {
                int32_t r;
                memcpy(&r, held, 4);
                r = r / p;                            /* divided once, at the end */
                memcpy(held, &r, 4);
            }
            for (int k = 0; k < p; ++k) memcpy((char *)y[k] + e * s, held, s);
        }
    }
    return 0;
}

/* AllReduce followed by the merge into the residual stream and RMSNorm,
 * fused in the all-reduce ("Inside NCCL AllReduce", last section: in a
 * decoding path the residual merge and the RMSNorm after the all-reduce run
 * inside the all-reduce kernel).  The pages give no formula; the plain reading, per element of
 * a [rows, hidden] buffer:
 *   y   = the sum AllReduce of the p inputs (schedule order, fp32, rounded)
 *   h   = round(fl32(y) + fl32(residual))            -- the merge
 *   out = round(h / sqrt(mean_row(h^2) + eps) * gamma) -- RMSNorm (Zhang and
 *         Sennrich, 2019); the norm is computed here in fp64
 * out goes to every rank; residual_out receives h.  dtype f32/f16/bf16. */
int oracle_allreduce_residual_rmsnorm(int p, uint64_t rows, uint64_t hidden, int dtype, int schedule,
                                      const void *const *x, const void *residual, const void *gamma,
                                      double eps, void *out, void *residual_out)
{
    if (dtype == OR_I32 || hidden == 0) return -1;
    if (check_args(p, dtype, OR_SUM, schedule)) return -1;
    uint64_t n = rows * hidden;
    int order[64];
    for (uint64_t row = 0; row < rows; ++row) {
        double ss = 0.0;
        for (uint64_t j = 0; j < hidden; ++j) {
            uint64_t e = row * hidden + j;
            uint64_t q = n / (uint64_t)p, r = n % (uint64_t)p;
            uint64_t c = (e < r * (q + 1)) ? e / (q + 1) : r + (e - r * (q + 1)) / q;
            oracle_chunk_order(p, schedule, (int)c, order);
            unsigned char ybuf[4];
            reduce_element(p, dtype, OR_SUM, order, x, e, ybuf, 0);
            float h = load_f(dtype, ybuf, 0) + load_f(dtype, residual, e);
            store_f(dtype, residual_out, e, h);
            double hv = (double)load_f(dtype, residual_out, e);
            ss += hv * hv;
        }
        double inv = 1.0 / sqrt(ss / (double)hidden + eps);
        for (uint64_t j = 0; j < hidden; ++j) {
            uint64_t e = row * hidden + j;
            double hv = (double)load_f(dtype, residual_out, e);
            double g = (double)load_f(dtype, gamma, j);
            store_f(dtype, out, e, (float)(hv * inv * g));
        }
    }
    return 0;
}

/* ReduceScatter: rank r's output y[r] receives chunk r of the reduction,
 * n/p elements written from offset 0.  Requires n % p == 0. */
int oracle_reduce_scatter(int p, uint64_t n, int dtype, int op, int schedule,
                          const void *const *x, void *const *y)
{
    if (check_args(p, dtype, op, schedule)) return -1;
    if (n % (uint64_t)p) return -1;
    int order[64];
    for (int r = 0; r < p; ++r) {
        uint64_t b, en;
        oracle_chunk_bounds(p, n, r, &b, &en);
        oracle_chunk_order(p, schedule, r, order);
        for (uint64_t e = b; e < en; ++e)
            reduce_element(p, dtype, op, order, x, e, y[r], e - b);
    }
    return 0;
}

/* AllGather: rank r contributes chunk r of its own buffer x[r] (elements
 * [r*n/p, (r+1)*n/p)); every rank's output y[k] receives all n elements,
 * chunk r at offset r*n/p.  Requires n % p == 0. */
int oracle_all_gather(int p, uint64_t n, int dtype, const void *const *x, void *const *y)
{
    if (p < 1 || p > 64 || dtype < OR_F32 || dtype > OR_I32) return -1;
    if (n % (uint64_t)p) return -1;
    size_t s = (dtype == OR_F32 || dtype == OR_I32) ? 4 : 2;
    for (int r = 0; r < p; ++r) {
        uint64_t b, en;
        oracle_chunk_bounds(p, n, r, &b, &en);
        for (int k = 0; k < p; ++k)
            memcpy((char *)y[k] + b * s, (const char *)x[r] + b * s, (size_t)(en - b) * s);
    }
    return 0;
}

/* AllReduce output at m chosen element indices idx[0..m): out[j] = y[idx[j]]
 * (identical on every rank).  For checking very large buffers element by
 * element without recomputing all of them. */
int oracle_allreduce_at(int p, uint64_t n, int dtype, int op, int schedule,
                        const void *const *x, const uint64_t *idx, uint64_t m, void *out)
{
    if (check_args(p, dtype, op, schedule)) return -1;
    uint64_t q = n / (uint64_t)p, r = n % (uint64_t)p;
    int order[64];
    for (uint64_t j = 0; j < m; ++j) {
        uint64_t e = idx[j];
        if (e >= n) return -1;
        /* the chunk holding e: the first r chunks have q+1 elements */
        uint64_t c = (e < r * (q + 1)) ? e / (q + 1) : r + (e - r * (q + 1)) / q;
        oracle_chunk_order(p, schedule, (int)c, order);
        reduce_element(p, dtype, op, order, x, e, out, j);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Alpha-beta cost model ("MSCCL, in depth", sections "Why generic          */
/* collectives leave time on the table" and "Worked example: all-pairs      */
/* versus ring on 8 GPUs").  Each synchronised step costs alpha; each byte  */
/* costs 1/(B * protocol efficiency).  Both schedules move 2(p-1)/p of the  */
/* buffer; the ring takes 2(p-1) steps, all-pairs takes 2.                  */
/* ------------------------------------------------------------------------ */

double oracle_time_ring(int p, double nbytes, double alpha_s, double bw_bytes_per_s, double eff)
{
    return 2.0 * (p - 1) * alpha_s + 2.0 * (p - 1) / p * nbytes / (bw_bytes_per_s * eff);
}

double oracle_time_allpairs(int p, double nbytes, double alpha_s, double bw_bytes_per_s, double eff)
{
    return 2.0 * alpha_s + 2.0 * (p - 1) / p * nbytes / (bw_bytes_per_s * eff);
}
