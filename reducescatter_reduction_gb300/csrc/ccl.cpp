// Host front end of the C ABI declared in include/ccl.h: communicators,
// argument and alias checks, the schedule builder and its validator, the
// alpha-beta cost model, and the dispatch to the kernel translation units.
#include "ccl.h"

#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>

#include "internal.h"

using namespace ccl;

struct ccl_comm {
    int p = 0;
    int device = 0;
    int num_sms = 0;
    void *in[kMaxRanks] = {};
    void *out[kMaxRanks] = {};
    int sm_budget = 0;
    int variant = CCL_VARIANT_AUTO;
    size_t pipe_bytes = 0;
    unsigned *d_status = nullptr;   // 256-byte device status block
    bool has_custom = false;
    uint8_t custom[kMaxRanks * kMaxRanks] = {};
    Table table;                    // last built table (one-entry cache)
    int table_sched = -1;
    bool table_valid = false;
    uint64_t launches = 0;
    char last[320] = "";
    long long wait_limit_ns = 2000000000LL;  // bounded device waits: 2 s
    int stall_test = 0;
};

// ---------------------------------------------------------------------------
// Errors.
// ---------------------------------------------------------------------------

static thread_local std::string g_err;

static ccl_status_t fail(ccl_status_t st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return st;
}

namespace ccl {
// Lets other translation units of the library report through ccl_last_error().
ccl_status_t record_error(ccl_status_t st, const char *msg)
{
    g_err = msg;
    return st;
}
}  // namespace ccl

static ccl_status_t cuda_fail(cudaError_t err, const char *what)
{
    return fail(CCL_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(err), cudaGetErrorString(err));
}

static bool debug_on()
{
    static int on = -1;
    if (on < 0) {
        const char *e = getenv("CCL_DEBUG");
        on = (e && *e && strcmp(e, "0") != 0) ? 1 : 0;
    }
    return on == 1;
}

// Restores the caller's current device when a call had to switch to the
// communicator's device.
struct DeviceGuard {
    int prev = -1;
    bool switched = false;
    cudaError_t err = cudaSuccess;
    explicit DeviceGuard(int dev)
    {
        err = cudaGetDevice(&prev);
        if (err == cudaSuccess && prev != dev) {
            err = cudaSetDevice(dev);
            switched = (err == cudaSuccess);
        }
    }
    ~DeviceGuard()
    {
        if (switched) cudaSetDevice(prev);
    }
};

// ---------------------------------------------------------------------------
// Schedule builder.
// ---------------------------------------------------------------------------

// p balanced chunks, the first n % p one element larger.
static void chunk_bounds(int p, uint64_t n, uint64_t *bounds)
{
    const uint64_t q = n / uint64_t(p), r = n % uint64_t(p);
    for (int c = 0; c <= p; ++c) {
        const uint64_t uc = uint64_t(c);
        bounds[c] = uc * q + (uc < r ? uc : r);
    }
}

// Ring ("Inside NCCL AllReduce", "The ring, exactly as the kernel runs it"):
// a chunk starts at the rank after its owner and walks the ring, so the owner
// adds the last contribution.  All-pairs ("MSCCL, in depth", "Writing an
// algorithm in MSCCLang"): the owner folds what every rank sent, rank 0 first.
static void chunk_orders(int p, int schedule, uint8_t *order)
{
    for (int c = 0; c < p; ++c)
        for (int k = 0; k < p; ++k)
            order[c * p + k] = uint8_t(schedule == CCL_SCHED_RING ? (c + 1 + k) % p : k);
}

static bool orders_valid(int p, const uint8_t *order)
{
    for (int c = 0; c < p; ++c) {
        uint64_t seen = 0;
        for (int k = 0; k < p; ++k) {
            const int r = order[c * p + k];
            if (r >= p || ((seen >> r) & 1u)) return false;
            seen |= uint64_t(1) << r;
        }
    }
    return true;
}

extern "C" ccl_status_t ccl_schedule_build(int p, uint64_t n, ccl_schedule_t schedule,
                                           uint64_t *bounds, uint8_t *order)
{
    if (p < 1 || p > kMaxRanks) return fail(CCL_ERR_INVALID_ARG, "p=%d outside [1, %d]", p, kMaxRanks);
    if (!bounds || !order) return fail(CCL_ERR_INVALID_ARG, "NULL output array");
    if (schedule != CCL_SCHED_RING && schedule != CCL_SCHED_ALLPAIRS)
        return fail(CCL_ERR_INVALID_ARG, "schedule %d is not ring or all-pairs", int(schedule));
    chunk_bounds(p, n, bounds);
    chunk_orders(p, schedule, order);
    return CCL_OK;
}

extern "C" ccl_status_t ccl_schedule_check(int p, uint64_t n, const uint64_t *bounds,
                                           const uint8_t *order)
{
    if (p < 1 || p > kMaxRanks) return fail(CCL_ERR_INVALID_ARG, "p=%d outside [1, %d]", p, kMaxRanks);
    if (!bounds || !order) return fail(CCL_ERR_INVALID_ARG, "NULL table");
    if (bounds[0] != 0 || bounds[p] != n)
        return fail(CCL_ERR_INVALID_ARG, "chunks do not cover [0, %llu)", (unsigned long long)n);
    for (int c = 0; c < p; ++c)
        if (bounds[c] > bounds[c + 1]) return fail(CCL_ERR_INVALID_ARG, "chunk %d bounds decrease", c);
    if (!orders_valid(p, order))
        return fail(CCL_ERR_INVALID_ARG, "an order row is not a permutation of the ranks");
    return CCL_OK;
}

// ---------------------------------------------------------------------------
// Alpha-beta cost model ("MSCCL, in depth", sections "Why generic
// collectives leave time on the table" and "Worked example: all-pairs versus
// ring on 8 GPUs").  Defaults are the worked example's assumptions.
// ---------------------------------------------------------------------------

static const ccl_cost_params_t kPageParams = {2e-6, 300e9, 120.0 / 128.0, 0.5};

extern "C" double ccl_cost_estimate(int p, double nbytes, ccl_schedule_t schedule,
                                    const ccl_cost_params_t *params)
{
    const ccl_cost_params_t &m = params ? *params : kPageParams;
    if (p < 1 || nbytes < 0 || m.bw_bytes_per_s <= 0) return -1.0;
    const double moved = 2.0 * (p - 1) / p * nbytes;
    if (schedule == CCL_SCHED_RING) {
        if (m.eff_ring <= 0) return -1.0;
        return 2.0 * (p - 1) * m.alpha_s + moved / (m.bw_bytes_per_s * m.eff_ring);
    }
    if (schedule == CCL_SCHED_ALLPAIRS) {
        if (m.eff_allpairs <= 0) return -1.0;
        return 2.0 * m.alpha_s + moved / (m.bw_bytes_per_s * m.eff_allpairs);
    }
    return -1.0;
}

extern "C" ccl_schedule_t ccl_select_schedule(int p, double nbytes, const ccl_cost_params_t *params)
{
    const double tr = ccl_cost_estimate(p, nbytes, CCL_SCHED_RING, params);
    const double ta = ccl_cost_estimate(p, nbytes, CCL_SCHED_ALLPAIRS, params);
    return (ta >= 0 && ta < tr) ? CCL_SCHED_ALLPAIRS : CCL_SCHED_RING;
}

// Environment overrides, as NCCL's NCCL_ALGO / NCCL_PROTO ("Inside NCCL
// AllReduce", section on the tuner): CCL_SCHEDULE=ring|allpairs|auto,
// CCL_VARIANT=ldst|tma|tma_bulkred|auto and CCL_SM_BUDGET=<k> apply only where
// the call or the communicator left the choice open (schedule AUTO, variant
// AUTO, SM budget 0).  An unset or empty variable changes nothing; any other
// value that is not one of the listed ones is an error, never ignored.
static bool env_schedule(int *out)
{
    const char *e = getenv("CCL_SCHEDULE");
    if (!e || !*e || strcmp(e, "auto") == 0) return true;
    if (strcmp(e, "ring") == 0) *out = CCL_SCHED_RING;
    else if (strcmp(e, "allpairs") == 0) *out = CCL_SCHED_ALLPAIRS;
    else return false;
    return true;
}

static bool env_variant(int *out)
{
    const char *e = getenv("CCL_VARIANT");
    if (!e || !*e || strcmp(e, "auto") == 0) return true;
    if (strcmp(e, "ldst") == 0) *out = CCL_VARIANT_LDST;
    else if (strcmp(e, "tma") == 0) *out = CCL_VARIANT_TMA;
    else if (strcmp(e, "tma_bulkred") == 0) *out = CCL_VARIANT_TMA_BULKRED;
    else return false;
    return true;
}

static bool env_sm_budget(int *out)
{
    const char *e = getenv("CCL_SM_BUDGET");
    if (!e || !*e) return true;
    char *end = nullptr;
    const long v = strtol(e, &end, 10);
    if (*end != '\0' || v < 0 || v > 1000000) return false;
    *out = int(v);
    return true;
}

// schedule AUTO: CCL_SCHEDULE if set, else the cost model.  -1 if the
// variable holds something else.
static int resolve_schedule(const ccl_comm *c, int schedule, double nbytes)
{
    if (schedule != CCL_SCHED_AUTO) return schedule;
    int s = CCL_SCHED_AUTO;
    if (!env_schedule(&s)) return -1;
    if (s != CCL_SCHED_AUTO) return s;
    return ccl_select_schedule(c->p, nbytes, nullptr);
}

static const Table *get_table(ccl_comm *c, uint64_t n, int schedule)
{
    Table &t = c->table;
    if (!(c->table_valid && t.n == n && c->table_sched == schedule && schedule != CCL_SCHED_CUSTOM)) {
        t.p = c->p;
        t.n = n;
        chunk_bounds(c->p, n, t.bound);
        if (schedule == CCL_SCHED_CUSTOM) memcpy(t.order, c->custom, size_t(c->p) * c->p);
        else chunk_orders(c->p, schedule, t.order);
        c->table_sched = schedule;
        c->table_valid = true;
    }
    return &t;
}

// ---------------------------------------------------------------------------
// Communicator.
// ---------------------------------------------------------------------------

extern "C" int ccl_version(void) { return CCL_VERSION; }

extern "C" const char *ccl_last_error(void) { return g_err.c_str(); }

extern "C" ccl_status_t ccl_comm_create(ccl_comm_t *out, int p, void *const *rank_ptrs)
{
    if (!out) return fail(CCL_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (p < 1 || p > kMaxRanks) return fail(CCL_ERR_INVALID_ARG, "p=%d outside [1, %d]", p, kMaxRanks);
    if (!rank_ptrs) return fail(CCL_ERR_INVALID_ARG, "rank_ptrs is NULL");
    for (int r = 0; r < p; ++r)
        if (!rank_ptrs[r]) return fail(CCL_ERR_INVALID_ARG, "rank_ptrs[%d] is NULL", r);
    ccl_comm *c = new (std::nothrow) ccl_comm;
    if (!c) return fail(CCL_ERR_NOMEM, "host allocation failed");
    c->p = p;
    for (int r = 0; r < p; ++r) c->in[r] = c->out[r] = rank_ptrs[r];
    cudaError_t err = cudaGetDevice(&c->device);
    if (err == cudaSuccess)
        err = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
    if (err == cudaSuccess) err = cudaMalloc(&c->d_status, 256);
    if (err == cudaSuccess) err = cudaMemset(c->d_status, 0, 256);
    if (err != cudaSuccess) {
        if (c->d_status) cudaFree(c->d_status);
        delete c;
        if (err == cudaErrorMemoryAllocation) return fail(CCL_ERR_NOMEM, "device status block: out of memory");
        return cuda_fail(err, "ccl_comm_create");
    }
    *out = c;
    return CCL_OK;
}

extern "C" ccl_status_t ccl_comm_set_outputs(ccl_comm_t c, void *const *out_ptrs)
{
    if (!c) return fail(CCL_ERR_INVALID_ARG, "comm is NULL");
    if (!out_ptrs) {
        for (int r = 0; r < c->p; ++r) c->out[r] = c->in[r];
        return CCL_OK;
    }
    for (int r = 0; r < c->p; ++r)
        if (!out_ptrs[r]) return fail(CCL_ERR_INVALID_ARG, "out_ptrs[%d] is NULL", r);
    for (int r = 0; r < c->p; ++r) c->out[r] = out_ptrs[r];
    return CCL_OK;
}

extern "C" ccl_status_t ccl_comm_set_schedule(ccl_comm_t c, const uint8_t *order)
{
    if (!c) return fail(CCL_ERR_INVALID_ARG, "comm is NULL");
    if (!order) return fail(CCL_ERR_INVALID_ARG, "order is NULL");
    if (!orders_valid(c->p, order))
        return fail(CCL_ERR_INVALID_ARG, "an order row is not a permutation of the ranks");
    memcpy(c->custom, order, size_t(c->p) * c->p);
    c->has_custom = true;
    c->table_valid = false;
    return CCL_OK;
}

extern "C" ccl_status_t ccl_set_launch(ccl_comm_t c, int sm_budget, int variant, size_t pipe_bytes)
{
    if (!c) return fail(CCL_ERR_INVALID_ARG, "comm is NULL");
    if (sm_budget < 0) return fail(CCL_ERR_INVALID_ARG, "sm_budget %d < 0", sm_budget);
    if (variant < CCL_VARIANT_AUTO || variant > CCL_VARIANT_ONE_PHASE)
        return fail(CCL_ERR_INVALID_ARG, "unknown variant %d", variant);
    if (pipe_bytes != 0 && (pipe_bytes % 16 || pipe_bytes < 1024 || pipe_bytes > 32768))
        return fail(CCL_ERR_INVALID_ARG, "pipeline_chunk_bytes %zu not a multiple of 16 in [1024, 32768]",
                    pipe_bytes);
    c->sm_budget = sm_budget;
    c->variant = variant;
    c->pipe_bytes = pipe_bytes;
    return CCL_OK;
}

extern "C" ccl_status_t ccl_comm_set_debug(ccl_comm_t c, long long wait_limit_ns, int stall_test)
{
    if (!c) return fail(CCL_ERR_INVALID_ARG, "comm is NULL");
    if (wait_limit_ns < 0 || stall_test < 0 || stall_test > 2)
        return fail(CCL_ERR_INVALID_ARG, "wait_limit_ns %lld / stall_test %d out of range", wait_limit_ns, stall_test);
    c->wait_limit_ns = wait_limit_ns ? wait_limit_ns : 2000000000LL;
    c->stall_test = stall_test;
    return CCL_OK;
}

extern "C" ccl_status_t ccl_comm_destroy(ccl_comm_t c)
{
    if (!c) return CCL_OK;
    ccl_status_t st = CCL_OK;
    if (c->d_status) {
        DeviceGuard g(c->device);
        cudaError_t err = cudaFree(c->d_status);
        if (err != cudaSuccess) st = cuda_fail(err, "ccl_comm_destroy");
    }
    delete c;
    return st;
}

extern "C" ccl_status_t ccl_comm_check(ccl_comm_t c)
{
    if (!c) return fail(CCL_ERR_INVALID_ARG, "comm is NULL");
    DeviceGuard g(c->device);
    if (g.err != cudaSuccess) return cuda_fail(g.err, "ccl_comm_check");
    unsigned st[4] = {0, 0, 0, 0};
    cudaError_t err = cudaDeviceSynchronize();
    if (err == cudaSuccess) err = cudaMemcpy(st, c->d_status, sizeof st, cudaMemcpyDeviceToHost);
    if (err != cudaSuccess) return cuda_fail(err, "ccl_comm_check");
    if (st[0] != 0) {
        cudaMemset(c->d_status, 0, 256);
        if (st[0] == kBoundsCode)
            return fail(CCL_ERR_BOUNDS, "an access outside a rank buffer was computed and skipped (site %u, block %u, "
                        "index %u)", st[3], st[1], st[2]);
        return fail(CCL_ERR_TIMEOUT, "a bounded device wait gave up (code %u, block %u, stage %u)", st[0],
                    st[1], st[2]);
    }
    return CCL_OK;
}

extern "C" int ccl_bounds_checked(void)
{
#ifdef CCL_BOUNDS_CHECK
    return 1;
#else
    return 0;
#endif
}

extern "C" ccl_status_t ccl_comm_last_launch(ccl_comm_t c, char *buf, size_t len)
{
    if (!c || !buf || len == 0) return fail(CCL_ERR_INVALID_ARG, "NULL comm or buffer");
    snprintf(buf, len, "%s", c->last);
    return CCL_OK;
}

extern "C" uint64_t ccl_comm_launch_count(ccl_comm_t c) { return c ? c->launches : 0; }

// ---------------------------------------------------------------------------
// Argument checks shared by the collectives.
// ---------------------------------------------------------------------------

static const char *kOpName[] = {"sum", "prod", "min", "max", "avg"};
static const char *kDtypeName[] = {"f32", "f16", "bf16", "i32"};
static const char *kSchedName[] = {"auto", "ring", "allpairs", "custom"};
static const char *kCollName[] = {"allreduce", "reduce_scatter", "all_gather"};
static const char *kVariantName[] = {"auto", "ldst", "tma", "tma_bulkred", "ring_stepwise", "one_phase"};

enum Coll { COLL_AR = 0, COLL_RS = 1, COLL_AG = 2 };

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

static bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.lo < a.hi && b.lo < b.hi; }

// Every output must be disjoint from every other output and from everything
// any rank reads, except the exact in-place alias of its own rank:
//   AR: out[r] == in[r];  RS: out[r] == in[r] + chunk r;  AG: out[r] == in[r].
// With those aliases each element is read and written by one thread only.
// *alias is set when an output is (part of) an input: the kernels then load
// with coherent loads instead of ld.global.nc.
static ccl_status_t check_aliases(const ccl_comm *c, int coll, uint64_t n, size_t s, uint64_t *self_mask,
                                  bool *alias = nullptr)
{
    const int p = c->p;
    const uint64_t chunk = n / uint64_t(p);
    Range rd[kMaxRanks], wr[kMaxRanks];
    for (int r = 0; r < p; ++r) {
        const uintptr_t in = uintptr_t(c->in[r]), out = uintptr_t(c->out[r]);
        if (coll == COLL_AG) rd[r] = {in + r * chunk * s, in + (r + 1) * chunk * s};
        else rd[r] = {in, in + n * s};
        if (coll == COLL_RS) wr[r] = {out, out + chunk * s};
        else wr[r] = {out, out + n * s};
    }
    *self_mask = 0;
    if (alias) *alias = false;
    for (int k = 0; k < p; ++k) {
        for (int j = k + 1; j < p; ++j)
            if (overlap(wr[k], wr[j])) return fail(CCL_ERR_INVALID_ARG, "outputs of ranks %d and %d overlap", k, j);
        for (int j = 0; j < p; ++j) {
            if (!overlap(wr[k], rd[j])) continue;
            bool ok = false;
            if (j == k) {
                const uintptr_t in = uintptr_t(c->in[k]), out = uintptr_t(c->out[k]);
                if (coll == COLL_AR || coll == COLL_AG) ok = (out == in);
                else ok = (out == in + k * chunk * s);
            }
            if (!ok) return fail(CCL_ERR_INVALID_ARG, "output of rank %d overlaps the input of rank %d", k, j);
            if (coll == COLL_AG) *self_mask |= uint64_t(1) << k;
            if (alias) *alias = true;
        }
    }
    return CCL_OK;
}

static ccl_status_t run(ccl_comm *c, int coll, int op, int dtype, size_t n, int schedule, void *stream)
{
    if (!c) return fail(CCL_ERR_INVALID_ARG, "comm is NULL");
    if (dtype < CCL_F32 || dtype > CCL_I32) return fail(CCL_ERR_INVALID_ARG, "unknown dtype %d", dtype);
    if (coll != COLL_AG && (op < CCL_SUM || op > CCL_AVG)) return fail(CCL_ERR_INVALID_ARG, "unknown op %d", op);
    if (coll != COLL_AG && (schedule < CCL_SCHED_AUTO || schedule > CCL_SCHED_CUSTOM))
        return fail(CCL_ERR_INVALID_ARG, "unknown schedule %d", schedule);
    if (schedule == CCL_SCHED_CUSTOM && !c->has_custom)
        return fail(CCL_ERR_INVALID_ARG, "custom schedule requested but none set");
    const int p = c->p;
    const size_t s = elem_bytes(dtype);
    if (coll != COLL_AR && n % size_t(p) != 0)
        return fail(CCL_ERR_INVALID_ARG, "%s needs n %% p == 0 (n=%zu, p=%d)", kCollName[coll], n, p);
    if (n > (SIZE_MAX / 2) / s) return fail(CCL_ERR_INVALID_ARG, "n=%zu too large", n);
    int sm_budget = c->sm_budget;
    if (sm_budget == 0 && !env_sm_budget(&sm_budget))
        return fail(CCL_ERR_INVALID_ARG, "CCL_SM_BUDGET=%s is not a count of SMs", getenv("CCL_SM_BUDGET"));
    // AUTO: CCL_VARIANT if set; else the ld/st kernel, or the TMA variant
    // where the measured launch table (launch_table.cpp; T-CCL, "Launch
    // Configuration Tuning") estimates it faster and the layout allows it.
    // AllGather has only the ld/st kernel.
    int variant = c->variant;
    if (variant == CCL_VARIANT_AUTO && coll != COLL_AG && !env_variant(&variant))
        return fail(CCL_ERR_INVALID_ARG, "CCL_VARIANT=%s is not ldst, tma, tma_bulkred or auto", getenv("CCL_VARIANT"));
    if (variant == CCL_VARIANT_AUTO) {
        variant = CCL_VARIANT_LDST;
        if (coll != COLL_AG && n > 0 &&
            launch_table_prefers_tma(p, int(s), sm_budget, c->num_sms, double(n) * double(s))) {
            uint64_t bounds[kMaxRanks + 1];
            chunk_bounds(p, n, bounds);
            bool ok = true;
            for (int r = 0; r < p && ok; ++r)
                ok = uintptr_t(c->in[r]) % 16 == 0 && uintptr_t(c->out[r]) % 16 == 0;
            for (int k = 0; k <= p && ok; ++k) ok = (bounds[k] * s) % 16 == 0;
            uint32_t tile, stages;
            size_t smem;
            uint32_t ranks;
            const bool fits = p > kTmaNarrowMaxRanks ? tma_wide_geometry(p, c->pipe_bytes, sm_budget, &tile, &ranks, &stages, &smem)
                                                     : tma_geometry(p, c->pipe_bytes, sm_budget, &tile, &stages, &smem);
            if (ok && fits) variant = CCL_VARIANT_TMA;
        }
    }
    if ((variant == CCL_VARIANT_RING_STEPWISE || variant == CCL_VARIANT_ONE_PHASE) && coll != COLL_AR)
        return fail(CCL_ERR_UNSUPPORTED, "the %s executor is an AllReduce", kVariantName[variant]);
    if (variant == CCL_VARIANT_RING_STEPWISE && schedule != CCL_SCHED_AUTO && schedule != CCL_SCHED_RING)
        return fail(CCL_ERR_UNSUPPORTED, "the stepwise ring runs the ring schedule only");
    if ((variant == CCL_VARIANT_TMA || variant == CCL_VARIANT_TMA_BULKRED) && coll == COLL_AG)
        return fail(CCL_ERR_UNSUPPORTED, "AllGather has no TMA variant (use ld/st)");
    if (variant == CCL_VARIANT_TMA_BULKRED && !bulkred_supported(dtype, op))
        return fail(CCL_ERR_UNSUPPORTED,
                    "the bulk-reduce variant has sum (f32/f16/bf16/i32) and min/max (f16/bf16/i32) only");
    if (variant == CCL_VARIANT_TMA_BULKRED && coll == COLL_AR && n % size_t(p) != 0)
        return fail(CCL_ERR_UNSUPPORTED, "the bulk-reduce AllReduce needs n %% p == 0 (n=%zu, p=%d)", n, p);
    if (n == 0) return CCL_OK;

    uint64_t self_mask = 0;
    bool alias = false;
    ccl_status_t st = check_aliases(c, coll, n, s, &self_mask, &alias);
    if (st != CCL_OK) return st;
    if (variant == CCL_VARIANT_ONE_PHASE)
        for (int r = 0; r < p; ++r)
            if (c->out[r] == c->in[r])  // rank r's output would overwrite an input other ranks still read
                return fail(CCL_ERR_UNSUPPORTED, "the one-phase executor needs outputs distinct from the inputs");

    DeviceGuard g(c->device);
    if (g.err != cudaSuccess) return cuda_fail(g.err, kCollName[coll]);

    Launch L;
    L.p = p;
    L.op = op;
    L.dtype = dtype;
    L.mode = coll == COLL_RS ? MODE_RS : MODE_AR;
    L.n = n;
    bool aligned = true;
    for (int r = 0; r < p; ++r) {
        L.src[r] = c->in[r];
        L.dst[r] = c->out[r];
        aligned = aligned && (uintptr_t(c->in[r]) % 16 == 0) && (uintptr_t(c->out[r]) % 16 == 0);
    }
    L.vec = aligned && (coll == COLL_AR || (n / p * s) % 16 == 0);
    L.self_mask = self_mask;
    L.alias = alias;
    L.device = c->device;
    L.num_sms = c->num_sms;
    L.sm_budget = sm_budget;
    L.pipe_bytes = c->pipe_bytes;
    L.status = c->d_status;
    L.wait_limit_ns = c->wait_limit_ns;
    L.stall_test = c->stall_test;
    L.stream = static_cast<cudaStream_t>(stream);

    int sched = CCL_SCHED_RING;
    if (coll != COLL_AG) {
        sched = variant == CCL_VARIANT_RING_STEPWISE ? int(CCL_SCHED_RING)
                                                     : resolve_schedule(c, schedule, double(n) * double(s));
        if (sched < 0)
            return fail(CCL_ERR_INVALID_ARG, "CCL_SCHEDULE=%s is not ring, allpairs or auto", getenv("CCL_SCHEDULE"));
        L.table = get_table(c, n, sched);
    }
    if (variant == CCL_VARIANT_RING_STEPWISE || variant == CCL_VARIANT_ONE_PHASE) {
        // 16-byte groups only where no group straddles a chunk boundary
        bool ok = aligned;
        for (int k = 0; k <= p && ok; ++k) ok = (L.table->bound[k] * s) % 16 == 0;
        L.vec = ok;
    }
    if (variant == CCL_VARIANT_TMA || variant == CCL_VARIANT_TMA_BULKRED) {
        // bulk copies move 16-byte multiples between 16-byte aligned addresses
        bool ok = aligned;
        for (int k = 0; k <= p && ok; ++k) ok = (L.table->bound[k] * s) % 16 == 0;
        if (!ok)
            return fail(CCL_ERR_UNSUPPORTED,
                        "the TMA variant needs 16-byte aligned pointers and chunk boundaries (n=%zu, p=%d)", n, p);
        uint32_t tile, stages;
        size_t smem;
        uint32_t ranks;
        const bool fits = variant == CCL_VARIANT_TMA
                              ? (p > kTmaNarrowMaxRanks ? tma_wide_geometry(p, c->pipe_bytes, sm_budget, &tile, &ranks, &stages, &smem)
                                                        : tma_geometry(p, c->pipe_bytes, sm_budget, &tile, &stages, &smem))
                              : bulkred_geometry(p, c->pipe_bytes, &tile, &ranks, &stages, &smem);
        if (!fits)
            return fail(CCL_ERR_INVALID_ARG,
                        "pipeline_chunk_bytes %zu: two pipeline stages of that tile size do not fit in shared memory (p=%d)",
                        c->pipe_bytes, p);
    }

    LaunchInfo info;
    cudaError_t err = cudaSuccess;
    if (coll == COLL_AG) {
        err = launch_gather(L, &info);
    } else if (variant == CCL_VARIANT_TMA) {
        switch (dtype) {
        case CCL_F32: err = launch_tma_f32(L, &info); break;
        case CCL_F16: err = launch_tma_f16(L, &info); break;
        case CCL_BF16: err = launch_tma_bf16(L, &info); break;
        default: err = launch_tma_i32(L, &info); break;
        }
    } else if ((variant == CCL_VARIANT_RING_STEPWISE && p > 1) || variant == CCL_VARIANT_ONE_PHASE) {
        err = launch_compare(L, &info, variant == CCL_VARIANT_RING_STEPWISE);
    } else if (variant == CCL_VARIANT_RING_STEPWISE) {
        // p = 1: no hop to take; the one contribution is the result
        switch (dtype) {
        case CCL_F32: err = launch_reduce_f32(L, &info); break;
        case CCL_F16: err = launch_reduce_f16(L, &info); break;
        case CCL_BF16: err = launch_reduce_bf16(L, &info); break;
        default: err = launch_reduce_i32(L, &info); break;
        }
    } else if (variant == CCL_VARIANT_TMA_BULKRED) {
        switch (dtype) {
        case CCL_F32: err = launch_bulkred_f32(L, &info); break;
        case CCL_F16: err = launch_bulkred_f16(L, &info); break;
        case CCL_BF16: err = launch_bulkred_bf16(L, &info); break;
        default: err = launch_bulkred_i32(L, &info); break;
        }
        if (err == cudaSuccess && coll == COLL_AR) {
            // every chunk now sits in its owner's output: broadcast it in place
            Launch G = L;
            for (int r = 0; r < p; ++r) G.src[r] = L.dst[r];
            G.self_mask = (p == 64) ? ~uint64_t(0) : ((uint64_t(1) << p) - 1);
            G.vec = aligned && (n / p * s) % 16 == 0;
            LaunchInfo ginfo;
            err = launch_gather(G, &ginfo);
            info.kernels += ginfo.kernels;
        }
    } else {
        switch (dtype) {
        case CCL_F32: err = launch_reduce_f32(L, &info); break;
        case CCL_F16: err = launch_reduce_f16(L, &info); break;
        case CCL_BF16: err = launch_reduce_bf16(L, &info); break;
        default: err = launch_reduce_i32(L, &info); break;
        }
    }
    c->launches += uint64_t(info.kernels);
    snprintf(c->last, sizeof c->last,
             "%s dtype=%s op=%s p=%d n=%zu schedule=%s variant=%s vec=%d grid=%d block=%d smem=%zu sm_budget=%d "
             "counter=%d inplace=%d",
             info.kernel, kDtypeName[dtype], coll == COLL_AG ? "copy" : kOpName[op], p, n,
             coll == COLL_AG ? "-" : kSchedName[sched], kVariantName[variant], L.vec ? 1 : 0, info.grid, info.block,
             info.smem, sm_budget, info.counter, alias ? 1 : 0);
    if (debug_on()) {
        // the launch table's estimate for this call (AllReduce of n*s bytes per rank)
        double est = -1.0;
        if ((variant == CCL_VARIANT_LDST || variant == CCL_VARIANT_TMA) && coll == COLL_AR &&
            !launch_table_estimate(p, int(s), sm_budget, c->num_sms, double(n) * double(s), variant, &est))
            est = -1.0;
        if (est >= 0) fprintf(stderr, "[ccl] %s est_time_us=%.2f\n", c->last, est);
        else fprintf(stderr, "[ccl] %s est_time_us=-\n", c->last);
    }
    if (err != cudaSuccess) return cuda_fail(err, kCollName[coll]);
    return CCL_OK;
}

extern "C" ccl_status_t ccl_allreduce(ccl_comm_t c, ccl_op_t op, ccl_dtype_t dtype, size_t n,
                                      ccl_schedule_t schedule, void *stream)
{
    return run(c, COLL_AR, op, dtype, n, schedule, stream);
}

extern "C" ccl_status_t ccl_reduce_scatter(ccl_comm_t c, ccl_op_t op, ccl_dtype_t dtype, size_t n,
                                           ccl_schedule_t schedule, void *stream)
{
    return run(c, COLL_RS, op, dtype, n, schedule, stream);
}

extern "C" ccl_status_t ccl_all_gather(ccl_comm_t c, ccl_dtype_t dtype, size_t n, void *stream)
{
    return run(c, COLL_AG, CCL_SUM, dtype, n, CCL_SCHED_RING, stream);
}

extern "C" ccl_status_t ccl_allreduce_residual_rmsnorm(ccl_comm_t c, ccl_dtype_t dtype, size_t rows, size_t hidden,
                                                       const void *residual_in, void *residual_out, const void *gamma,
                                                       float eps, ccl_schedule_t schedule, void *stream)
{
    if (!c) return fail(CCL_ERR_INVALID_ARG, "comm is NULL");
    if (dtype == CCL_I32) return fail(CCL_ERR_UNSUPPORTED, "RMSNorm needs a floating-point dtype");
    if (dtype < CCL_F32 || dtype > CCL_BF16) return fail(CCL_ERR_INVALID_ARG, "unknown dtype %d", int(dtype));
    if (schedule < CCL_SCHED_AUTO || schedule > CCL_SCHED_CUSTOM)
        return fail(CCL_ERR_INVALID_ARG, "unknown schedule %d", int(schedule));
    if (schedule == CCL_SCHED_CUSTOM && !c->has_custom)
        return fail(CCL_ERR_INVALID_ARG, "custom schedule requested but none set");
    if (hidden == 0) return fail(CCL_ERR_INVALID_ARG, "hidden must be positive");
    if (!(eps >= 0.0f) || eps > 3.0e38f) return fail(CCL_ERR_INVALID_ARG, "eps must be finite and >= 0");
    const size_t s = elem_bytes(dtype);
    if (rows > (SIZE_MAX / 4) / hidden / s) return fail(CCL_ERR_INVALID_ARG, "rows * hidden too large");
    const size_t n = rows * hidden;
    if (n == 0) return CCL_OK;
    if (!residual_in || !residual_out || !gamma) return fail(CCL_ERR_INVALID_ARG, "NULL residual or gamma");
    const int p = c->p;

    uint64_t self_mask = 0;
    ccl_status_t st = check_aliases(c, COLL_AR, n, s, &self_mask);
    if (st != CCL_OK) return st;
    const Range ri = {uintptr_t(residual_in), uintptr_t(residual_in) + n * s};
    const Range ro = {uintptr_t(residual_out), uintptr_t(residual_out) + n * s};
    const Range gm = {uintptr_t(gamma), uintptr_t(gamma) + hidden * s};
    if (ro.lo != ri.lo && overlap(ro, ri)) return fail(CCL_ERR_INVALID_ARG, "residual_out partly overlaps residual_in");
    if (overlap(ro, gm)) return fail(CCL_ERR_INVALID_ARG, "gamma overlaps residual_out");
    for (int r = 0; r < p; ++r) {
        const Range in = {uintptr_t(c->in[r]), uintptr_t(c->in[r]) + n * s};
        const Range out = {uintptr_t(c->out[r]), uintptr_t(c->out[r]) + n * s};
        if (overlap(ro, in) || overlap(ro, out)) return fail(CCL_ERR_INVALID_ARG, "residual_out overlaps rank %d", r);
        if (overlap(ri, out) || overlap(gm, out))
            return fail(CCL_ERR_INVALID_ARG, "the output of rank %d overlaps the residual or gamma", r);
    }

    DeviceGuard g(c->device);
    if (g.err != cudaSuccess) return cuda_fail(g.err, "allreduce_residual_rmsnorm");
    Launch L;
    L.p = p;
    L.op = CCL_SUM;
    L.dtype = dtype;
    L.mode = MODE_AR;
    L.n = n;
    const size_t vec_elems = 16 / s;
    bool aligned = uintptr_t(residual_in) % 16 == 0 && uintptr_t(residual_out) % 16 == 0 &&
                   uintptr_t(gamma) % 16 == 0 && hidden % vec_elems == 0;
    for (int r = 0; r < p; ++r) {
        L.src[r] = c->in[r];
        L.dst[r] = c->out[r];
        aligned = aligned && uintptr_t(c->in[r]) % 16 == 0 && uintptr_t(c->out[r]) % 16 == 0;
    }
    L.device = c->device;
    L.num_sms = c->num_sms;
    L.stream = static_cast<cudaStream_t>(stream);
    L.status = c->d_status;
    L.wait_limit_ns = c->wait_limit_ns;
    L.stall_test = c->stall_test;
    const int sched = resolve_schedule(c, schedule, double(n) * double(s));
    if (sched < 0)
        return fail(CCL_ERR_INVALID_ARG, "CCL_SCHEDULE=%s is not ring, allpairs or auto", getenv("CCL_SCHEDULE"));
    L.table = get_table(c, n, sched);
    for (int k = 0; k <= p && aligned; ++k) aligned = L.table->bound[k] % vec_elems == 0;
    L.vec = aligned;
    NormLaunch N;
    N.residual = residual_in;
    N.residual_out = residual_out;
    N.gamma = gamma;
    N.rows = rows;
    N.hidden = hidden;
    N.eps = eps;
    LaunchInfo info;
    cudaError_t err = launch_allreduce_rmsnorm(L, N, &info);
    c->launches += uint64_t(info.kernels);
    snprintf(c->last, sizeof c->last,
             "%s dtype=%s op=sum p=%d n=%zu rows=%zu hidden=%zu schedule=%s vec=%d grid=%d block=%d", info.kernel,
             kDtypeName[dtype], p, n, rows, hidden, kSchedName[sched], L.vec ? 1 : 0, info.grid, info.block);
    if (debug_on()) fprintf(stderr, "[ccl] %s\n", c->last);
    if (err != cudaSuccess) return cuda_fail(err, "allreduce_residual_rmsnorm");
    return CCL_OK;
}
