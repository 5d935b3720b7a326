// ccl_allreduce_static: AllReduce for callers that cannot allocate device
// memory.
//
// Who needs it: code that runs where device allocation is off limits -- a
// plug-in inside a host application (an inference server, a framework's
// memory pool) that owns all device memory and forbids further cudaMalloc, a
// process that has already committed its memory budget, or code that must not
// meet an out-of-memory failure once it runs.  The communicator API allocates
// a small status block per communicator; this entry point allocates nothing.
//
// What it runs: the TMA variant's AllReduce kernel (tma.cuh) with its static
// tile split (no tile counter).  That kernel's only memory beyond the
// caller's inputs and outputs is then the status record its bounded waits
// write when one gives up.  Here the record lives in
// a file-scope device array of this library, kStaticScratchBytes long, which
// every GPU that loads the library holds until the process exits.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "ccl.h"
#include "internal.h"

namespace {

constexpr size_t kStaticScratchBytes = 256;               // the array's size: the stated maximum
constexpr size_t kStatusBytes = 4 * sizeof(unsigned);     // code, block, tile, thread
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Per-device set-up: the array's device address (host code cannot use the
// symbol itself, which only names a host-side stand-in) and the SM count.
struct DeviceSlot {
    bool ready = false;
    void *scratch = nullptr;
    int num_sms = 0;
};
std::mutex g_mu;
DeviceSlot g_slots[kMaxDevices];

// Test hook (ccl_allreduce_static_set_debug): the bound on each wait of the
// kernel and the producer's withheld tile.
constexpr long long kDefaultWaitNs = 2000000000LL;
std::atomic<long long> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_stall{0};

ccl_status_t fail(ccl_status_t st, const char *fmt, ...)
{
    char buf[400];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    return ccl::record_error(st, buf);
}

ccl_status_t cuda_fail(cudaError_t err, const char *what)
{
    return fail(CCL_ERR_CUDA, "ccl_allreduce_static: %s: %s (%s)", what, cudaGetErrorName(err),
                cudaGetErrorString(err));
}

bool disjoint(uintptr_t a, uintptr_t b, size_t bytes) { return a + bytes <= b || b + bytes <= a; }

}  // namespace

extern "C" ccl_status_t ccl_allreduce_static(int p, void *const *in_ptrs, void *const *out_ptrs, ccl_op_t op,
                                             ccl_dtype_t dtype, size_t n, ccl_schedule_t schedule, void *stream)
{
    using namespace ccl;
    if (p < 1 || p > kMaxRanks) return fail(CCL_ERR_INVALID_ARG, "ccl_allreduce_static: p=%d outside [1, %d]", p, kMaxRanks);
    if (!in_ptrs || !out_ptrs) return fail(CCL_ERR_INVALID_ARG, "ccl_allreduce_static: NULL pointer array");
    for (int r = 0; r < p; ++r)
        if (!in_ptrs[r] || !out_ptrs[r])
            return fail(CCL_ERR_INVALID_ARG, "ccl_allreduce_static: buffer %d is NULL", r);
    if (op < CCL_SUM || op > CCL_AVG) return fail(CCL_ERR_INVALID_ARG, "ccl_allreduce_static: unknown op %d", int(op));
    if (dtype < CCL_F32 || dtype > CCL_I32)
        return fail(CCL_ERR_INVALID_ARG, "ccl_allreduce_static: unknown dtype %d", int(dtype));
    if (schedule != CCL_SCHED_AUTO && schedule != CCL_SCHED_RING && schedule != CCL_SCHED_ALLPAIRS)
        return fail(CCL_ERR_INVALID_ARG, "ccl_allreduce_static: schedule must be auto, ring or all-pairs");
    // The kernel's scratch is one status record, the same for every p and n;
    // anything that needed more than the static array would be refused here.
    if (kStatusBytes > kStaticScratchBytes)
        return fail(CCL_ERR_INVALID_ARG, "ccl_allreduce_static: needs %zu scratch bytes, the static array holds %zu",
                    kStatusBytes, kStaticScratchBytes);
    const size_t s = elem_bytes(dtype);
    if (n > (SIZE_MAX / 2) / s) return fail(CCL_ERR_INVALID_ARG, "ccl_allreduce_static: n=%zu too large", n);

    // Aliasing: in place (out[r] == in[r]) or disjoint from every buffer.
    const size_t bytes = n * s;
    for (int k = 0; k < p; ++k) {
        const uintptr_t o = uintptr_t(out_ptrs[k]);
        for (int j = 0; j < p; ++j) {
            if (j != k && !disjoint(o, uintptr_t(out_ptrs[j]), bytes))
                return fail(CCL_ERR_INVALID_ARG, "ccl_allreduce_static: outputs of ranks %d and %d overlap", k, j);
            const uintptr_t i = uintptr_t(in_ptrs[j]);
            if (!disjoint(o, i, bytes) && !(j == k && o == i))
                return fail(CCL_ERR_INVALID_ARG, "ccl_allreduce_static: output of rank %d overlaps input of rank %d", k, j);
        }
    }

    // Schedule table (ring / all-pairs through the public builder).
    const int sched = schedule == CCL_SCHED_AUTO ? int(ccl_select_schedule(p, double(bytes), nullptr)) : int(schedule);
    Table table;
    table.p = p;
    table.n = n;
    if (ccl_schedule_build(p, n, ccl_schedule_t(sched), table.bound, table.order) != CCL_OK)
        return fail(CCL_ERR_INVALID_ARG, "ccl_allreduce_static: schedule table could not be built");

    // The TMA kernel moves 16-byte multiples between 16-byte aligned addresses.
    bool ok = true;
    for (int r = 0; r < p; ++r)
        ok = ok && uintptr_t(in_ptrs[r]) % 16 == 0 && uintptr_t(out_ptrs[r]) % 16 == 0;
    for (int c = 0; c <= p && ok; ++c) ok = (table.bound[c] * s) % 16 == 0;
    if (!ok)
        return fail(CCL_ERR_UNSUPPORTED,
                    "ccl_allreduce_static: needs 16-byte aligned buffers and chunk boundaries (n=%zu, p=%d)", n, p);
    uint32_t tile, stages, ranks;
    size_t smem;
    if (!(p > kTmaNarrowMaxRanks ? tma_wide_geometry(p, 0, 0, &tile, &ranks, &stages, &smem)
                                 : tma_geometry(p, 0, 0, &tile, &stages, &smem)))
        return fail(CCL_ERR_UNSUPPORTED, "ccl_allreduce_static: no shared-memory pipeline fits p=%d", p);
    if (n == 0) return CCL_OK;

    // Set-up, once per device, with that device current.
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(CCL_ERR_UNSUPPORTED, "ccl_allreduce_static: device %d", dev);
    void *scratch = nullptr;
    int num_sms = 0;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        DeviceSlot &slot = g_slots[dev];
        if (!slot.ready) {
            err = cudaGetSymbolAddress(&slot.scratch, g_static_scratch);
            if (err != cudaSuccess) return cuda_fail(err, "cudaGetSymbolAddress");
            err = cudaDeviceGetAttribute(&slot.num_sms, cudaDevAttrMultiProcessorCount, dev);
            if (err != cudaSuccess) return cuda_fail(err, "cudaDeviceGetAttribute");
            slot.ready = true;
        }
        scratch = slot.scratch;
        num_sms = slot.num_sms;
    }

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // A bounded wait that gave up in the previous call on this device left its
    // record here: report it (after the work already queued on `stream` is done)
    // instead of launching.
    unsigned prev[4] = {0, 0, 0, 0};
    err = cudaMemcpyAsync(prev, scratch, kStatusBytes, cudaMemcpyDeviceToHost, st);
    if (err == cudaSuccess) err = cudaStreamSynchronize(st);
    if (err != cudaSuccess) return cuda_fail(err, "reading the status record");
    // The record must start at zero for this call.
    err = cudaMemsetAsync(scratch, 0, kStatusBytes, st);
    if (err != cudaSuccess) return cuda_fail(err, "clearing the status record");
    if (prev[0] == kBoundsCode)
        return fail(CCL_ERR_BOUNDS,
                    "ccl_allreduce_static: the previous call computed an access outside a rank buffer and skipped it "
                    "(site %u, block %u, index %u); its outputs are incomplete",
                    prev[3], prev[1], prev[2]);
    if (prev[0] != 0)
        return fail(CCL_ERR_TIMEOUT,
                    "ccl_allreduce_static: a bounded device wait of the previous call gave up "
                    "(code %u, block %u, tile %u); its outputs are incomplete",
                    prev[0], prev[1], prev[2]);

    Launch L;
    L.p = p;
    L.op = op;
    L.dtype = dtype;
    L.mode = MODE_AR;
    L.n = n;
    for (int r = 0; r < p; ++r) {
        L.src[r] = in_ptrs[r];
        L.dst[r] = out_ptrs[r];
    }
    L.table = &table;
    L.vec = true;
    L.device = dev;
    L.num_sms = num_sms;
    L.sm_budget = 0;
    L.pipe_bytes = 0;
    L.status = static_cast<unsigned *>(scratch);
    L.tile_counter = false;  // the static split: nothing shared between calls but the status record
    L.wait_limit_ns = g_wait_ns.load();
    L.stall_test = g_stall.load();
    L.stream = st;
    LaunchInfo info;
    switch (dtype) {
    case CCL_F32: err = launch_tma_f32(L, &info); break;
    case CCL_F16: err = launch_tma_f16(L, &info); break;
    case CCL_BF16: err = launch_tma_bf16(L, &info); break;
    default: err = launch_tma_i32(L, &info); break;
    }
    if (err != cudaSuccess) return cuda_fail(err, "kernel launch");
    return CCL_OK;
}

extern "C" ccl_status_t ccl_allreduce_static_set_debug(long long wait_limit_ns, int stall_test)
{
    if (wait_limit_ns < 0 || stall_test < 0 || stall_test > 1)
        return fail(CCL_ERR_INVALID_ARG, "ccl_allreduce_static_set_debug: wait_limit_ns %lld / stall_test %d out of range",
                    wait_limit_ns, stall_test);
    g_wait_ns.store(wait_limit_ns ? wait_limit_ns : kDefaultWaitNs);
    g_stall.store(stall_test);
    return CCL_OK;
}
