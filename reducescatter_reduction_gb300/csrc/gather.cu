// AllGather as a broadcast store.
//
// "Inside NCCL AllReduce", section "The ring, exactly as the kernel runs it":
// in the all-gather half the finished chunks circulate unchanged; T-CCL,
// section "Chunk and Window Decomposition", fans one load out to every
// destination.  With all ranks in one GPU's memory: chunk c is read once from
// its owner's buffer and stored to every rank's output at the same offset
// (n*s read, p*n*s written; in place, the owner's own copy is skipped).
#include "device.cuh"

namespace ccl {

constexpr int kGatherThreads = 256;        // whole GPU: one unit per thread
constexpr int kGatherBudgetThreads = 1024; // SM budget: one persistent CTA per SM carries its load queue

template <int PM>
struct GatherArgs {
    const void *src[PM];    // rank r's buffer; only its chunk r is read
    void *dst[PM];          // rank outputs, n elements each
    uint64_t chunk_units;   // units (of U bytes) per chunk
    uint64_t nunits;        // p * chunk_units
    int p;
    uint64_t self_mask;     // bit c: dst[c] == src[c], so the owner's chunk is not rewritten
    uint64_t buf_units;     // units in every rank buffer (checked build: the extent each access is tested against)
    unsigned *status;       // the communicator's status block (checked build: where a violation is recorded)
};

template <int U> struct Unit;
template <> struct Unit<16> {
    using type = uint4;
    __device__ static uint4 load(const char *p) { return ld_stream_v4(p); }
    __device__ static void store(char *p, const uint4 &v) { st_stream_v4(p, v); }
};
template <> struct Unit<4> {
    using type = uint32_t;
    __device__ static uint32_t load(const char *p) { return *reinterpret_cast<const uint32_t *>(p); }
    __device__ static void store(char *p, uint32_t v) { *reinterpret_cast<uint32_t *>(p) = v; }
};
template <> struct Unit<2> {
    using type = uint16_t;
    __device__ static uint16_t load(const char *p) { return *reinterpret_cast<const uint16_t *>(p); }
    __device__ static void store(char *p, uint16_t v) { *reinterpret_cast<uint16_t *>(p) = v; }
};

template <int P, int U, int THREADS>
__global__ void __launch_bounds__(THREADS, 1)
    gather_kernel(const __grid_constant__ GatherArgs<(P > 0 ? P : kMaxRanks)> a)
{
    grid_dependency_wait();
    if (THREADS == kGatherThreads) grid_dependents_launch();  // not in the persistent SM-budget kernel
    const int p = P > 0 ? P : a.p;
    const uint64_t tid = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
    int c = 0;
    uint64_t cend = a.chunk_units;
    const char *sc = static_cast<const char *>(a.src[0]);
    for (uint64_t u = tid; u < a.nunits; u += stride) {
        if (u >= cend) {
            c = int(u / a.chunk_units);
            cend = uint64_t(c + 1) * a.chunk_units;
            sc = static_cast<const char *>(a.src[c]);
        }
        if (!in_bounds(u < a.buf_units && u >= uint64_t(c) * a.chunk_units && c < p, a.status, kSiteGather, u)) continue;
        const auto v = Unit<U>::load(sc + u * U);
        if constexpr (P > 0) {
#pragma unroll
            for (int k = 0; k < P; ++k)
                if (!(k == c && ((a.self_mask >> c) & 1u))) Unit<U>::store(static_cast<char *>(a.dst[k]) + u * U, v);
        } else {
            for (int k = 0; k < p; ++k)
                if (!(k == c && ((a.self_mask >> c) & 1u))) Unit<U>::store(static_cast<char *>(a.dst[k]) + u * U, v);
        }
    }
}

template <int P, int U>
static cudaError_t gather_launch(const Launch &L, LaunchInfo *info)
{
    constexpr int PM = P > 0 ? P : kMaxRanks;
    GatherArgs<PM> a;
    for (int k = 0; k < L.p; ++k) {
        a.src[k] = L.src[k];
        a.dst[k] = L.dst[k];
    }
    const uint64_t chunk_bytes = L.n / L.p * elem_bytes(L.dtype);
    a.chunk_units = chunk_bytes / U;
    a.nunits = a.chunk_units * L.p;
    a.p = L.p;
    a.self_mask = L.self_mask;
    a.buf_units = uint64_t(L.n) * elem_bytes(L.dtype) / U;
    a.status = L.status;

    // the persistent large-CTA kernel only when the message does not already
    // fit in at most `budget` small CTAs
    const uint64_t small_grid = (a.nunits + kGatherThreads - 1) / kGatherThreads;
    const bool budget = L.sm_budget > 0 && L.sm_budget < L.num_sms && small_grid > uint64_t(L.sm_budget);
    auto kern = budget ? gather_kernel<P, U, kGatherBudgetThreads> : gather_kernel<P, U, kGatherThreads>;
    const int threads = budget ? kGatherBudgetThreads : kGatherThreads;
    // one unit per thread; the block scheduler streams CTAs through the SMs
    uint64_t want = (a.nunits + threads - 1) / threads;
    if (want < 1) want = 1;
    uint64_t cap = uint64_t(0x7fffffff);
    size_t smem = 0;
    if (budget) {
        cap = uint64_t(L.sm_budget);
        smem = 120 * 1024;  // at most one CTA per SM
        static std::atomic<unsigned long long> attr{0};  // devices on which the limit is raised
        {
            const cudaError_t err = allow_dynamic_smem(kern, smem, L.device, attr);
            if (err != cudaSuccess) return err;
        }
    }
    const int grid = int(want < cap ? want : cap);
    cudaError_t err = launch_dependent(kern, unsigned(grid), unsigned(threads), smem, L.stream, a);
    if (err != cudaSuccess) return err;
    if (info) {
        info->kernel = "all_gather_ldst";
        info->grid = grid;
        info->block = threads;
        info->smem = smem;
        info->kernels = 1;
    }
    return cudaGetLastError();
}

template <int U>
static cudaError_t gather_unit(const Launch &L, LaunchInfo *info)
{
    switch (L.p) {
    case 2: return gather_launch<2, U>(L, info);
    case 4: return gather_launch<4, U>(L, info);
    case 8: return gather_launch<8, U>(L, info);
    case 16: return gather_launch<16, U>(L, info);
    default: return gather_launch<0, U>(L, info);
    }
}

cudaError_t launch_gather(const Launch &L, LaunchInfo *info)
{
    if (L.vec) return gather_unit<16>(L, info);
    return elem_bytes(L.dtype) == 2 ? gather_unit<2>(L, info) : gather_unit<4>(L, info);
}

}  // namespace ccl
