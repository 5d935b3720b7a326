// Multi-source reduce: the core of ReduceScatter and, fused with the
// broadcast store, of AllReduce.
//
// "Inside NCCL AllReduce", section "The ring, exactly as the kernel runs it":
// the ring all-reduce is one fused loop whose workhorse step receives a
// partial sum, adds the local contribution in registers and forwards it,
// never storing partials in between.  With all p ranks in one GPU's memory
// the p-1 hops of a chunk collapse into one thread: it loads the p
// contributions of a 16-byte group (one 128-bit load per rank), folds them in
// fp32 in exactly the chunk's rank order, rounds once, and stores the result
// to every rank (AllReduce) or to the chunk's owner (ReduceScatter).  Bytes
// moved are the minimum: p*n*s read, p*n*s (AR) or n*s (RS) written.
//
// Work split: the buffer is a flat sequence of 16-byte groups, one per
// thread: the grid covers the buffer once and the hardware block scheduler
// streams CTAs through the SMs (measured faster on GB300 than a persistent
// grid-stride sweep: 6.86 vs 6.41 TB/s at p=8).  An SM budget caps the grid
// instead, and the loop then strides.  A group lying wholly in one chunk takes
// the vector path; a group straddling a chunk boundary (only when a chunk size
// is not a multiple of the group) and the sub-group tail are done element by
// element with each element's own chunk order.
#pragma once

#include "device.cuh"

namespace ccl {

// Threads per CTA.  Whole GPU (one group per thread, the block scheduler
// streaming CTAs): 256 for p <= 8, 128 where the p loads in flight need more
// registers (p = 16: 110 registers) so that CTAs stay small.  Under an SM
// budget (one persistent CTA per SM) the CTA must carry the SM's whole load
// queue: 1024 threads for p <= 8, 512 otherwise -- measured on GB300 at 8 SMs,
// p=8: 808 GB/s with 1024 threads against 368 with 256.
template <int P>
constexpr int reduce_threads() { return (P == 0 || P >= 16) ? 128 : 256; }
template <int P>
constexpr int reduce_budget_threads() { return (P == 0 || P >= 16) ? 512 : 1024; }

template <int PM>
struct ReduceArgs {
    const void *src[PM];        // rank inputs
    void *dst[PM];              // rank outputs (RS: dst[c] receives chunk c from offset 0)
    uint64_t bound[PM + 1];     // chunk c = elements [bound[c], bound[c+1])
    uint8_t order[PM][PM];      // order[c][k]: k-th rank folded into chunk c
    uint64_t n;                 // elements per rank
    int p;
    int vec;                    // 1: 16-byte groups allowed (all pointers aligned)
    float scale;                // avg: fl32(1/p)
    unsigned *status;           // status block: words 8-9 group counter, 10 finished CTAs
    int dynamic;                // 1: warps beyond their first block take groups from the counter
};

// One element e of chunk c, folded in the chunk's order.
template <typename T, int OP, int MODE, int PM>
__device__ __forceinline__ void reduce_one(const ReduceArgs<PM> &a, int p, int c, uint64_t e)
{
    using Tr = Traits<T>;
    using F = Fold<T, OP>;
    // every rank buffer holds n elements; chunk c is [bound[c], bound[c+1])
    if (!in_bounds(e < a.n && e >= a.bound[c] && e < a.bound[c + 1], a.status, kSiteReduceElem, e)) return;
    if constexpr (kSelect16<T, OP>) {
        // min/max of a 16-bit type: keep the chosen input's own bits, as the
        // packed group fold does (the fp32 compare picks the same operand)
        const uint16_t *s0 = static_cast<const uint16_t *>(a.src[a.order[c][0]]);
        uint16_t keep = s0[e];
        float acc = Tr::load1(s0, e);
        for (int k = 1; k < p; ++k) {
            const uint16_t *sk = static_cast<const uint16_t *>(a.src[a.order[c][k]]);
            const float v = Tr::load1(sk, e);
            if (OP == OP_MIN ? v < acc : v > acc) {
                acc = v;
                keep = sk[e];
            }
        }
        if constexpr (MODE == MODE_AR) {
            for (int k = 0; k < p; ++k) static_cast<uint16_t *>(a.dst[k])[e] = keep;
        } else {
            static_cast<uint16_t *>(a.dst[c])[e - a.bound[c]] = keep;
        }
        return;
    }
    auto acc = F::first(Tr::load1(a.src[a.order[c][0]], e), a.scale);
    for (int k = 1; k < p; ++k)
        acc = F::fold(acc, Tr::load1(a.src[a.order[c][k]], e), a.scale);
    const auto out = F::finish(acc, p);
    if constexpr (MODE == MODE_AR) {
        for (int k = 0; k < p; ++k) Tr::store1(a.dst[k], e, out);
    } else {
        Tr::store1(a.dst[c], e - a.bound[c], out);
    }
}

// P > 0: p fixed at compile time (loads fully unrolled); P == 0: any p up to
// kMaxRanks, loads issued eight at a time.
template <typename T, int OP, int P, int MODE, bool DYN, bool NC>
__device__ __forceinline__ void reduce_body(const ReduceArgs<(P > 0 ? P : kMaxRanks)> &a)
{
    using Tr = Traits<T>;
    using Acc = typename Tr::Acc;
    constexpr int VEC = Tr::VEC;
    constexpr int ES = int(sizeof(Acc));     // element bytes of the 4-byte types
    constexpr int S = (VEC == 8) ? 2 : ES;   // element bytes
    const int p = P > 0 ? P : a.p;

    const uint64_t tid = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
    const uint64_t ngroups = a.vec ? a.n / VEC : 0;

    int c = 0;
    uint64_t cend = a.bound[1];
    const char *sp[P > 0 ? P : 1];  // P > 0: chunk c's sources, already in fold order
    if constexpr (P > 0) {
#pragma unroll
        for (int k = 0; k < P; ++k) sp[k] = static_cast<const char *>(a.src[a.order[0][k]]);
    }

    auto seek = [&](uint64_t e) {
        if (e >= cend) {  // next chunk(s); empty chunks are skipped
            do { ++c; } while (e >= a.bound[c + 1]);
            cend = a.bound[c + 1];
            if constexpr (P > 0) {
#pragma unroll
                for (int k = 0; k < P; ++k) sp[k] = static_cast<const char *>(a.src[a.order[c][k]]);
            }
        }
    };
    auto group = [&](uint64_t g) {
        const uint64_t e = g * VEC;
        seek(e);
        if (!in_bounds(e + VEC <= a.n && e >= a.bound[c], a.status, kSiteReduceGroup, e)) return;
        if (e + VEC > cend) {  // straddles a chunk boundary: per element
            int cj = c;
            for (int j = 0; j < VEC; ++j) {
                while (e + j >= a.bound[cj + 1]) ++cj;
                reduce_one<T, OP, MODE>(a, p, cj, e + j);
            }
            return;
        }
        GroupFold<T, OP> acc;
        if constexpr (P > 0) {
            uint4 r[P];
#pragma unroll
            for (int k = 0; k < P; ++k) r[k] = ld_in_v4<NC>(sp[k] + e * S);
            acc.first(r[0], a.scale);
#pragma unroll
            for (int k = 1; k < P; ++k) acc.fold(r[k], a.scale);
        } else {
            for (int k0 = 0; k0 < p; k0 += 8) {
                uint4 r[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (k0 + j < p)
                        r[j] = ld_in_v4<NC>(static_cast<const char *>(a.src[a.order[c][k0 + j]]) + e * S);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (k0 + j < p) {
                        if (k0 + j == 0) acc.first(r[j], a.scale);
                        else acc.fold(r[j], a.scale);
                    }
                }
            }
        }
        const uint4 out = acc.finish(p);
        if constexpr (MODE == MODE_AR) {
            if constexpr (P > 0) {
#pragma unroll
                for (int k = 0; k < P; ++k) st_stream_v4(static_cast<char *>(a.dst[k]) + e * S, out);
            } else {
                for (int k = 0; k < p; ++k) st_stream_v4(static_cast<char *>(a.dst[k]) + e * S, out);
            }
        } else {
            st_stream_v4(static_cast<char *>(a.dst[c]) + (e - a.bound[c]) * S, out);
        }
    };
    // Under an SM budget with p <= 4 each thread takes GB groups at a time
    // (g0, g0 + step, ...), all loads issued before the first fold, so that
    // it has eight 16-byte loads in flight as at p = 8 (one group of p loads
    // left the SM's load queue short: p=2 on 8 SMs moved 86 GB/s per SM,
    // stalled on its loads).  Each group is folded as by group(): same bits.
    constexpr int GB = (DYN && P > 0 && P <= 4) ? 8 / P : 1;
    auto batch = [&](uint64_t g0, uint64_t step) {  // GB groups, all < ngroups
        if constexpr (GB > 1) {
            seek(g0 * VEC);
            if ((g0 + uint64_t(GB - 1) * step) * VEC + VEC > cend) {  // not all in this chunk
#pragma unroll 1
                for (int i = 0; i < GB; ++i) group(g0 + uint64_t(i) * step);
                return;
            }
            const uint64_t elast = (g0 + uint64_t(GB - 1) * step) * VEC;
            if (!in_bounds(elast + VEC <= a.n && g0 * VEC >= a.bound[c], a.status, kSiteReduceGroup, elast)) return;
            uint4 r[GB][P > 0 ? P : 1];
#pragma unroll
            for (int i = 0; i < GB; ++i)
#pragma unroll
                for (int k = 0; k < P; ++k) r[i][k] = ld_in_v4<NC>(sp[k] + (g0 + uint64_t(i) * step) * VEC * S);
#pragma unroll
            for (int i = 0; i < GB; ++i) {
                const uint64_t e = (g0 + uint64_t(i) * step) * VEC;
                GroupFold<T, OP> acc;
                acc.first(r[i][0], a.scale);
#pragma unroll
                for (int k = 1; k < P; ++k) acc.fold(r[i][k], a.scale);
                const uint4 out = acc.finish(p);
                if constexpr (MODE == MODE_AR) {
#pragma unroll
                    for (int k = 0; k < P; ++k) st_stream_v4(static_cast<char *>(a.dst[k]) + e * S, out);
                } else {
                    st_stream_v4(static_cast<char *>(a.dst[c]) + (e - a.bound[c]) * S, out);
                }
            }
        } else {
            group(g0);
        }
    };
    if (!DYN || !a.dynamic) {
        if constexpr (GB > 1) {
            uint64_t g = tid;
            for (; g + uint64_t(GB - 1) * stride < ngroups; g += uint64_t(GB) * stride) batch(g, stride);
            for (; g < ngroups; g += stride) group(g);
        } else {
            for (uint64_t g = tid; g < ngroups; g += stride) group(g);
        }
    } else {
        // Each warp takes blocks of 32 * kWarpGrab consecutive groups: its
        // first statically, the rest from the status block's group counter,
        // so that SMs that run faster take more -- with no CTA barrier (a
        // CTA-wide grab cost more in barriers than it gained).  Measured at
        // p=16 on 90 SMs: 6545 -> 6866 GB/s; p=2 on 76 SMs 5046 -> 5272; no
        // change at 8-32 SMs.
        constexpr int kWarpGrab = 16;
        static_assert(kWarpGrab % GB == 0, "a warp's block is whole batches");
        const uint32_t lane = threadIdx.x & 31u;
        const uint64_t per = 32ull * kWarpGrab;
        const uint64_t warps = uint64_t(gridDim.x) * (blockDim.x / 32);
        unsigned long long *next = reinterpret_cast<unsigned long long *>(a.status + 8);
        uint64_t base = (uint64_t(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32) * per;
        while (base < ngroups) {
            unsigned long long nb = 0;
            if (lane == 0) nb = warps * per + atomicAdd(next, (unsigned long long)per);
#pragma unroll 1
            for (int j = 0; j < kWarpGrab; j += GB) {
                const uint64_t g = base + lane + uint64_t(j) * 32;
                if (g + uint64_t(GB - 1) * 32 < ngroups) {
                    batch(g, 32);
                } else {
                    for (int i = 0; i < GB; ++i)
                        if (g + uint64_t(i) * 32 < ngroups) group(g + uint64_t(i) * 32);
                }
            }
            base = __shfl_sync(0xffffffffu, nb, 0);
        }
    }

    // Elements after the last whole group (every element when vec == 0).
    int ct = 0;
    for (uint64_t e = ngroups * VEC + tid; e < a.n; e += stride) {
        while (e >= a.bound[ct + 1]) ++ct;
        reduce_one<T, OP, MODE>(a, p, ct, e);
    }
}

// Whole GPU: the compiler's own register choice (62 at p=8 bf16: four
// 256-thread CTAs per SM).
// Launched as a dependent: the next kernel may be scheduled once the last
// wave of CTAs is running.
template <typename T, int OP, int P, int MODE, bool NC>
__global__ void __launch_bounds__(reduce_threads<P>())
    reduce_kernel(const __grid_constant__ ReduceArgs<(P > 0 ? P : kMaxRanks)> a)
{
    grid_dependency_wait();
    grid_dependents_launch();
    reduce_body<T, OP, P, MODE, false, NC>(a);
}

// fp32 sum, prod and avg at p = 5 or 6 through the generic kernel: the same
// body with eight 128-thread CTAs per SM asked of the compiler (64
// registers, no spills) instead of its seven.  Measured on GB300 over 4 GiB
// of inputs, fp32 sum: p=5 6.60 -> 7.15 TB/s, p=6 6.93 -> 7.13.  int32, min
// and max, and p = 7, gained nothing (within 0.4 % either way).
template <typename T, int OP, int P, int MODE, bool NC>
__global__ void __launch_bounds__(reduce_threads<P>(), 8)
    reduce_kernel_occ8(const __grid_constant__ ReduceArgs<(P > 0 ? P : kMaxRanks)> a)
{
    grid_dependency_wait();
    grid_dependents_launch();
    reduce_body<T, OP, P, MODE, false, NC>(a);
}

// fp16/bf16 min/max at p = 8 (the packed select fold): the same body, with
// five CTAs per SM asked of the compiler (48 registers, no spills) instead
// of its own four.  The compare -> select chain keeps each thread's loads
// outstanding for longer than a sum's adds do, so more resident threads pay:
// 6.72 -> 6.89 TB/s on GB300 (six CTAs: 6.81; at p = 4 neither helped).
template <typename T, int OP, int P, int MODE, bool NC>
__global__ void __launch_bounds__(reduce_threads<P>(), 5)
    reduce_kernel_occ5(const __grid_constant__ ReduceArgs<(P > 0 ? P : kMaxRanks)> a)
{
    grid_dependency_wait();
    grid_dependents_launch();
    reduce_body<T, OP, P, MODE, false, NC>(a);
}

// SM budget: one large CTA per SM, so the full register file per thread.
// Persistent, so the next kernel is scheduled only as its CTAs exit.
template <typename T, int OP, int P, int MODE, bool NC>
__global__ void __launch_bounds__(reduce_budget_threads<P>(), 1)
    reduce_budget_kernel(const __grid_constant__ ReduceArgs<(P > 0 ? P : kMaxRanks)> a)
{
    grid_dependency_wait();
    reduce_body<T, OP, P, MODE, true, NC>(a);
    if (a.dynamic) {
        __syncthreads();
        if (threadIdx.x == 0 && atomicAdd(a.status + 10, 1u) == gridDim.x - 1) {
            atomicExch(reinterpret_cast<unsigned long long *>(a.status + 8), 0ull);
            atomicExch(a.status + 10, 0u);
        }
    }
}

// ---------------------------------------------------------------------------
// Host side: pick the instantiation, fill the argument block, size the grid.
// ---------------------------------------------------------------------------

template <typename T, int OP, int P, int MODE, bool NC>
static cudaError_t launch_p(const Launch &L, LaunchInfo *info)
{
    constexpr int PM = P > 0 ? P : kMaxRanks;
    ReduceArgs<PM> a;
    for (int k = 0; k < L.p; ++k) {
        a.src[k] = L.src[k];
        a.dst[k] = L.dst[k];
    }
    for (int c = 0; c <= L.p; ++c) a.bound[c] = L.table->bound[c];
    for (int c = 0; c < L.p; ++c)
        for (int k = 0; k < L.p; ++k) a.order[c][k] = L.table->order[c * L.p + k];
    a.n = L.n;
    a.p = L.p;
    a.vec = L.vec ? 1 : 0;
    a.scale = 1.0f / float(L.p);
    a.status = L.status;
    a.dynamic = 0;

    // An SM budget takes the persistent large-CTA kernel, unless the whole
    // message already fits in at most `budget` small CTAs (small messages:
    // the regular kernel's latency, and still no more than budget CTAs).
    const uint64_t units = L.vec ? (L.n / Traits<T>::VEC + L.n % Traits<T>::VEC) : L.n;
    const uint64_t small_grid = (units + reduce_threads<P>() - 1) / reduce_threads<P>();
    const bool budget = L.sm_budget > 0 && L.sm_budget < L.num_sms && small_grid > uint64_t(L.sm_budget);
    auto kern = budget ? reduce_budget_kernel<T, OP, P, MODE, NC> : reduce_kernel<T, OP, P, MODE, NC>;
    if constexpr (kSelect16<T, OP> && P == 8) {
        if (!budget) kern = reduce_kernel_occ5<T, OP, P, MODE, NC>;
    }
    if constexpr (P == 0 && std::is_same<T, F32>::value && OP != OP_MIN && OP != OP_MAX) {
        if (!budget && L.p <= 6) kern = reduce_kernel_occ8<T, OP, P, MODE, NC>;
    }
    const int kThreads = budget ? reduce_budget_threads<P>() : reduce_threads<P>();
    uint64_t want = (units + kThreads - 1) / kThreads;
    if (want < 1) want = 1;
    uint64_t cap = uint64_t(0x7fffffff);
    size_t smem = 0;
    if (budget) {
        // persistent CTAs, at most one per SM: ask for more than half of an
        // SM's shared memory so that no two fit on one SM
        cap = uint64_t(L.sm_budget);
        smem = 120 * 1024;
        static std::atomic<unsigned long long> attr{0};  // devices on which the limit is raised
        {
            const cudaError_t err = allow_dynamic_smem(kern, smem, L.device, attr);
            if (err != cudaSuccess) return err;
        }
    }
    const int grid = int(want < cap ? want : cap);
    if (budget && a.vec) {
        // the counter pays off once every warp has about 16 blocks to take
        const uint64_t ngroups = L.n / Traits<T>::VEC;
        a.dynamic = ngroups >= 16ull * 32 * 16 * uint64_t(kThreads / 32) * uint64_t(grid) ? 1 : 0;
    }
    cudaError_t err = launch_dependent(kern, unsigned(grid), unsigned(kThreads), smem, L.stream, a);
    if (err != cudaSuccess) return err;
    if (info) {
        info->kernel = MODE == MODE_AR ? "allreduce_ldst" : "reduce_scatter_ldst";
        info->grid = grid;
        info->block = kThreads;
        info->smem = smem;
        info->kernels = 1;
        info->counter = a.dynamic;
    }
    return cudaGetLastError();
}

template <typename T, int OP, int MODE, bool NC>
static cudaError_t launch_op_mode(const Launch &L, LaunchInfo *info)
{
    switch (L.p) {
    case 2: return launch_p<T, OP, 2, MODE, NC>(L, info);
    case 3: return launch_p<T, OP, 3, MODE, NC>(L, info);
    case 4: return launch_p<T, OP, 4, MODE, NC>(L, info);
    case 8: return launch_p<T, OP, 8, MODE, NC>(L, info);
    case 16: return launch_p<T, OP, 16, MODE, NC>(L, info);
    default: return launch_p<T, OP, 0, MODE, NC>(L, info);
    }
}

template <typename T, int OP, bool NC>
static cudaError_t launch_op(const Launch &L, LaunchInfo *info)
{
    return L.mode == MODE_AR ? launch_op_mode<T, OP, MODE_AR, NC>(L, info)
                             : launch_op_mode<T, OP, MODE_RS, NC>(L, info);
}

// NC = true: no output overlaps an input (ld.global.nc); false: the in-place
// instantiation, compiled in its own translation unit.
template <typename T, bool NC>
static cudaError_t launch_reduce(const Launch &L, LaunchInfo *info)
{
    switch (L.op) {
    case OP_SUM: return launch_op<T, OP_SUM, NC>(L, info);
    case OP_PROD: return launch_op<T, OP_PROD, NC>(L, info);
    case OP_MIN: return launch_op<T, OP_MIN, NC>(L, info);
    case OP_MAX: return launch_op<T, OP_MAX, NC>(L, info);
    case OP_AVG: return launch_op<T, OP_AVG, NC>(L, info);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ccl
