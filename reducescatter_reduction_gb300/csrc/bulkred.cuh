// TMA bulk-reduce variant: the memory system applies the reduction.
//
// T-CCL, sections "TMA Transfer Engine" and "Pipelined Copy and Reduction":
// TMA also performs asynchronous element-wise reductions into global memory
// (add, min, max), so a shard's owner can accumulate every contribution
// without SM arithmetic.  Here, per tile of chunk c:
//
//   producer lane:  p x cp.async.bulk global->shared (every rank's tile)
//   issuer lane:    cp.async.bulk shared->global of the first contribution into
//                   the chunk's destination, wait until it has landed, then
//                   p-1 x cp.reduce.async.bulk shared->global into it
//
// This is the ReduceScatter core; an AllReduce is this kernel writing chunk c
// into rank c's output at the chunk's own offset, followed by the in-place
// AllGather broadcast.  The order in which the memory system applies the p-1
// reductions is not fixed, and fp16/bf16 partials are rounded to the element
// type at every step, so results are held to the reassociation bound
// |err| <= 2 p eps sum_k |x_k| instead of bit equality (min/max and int32 sum
// are exact in any order).  Supported: sum on f32/f16/bf16/i32, min/max on
// f16/bf16/i32 -- the combinations the PTX bulk-reduce instruction provides.
#pragma once

#include "tma.cuh"

namespace ccl {

constexpr int kBulkThreads = 64;  // one pipe: warp 0's lane 0 loads, warp 1's lane 0 issues
constexpr int kBulkMaxPipes = 4;

// Shared memory of one pipe: S stages of p tiles, its full/empty barriers and
// its control block, rounded up to 128 bytes so every pipe starts aligned.
__host__ __device__ constexpr size_t bulkred_pipe_bytes(int p, uint32_t tile, uint32_t stages)
{
    return (size_t(stages) * size_t(p) * tile + 2 * size_t(stages) * 8 + kTmaCtlBytes + 127) / 128 * 128;
}

template <typename T, int OP> struct BulkRed;

#define CCL_BULKRED(TYPE, OPC, PTXOP)                                                                        \
    template <> struct BulkRed<TYPE, OPC> {                                                                  \
        static constexpr bool ok = true;                                                                     \
        __device__ static void issue(void *dst, uint32_t src, uint32_t bytes)                                \
        {                                                                                                    \
            asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group." PTXOP " [%0], [%1], %2;" ::"l"(dst), \
                         "r"(src), "r"(bytes)                                                                \
                         : "memory");                                                                        \
        }                                                                                                    \
    };

CCL_BULKRED(F32, OP_SUM, "add.f32")
CCL_BULKRED(F16, OP_SUM, "add.noftz.f16")
CCL_BULKRED(BF16, OP_SUM, "add.noftz.bf16")
CCL_BULKRED(I32, OP_SUM, "add.u32")
CCL_BULKRED(F16, OP_MIN, "min.f16")
CCL_BULKRED(BF16, OP_MIN, "min.bf16")
CCL_BULKRED(I32, OP_MIN, "min.s32")
CCL_BULKRED(F16, OP_MAX, "max.f16")
CCL_BULKRED(BF16, OP_MAX, "max.bf16")
CCL_BULKRED(I32, OP_MAX, "max.s32")
#undef CCL_BULKRED

template <typename T, int OP> struct BulkRed {
    static constexpr bool ok = false;
    __device__ static void issue(void *, uint32_t, uint32_t) {}
};

// dst[c] is where chunk c's reduction goes: the RS output of rank c, or, for
// an AllReduce, rank c's output at the chunk's offset.
//
// A CTA runs blockDim.x / 64 independent pipes, each on its own shared-memory
// region and its own tiles (pipe j of CTA b starts at tile b*K + j; further
// tiles come from the status block's tile counter on large messages, else by
// a stride of gridDim.x*K; the producer passes each stage's tile and batch to
// the issuer).  The issuing lane's wait for each tile's first store to land
// serialises one pipe; several pipes per CTA keep several tiles' reductions in
// flight on one SM, which is what an SM budget (one CTA per SM) needs.  A
// stage holds R ranks of a tile; above 16 ranks R < p and a tile takes
// ceil(p/R) stages, the first storing its first rank and every later one only
// reducing into the tile's destination.
template <typename T, int OP, int P>
__global__ void __launch_bounds__(kBulkThreads * kBulkMaxPipes)
    bulkred_kernel(const __grid_constant__ TmaArgs<(P > 0 ? P : kMaxRanks)> a)
{
    constexpr int S_ELEM = (Traits<T>::VEC == 8) ? 2 : 4;
    extern __shared__ __align__(128) unsigned char smem[];
    const int p = P > 0 ? P : a.p;
    const uint32_t TB = a.tile_bytes, S = a.stages, R = a.ranks_per_stage;
    const uint32_t NB = (uint32_t(p) + R - 1) / R;   // stages per tile
    const uint32_t K = blockDim.x / kBulkThreads, j = threadIdx.x / kBulkThreads;
    const uint32_t lt = threadIdx.x % kBulkThreads;
    unsigned char *in_base = smem + size_t(j) * bulkred_pipe_bytes(int(R), TB, S);   // [S][R][TB]
    uint64_t *full = reinterpret_cast<uint64_t *>(in_base + size_t(S) * R * TB);
    uint64_t *empty = full + S;
    volatile TmaCtl *ctl = reinterpret_cast<volatile TmaCtl *>(empty + S);

    if (lt == 0) {
        for (uint32_t s = 0; s < S; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), 1);
        }
        ctl->abort = 0;
        ctl->issued = 0;
        ctl->consumed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async_smem();
    }
    __syncthreads();
    grid_dependency_wait();  // launched as a dependent: no global access before this

    const uint64_t ntiles = a.tstart[p];
    const uint64_t first = uint64_t(blockIdx.x) * K + j, step = uint64_t(gridDim.x) * K;
    unsigned long long *next = reinterpret_cast<unsigned long long *>(a.status + 4);
    if (lt == 0) {
        // producer: first tile static, the rest from the counter (or a stride)
        int c = 0;
        uint32_t i = 0;
        bool stopped = false;
        for (uint64_t t = first; t < ntiles && !stopped; t = a.dynamic ? step + atomicAdd(next, 1ull) : t + step) {
            while (t >= a.tstart[c + 1]) ++c;
            const uint64_t cb = a.bound[c] * S_ELEM, ce = a.bound[c + 1] * S_ELEM;
            const uint64_t off = cb + (t - a.tstart[c]) * TB;
            const uint32_t bytes = uint32_t(ce - off < TB ? ce - off : TB);
            for (uint32_t b = 0; b < NB; ++b, ++i) {
                const uint32_t s = i % S;
                if (i >= S && !bounded_wait(a, ctl, smem_addr(&empty[s]), ((i / S) - 1) & 1u, 2u, t)) {
                    stopped = true;
                    break;
                }
                const uint32_t nb = uint32_t(p) - b * R < R ? uint32_t(p) - b * R : R;
                if (!tile_in_bounds(a, cb, ce, off, bytes, kSiteBulkred, t)) {
                    ctl->abort = 1;
                    stopped = true;
                    break;
                }
                ctl->tile_of[s] = (t << 8) | b;
                const uint32_t bar = smem_addr(&full[s]);
                mbar_arrive_expect_tx(bar, nb * bytes);
                unsigned char *slot = in_base + size_t(s) * R * TB;
                for (uint32_t k = 0; k < nb; ++k)
                    bulk_load(smem_addr(slot + size_t(k) * TB),
                              static_cast<const char *>(a.src[a.order[c][b * R + k]]) + off, bytes, bar);
                ctl->issued = i + 1;
            }
        }
        if (!stopped) {
            const uint32_t s = i % S;
            if (i < S || bounded_wait(a, ctl, smem_addr(&empty[s]), ((i / S) - 1) & 1u, 2u, i)) {
                ctl->tile_of[s] = kNoTile;
                mbar_arrive(smem_addr(&full[s]));
            }
        }
    } else if (lt == 32) {
        // issuer
        int c = 0;
        for (uint32_t i = 0;; ++i) {
            const uint32_t s = i % S;
            if (!bounded_wait(a, ctl, smem_addr(&full[s]), (i / S) & 1u, 1u, i)) break;
            const unsigned long long meta = ctl->tile_of[s];
            if (meta == kNoTile) break;
            const uint64_t t = meta >> 8;
            const uint32_t b = uint32_t(meta & 255u);
            while (t >= a.tstart[c + 1]) ++c;
            const uint64_t cb = a.bound[c] * S_ELEM, ce = a.bound[c + 1] * S_ELEM;
            const uint64_t off = cb + (t - a.tstart[c]) * TB;
            const uint32_t bytes = uint32_t(ce - off < TB ? ce - off : TB);
            if (!tile_in_bounds(a, cb, ce, off, bytes, kSiteBulkred, t)) {
                ctl->abort = 1;
                break;
            }
            char *dst = static_cast<char *>(a.dst[c]) + (off - cb);
            const uint32_t nb = uint32_t(p) - b * R < R ? uint32_t(p) - b * R : R;
            const uint32_t slot = smem_addr(in_base + size_t(s) * R * TB);
            uint32_t k0 = 0;
            if (b == 0) {
                bulk_store(dst, slot, bytes);      // the first contribution lands first
                bulk_commit();
                bulk_wait_all();
                k0 = 1;
            }
            for (uint32_t k = k0; k < nb; ++k) BulkRed<T, OP>::issue(dst, slot + k * TB, bytes);
            bulk_commit();
            bulk_wait_read(0);                     // slots read: the stage may be refilled
            mbar_arrive(smem_addr(&empty[s]));
            ctl->consumed = i + 1;
        }
        bulk_wait_all();
    }
    __syncthreads();
    if (lt == 0 && ctl->abort) {
        const uint32_t issued = ctl->issued;
        for (uint32_t q = ctl->consumed; q < issued; ++q) {
            const uint32_t bar = smem_addr(&full[q % S]);
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(bar, (q / S) & 1u))
                if (global_ns() - t0 > uint64_t(a.wait_ns)) break;
        }
    }
    if (a.dynamic && threadIdx.x == 0) {
        if (atomicAdd(a.status + 6, 1u) == gridDim.x - 1) {
            atomicExch(reinterpret_cast<unsigned long long *>(a.status + 4), 0ull);
            atomicExch(a.status + 6, 0u);
        }
    }
}

template <typename T, int OP, int P>
static cudaError_t bulkred_launch_p(const Launch &L, LaunchInfo *info)
{
    constexpr int PM = P > 0 ? P : kMaxRanks;
    constexpr int S_ELEM = (Traits<T>::VEC == 8) ? 2 : 4;
    TmaArgs<PM> a;
    uint32_t tile = 0, ranks = 0, stages = 0;
    size_t smem = 0;
    if (!bulkred_geometry(L.p, L.pipe_bytes, &tile, &ranks, &stages, &smem)) return cudaErrorInvalidValue;
    uint64_t tiles = 0;
    for (int c = 0; c <= L.p; ++c) {
        a.bound[c] = L.table->bound[c];
        a.tstart[c] = tiles;
        if (c < L.p) tiles += ((L.table->bound[c + 1] - L.table->bound[c]) * S_ELEM + tile - 1) / tile;
    }
    for (int k = 0; k < L.p; ++k) {
        a.src[k] = L.src[k];
        // AllReduce: chunk c goes to rank c's output at its own offset
        a.dst[k] = L.mode == MODE_AR ? static_cast<char *>(L.dst[k]) + L.table->bound[k] * S_ELEM : L.dst[k];
    }
    for (int c = 0; c < L.p; ++c)
        for (int k = 0; k < L.p; ++k) a.order[c][k] = L.table->order[c * L.p + k];
    a.p = L.p;
    a.scale = 1.0f;
    a.tile_bytes = tile;
    a.stages = stages;
    a.status = L.status;
    a.wait_ns = L.wait_limit_ns;
    a.stall_test = 0;
    a.ranks_per_stage = ranks;
    a.grab = 1;  // unused here
    a.buf_bytes = uint64_t(L.n) * S_ELEM;

    auto kern = bulkred_kernel<T, OP, P>;
    static std::atomic<unsigned long long> attr{0};  // devices on which the limit is raised
    {
        const cudaError_t err = allow_dynamic_smem(kern, kTmaSmemLimit, L.device, attr);
        if (err != cudaSuccess) return err;
    }
    const size_t pipe = bulkred_pipe_bytes(int(ranks), tile, stages);
    uint64_t cap;
    uint32_t pipes = 1;
    if (L.sm_budget > 0 && L.sm_budget < L.num_sms) {
        // one CTA per SM (more than half of an SM's shared memory each), with
        // as many pipes as its shared memory holds
        pipes = uint32_t(kTmaSmemLimit / pipe);
        if (pipes > uint32_t(kBulkMaxPipes)) pipes = kBulkMaxPipes;
        if (pipes < 1) pipes = 1;
        smem = pipes * pipe;
        if (smem < 120 * 1024) smem = 120 * 1024;
        cap = uint64_t(L.sm_budget);
    } else {
        smem = pipe;
        int per_sm = 0;
        cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kBulkThreads, smem);
        if (err != cudaSuccess) return err;
        cap = uint64_t(L.num_sms) * (per_sm > 0 ? per_sm : 1);
    }
    const uint64_t ctas = (tiles + pipes - 1) / pipes;
    const int grid = int(ctas < cap ? (ctas ? ctas : 1) : cap);
    // the tile counter (as in the TMA variant): p=8 5236 -> 5565 GB/s, p=16
    // 5023 -> 5501, p=64 5118 -> 5570 on every SM; 4 % slower at p=2
    a.dynamic = L.tile_counter && tiles >= 16ull * uint64_t(grid) * pipes ? 1 : 0;
    const int block = int(pipes) * kBulkThreads;
    cudaError_t err = launch_dependent(kern, unsigned(grid), unsigned(block), smem, L.stream, a);
    if (err != cudaSuccess) return err;
    if (info) {
        info->kernel = MODE_AR == L.mode ? "allreduce_tma_bulkred" : "reduce_scatter_tma_bulkred";
        info->grid = grid;
        info->block = block;
        info->smem = smem;
        info->kernels = 1;
        info->counter = a.dynamic;
    }
    return cudaGetLastError();
}

template <typename T, int OP>
static cudaError_t bulkred_launch_op(const Launch &L, LaunchInfo *info)
{
    if constexpr (!BulkRed<T, OP>::ok) {
        return cudaErrorInvalidValue;
    } else {
        switch (L.p) {
        case 2: return bulkred_launch_p<T, OP, 2>(L, info);
        case 4: return bulkred_launch_p<T, OP, 4>(L, info);
        case 8: return bulkred_launch_p<T, OP, 8>(L, info);
        case 16: return bulkred_launch_p<T, OP, 16>(L, info);
        default: return bulkred_launch_p<T, OP, 0>(L, info);
        }
    }
}

template <typename T>
static cudaError_t launch_bulkred(const Launch &L, LaunchInfo *info)
{
    switch (L.op) {
    case OP_SUM: return bulkred_launch_op<T, OP_SUM>(L, info);
    case OP_MIN: return bulkred_launch_op<T, OP_MIN>(L, info);
    case OP_MAX: return bulkred_launch_op<T, OP_MAX>(L, info);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ccl
