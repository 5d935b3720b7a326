// TMA variant of the multi-source reduce: bulk copies into shared-memory
// stages, a register fold in the chunk's exact order, bulk fan-out stores.
//
// T-CCL, sections "TMA Transfer Engine" and "Pipelined Copy and Reduction":
// one elected thread issues bulk transfers that proceed asynchronously in the
// TMA unit; a D-stage shared-memory pipeline keeps some stages loading while
// others are being stored, each stage waiting for its load to complete before
// its store is issued, and for its previous store before it is reloaded.
// Here one CTA per SM (persistent; or k CTAs under an SM budget) walks the
// tiles -- on large messages taking them from a device-wide counter, a few
// at a time, until none are left; on small ones by a static stride.  A tile
// is T bytes of one chunk, taken from every rank:
//
//   producer (warp 0, one lane):  wait stage free -> expect p*T bytes ->
//                                 p x cp.async.bulk global->shared (rank k of
//                                 the chunk's order into slot k)
//   consumers (8 warps, each on   wait stage full and its out tile free ->
//   its own):                     fold slots 0..p-1 in fp32 -> packed result
//                                 into the stage's out tile -> release the
//                                 input slots, mark its part of the out tile
//   store warp (one lane):        wait until all 8 parts are in -> bulk
//                                 stores (every rank for AllReduce, the owner
//                                 for ReduceScatter) -> free the out tile once
//                                 they have read it
//
// No barrier joins the consumer warps: each waits on the stage's mbarriers
// itself, and the store warp hands the out tile back through its own
// mbarrier.  Measured on GB300 against one thread per CTA waiting and
// issuing behind a 256-thread named barrier (AllReduce, GB/s per SM):
// p=8 on 8/16/32 SMs 97 -> 105/104/103, p=4 on 16 SMs 70 -> 82, p=5 fp32
// +27-30 %, p=3 +11 %, p=2 +5-8 %, the whole GPU unchanged; the wide kernel
// in the same form against its barrier form: p=40 and 64 on 8-32 SMs 70 ->
// 93, on 76 SMs +25 %.
//
// Order, rounding and therefore every bit equal the ld/st kernel's.  Every
// wait is bounded by %globaltimer: on expiry the kernel records where it gave
// up in the communicator's status block, stops issuing work, waits (bounded)
// for its own copies in flight and returns; ccl_comm_check() reports
// CCL_ERR_TIMEOUT.  A tile may be shorter than T at the end of a chunk (always
// a multiple of 16 bytes: the host only selects this variant when every chunk
// boundary and pointer is 16-byte aligned).  The counter lives in the
// communicator's status block and the last CTA of a launch returns it to
// zero, so launches on one status block must be ordered (one stream, or
// synchronised), as every collective on one communicator already is.  From
// 14 ranks the wide kernel further down takes over (ranks through the stages
// eight at a time, 8 KB per copy).
#pragma once

#include "device.cuh"

namespace ccl {

constexpr int kTmaConsumerWarps = 8;
constexpr int kTmaConsumers = 32 * kTmaConsumerWarps;

template <int PM>
struct TmaArgs {
    const void *src[PM];
    void *dst[PM];
    uint64_t bound[PM + 1];     // chunk c = elements [bound[c], bound[c+1])
    uint64_t tstart[PM + 1];    // first tile of chunk c; tstart[p] = number of tiles
    uint8_t order[PM][PM];      // order[c][k]: k-th rank folded into chunk c
    int p;
    float scale;                // avg: fl32(1/p)
    uint32_t tile_bytes;        // T: bytes per rank per stage
    uint32_t stages;            // S
    unsigned *status;           // status block: [0] code, [1] block, [2] tile, [3] role
    long long wait_ns;          // bound on any single wait
    int stall_test;             // 1: the producer withholds its second tile (timeout test); 2: see tile_in_bounds
    int dynamic;                // 1: tiles beyond each CTA's first grab come from the tile counter
    uint32_t ranks_per_stage;   // wide kernel: R ranks of a tile per stage
    uint32_t grab;              // wide kernel: tiles per visit to the tile counter
    uint64_t buf_bytes;         // bytes of every rank buffer (checked build: the extent each copy is tested against)
};

// ---------------------------------------------------------------------------
// PTX wrappers: mbarrier, bulk copies, proxy fence, named barrier, timer.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void bulk_load(uint32_t dst_smem, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst_smem),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void bulk_store(void *dst, uint32_t src_smem, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src_smem), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Wait until at most `pending` of this thread's bulk groups still read shared memory.
__device__ __forceinline__ void bulk_wait_read(uint32_t pending)
{
    switch (pending) {
    case 0: asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.bulk.wait_group.read 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.bulk.wait_group.read 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.bulk.wait_group.read 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.bulk.wait_group.read 6;" ::: "memory"); break;
    default: asm volatile("cp.async.bulk.wait_group.read 7;" ::: "memory"); break;
    }
}

__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ uint4 lds_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts_v4(uint32_t addr, const uint4 &v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Shared control words beside the barriers.
struct TmaCtl {
    int abort;          // set by whichever role gives up first
    int go;             // consumer leader -> consumers: this tile may proceed
    uint32_t issued;    // tiles whose loads the producer issued
    uint32_t consumed;  // tiles the consumers finished reading
    unsigned long long tile_of[kTmaMaxStages];  // the tile loaded into each stage (kNoTile: no more work)
};
constexpr unsigned long long kNoTile = ~0ull;

// Tiles the narrow kernel takes per visit to the tile counter under an SM
// budget (one on the whole GPU).  Measured on GB300 (p=8 bf16, 256 MiB per
// rank, every SM): a static round-robin split reached 6.56 TB/s, one tile per
// visit 7.03, four 6.95 -- and four is 3-5 % faster than one under SM budgets
// (p=16 at 16 SMs: 1258 vs 1140 GB/s).
constexpr unsigned kTmaGrab = 4;

// Control words of the narrow kernel (tma_reduce_kernel).
struct TmaPipeCtl {
    int abort;          // set by whichever role gives up first
    uint32_t issued;    // stages whose loads the producer issued
    unsigned long long tile_of[kTmaMaxStages];  // producer -> consumers: the tile in each stage (kNoTile: done)
    unsigned long long out_of[kTmaMaxStages];   // consumers -> store warp: the tile in each out tile
    unsigned long long unused_grab;             // wide kernel: the grab asked for ahead and never taken
};

// Checked build: a tile's copies, `bytes` at byte offset `off` of chunk
// [cb, ce), lie inside the chunk and inside every rank buffer.  With
// stall_test == 2 the producer's check of its second stage reports a
// violation, so that a test can see the record (the copies are not made).
template <int PM>
__device__ __forceinline__ bool tile_in_bounds(const TmaArgs<PM> &a, uint64_t cb, uint64_t ce, uint64_t off,
                                               uint32_t bytes, unsigned site, uint64_t t, bool forced = false)
{
    return in_bounds(!forced && bytes > 0 && off >= cb && off + bytes <= ce && ce <= a.buf_bytes, a.status, site, t);
}

// Bounded wait on an mbarrier phase.  Returns false if the wait gave up
// (timeout, recorded in the status block) or another role aborted.
template <int PM, typename Ctl>
__device__ __forceinline__ bool bounded_wait(const TmaArgs<PM> &a, volatile Ctl *ctl, uint32_t bar,
                                             uint32_t parity, unsigned code, uint64_t tile)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (ctl->abort) return false;
        if (global_ns() - t0 > uint64_t(a.wait_ns)) {
            if (atomicCAS(&a.status[0], 0u, code) == 0u) {
                a.status[1] = blockIdx.x;
                a.status[2] = unsigned(tile);
                a.status[3] = threadIdx.x;
            }
            ctl->abort = 1;
            return false;
        }
    }
    return true;
}

constexpr int kTmaPipeThreads = kTmaConsumers + 64;   // producer warp, store warp, 8 consumer warps

template <typename T, int OP, int P, int MODE>
__global__ void __launch_bounds__(kTmaPipeThreads, 1)
    tma_reduce_kernel(const __grid_constant__ TmaArgs<(P > 0 ? P : kMaxRanks)> a)
{
    using Tr = Traits<T>;
    constexpr int VEC = Tr::VEC;
    constexpr int S_ELEM = (VEC == 8) ? 2 : 4;
    extern __shared__ __align__(128) unsigned char smem[];

    const int p = P > 0 ? P : a.p;
    const uint32_t TB = a.tile_bytes, S = a.stages;
    unsigned char *in_base = smem;                                   // [S][p][TB]
    unsigned char *out_base = smem + size_t(S) * p * TB;             // [S][TB]
    uint64_t *full = reinterpret_cast<uint64_t *>(out_base + size_t(S) * TB);
    uint64_t *empty = full + S;       // the 8 consumer warps have read the stage's input slots
    uint64_t *folded = empty + S;     // the 8 consumer warps have written their parts of out tile s
    uint64_t *out_free = folded + S;  // the stores of out tile s have read it
    volatile TmaPipeCtl *ctl = reinterpret_cast<volatile TmaPipeCtl *>(out_free + S);

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < S; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), kTmaConsumerWarps);
            mbar_init(smem_addr(&folded[s]), kTmaConsumerWarps);
            mbar_init(smem_addr(&out_free[s]), 1);
        }
        ctl->abort = 0;
        ctl->issued = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async_smem();
    }
    __syncthreads();
    // Launched as a dependent: the set-up above overlaps the previous
    // kernel's tail; no global memory is touched before this wait.
    grid_dependency_wait();

    const uint64_t ntiles = a.tstart[p];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            // Large messages (a.dynamic): tiles go out a.grab at a time,
            // each CTA's first grab statically (tiles blockIdx.x*G ...), the
            // rest from a device-wide counter (the status block's words 4-5),
            // so SMs that run faster take more.  Small messages: tile b, then
            // b + gridDim.x, ... with no counter, which keeps their latency.
            unsigned long long *next = reinterpret_cast<unsigned long long *>(a.status + 4);
            const unsigned long long G = a.dynamic ? a.grab : 1;
            int c = 0;
            unsigned long long t = blockIdx.x * G, left = G;   // the current grab: tiles t, t+1, ...
            for (uint32_t i = 0;; ++i) {
                const uint32_t s = i % S;
                if (i >= S && !bounded_wait(a, ctl, smem_addr(&empty[s]), ((i / S) - 1) & 1u, 2u, i)) break;
                if (a.stall_test == 1 && i == 1) break;  // withhold this stage: its consumers must time out
                if (left == 0) {
                    t = a.dynamic ? gridDim.x * G + atomicAdd(next, G) : t + gridDim.x;
                    left = G;
                } else if (i > 0) {
                    ++t;
                }
                --left;
                const uint32_t bar = smem_addr(&full[s]);
                if (t >= ntiles) {
                    ctl->tile_of[s] = kNoTile;
                    mbar_arrive(bar);                // no bytes: the consumers wake and stop
                    break;
                }
                ctl->tile_of[s] = t;
                while (t >= a.tstart[c + 1]) ++c;
                const uint64_t cb = a.bound[c] * S_ELEM, ce = a.bound[c + 1] * S_ELEM;
                const uint64_t off = cb + (t - a.tstart[c]) * TB;
                const uint32_t bytes = uint32_t(ce - off < TB ? ce - off : TB);
                if (!tile_in_bounds(a, cb, ce, off, bytes, kSiteTmaLoad, t, a.stall_test == 2 && i == 1)) {
                    ctl->abort = 1;
                    break;
                }
                mbar_arrive_expect_tx(bar, uint32_t(p) * bytes);
                unsigned char *slot = in_base + size_t(s) * p * TB;
                for (int k = 0; k < p; ++k)
                    bulk_load(smem_addr(slot + size_t(k) * TB),
                              static_cast<const char *>(a.src[a.order[c][k]]) + off, bytes, bar);
                ctl->issued = i + 1;
            }
        }
    } else if (warp == 1) {
        // ------------------------------ store warp ----------------------------
        if (lane == 0) {
            int c = 0;
            for (uint32_t i = 0;; ++i) {
                const uint32_t s = i % S;
                if (!bounded_wait(a, ctl, smem_addr(&folded[s]), (i / S) & 1u, 3u, i)) break;
                const unsigned long long t = ctl->out_of[s];
                if (t == kNoTile) break;
                while (t >= a.tstart[c + 1]) ++c;
                const uint64_t cb = a.bound[c] * S_ELEM, ce = a.bound[c + 1] * S_ELEM;
                const uint64_t off = cb + (t - a.tstart[c]) * TB;
                const uint32_t bytes = uint32_t(ce - off < TB ? ce - off : TB);
                if (!tile_in_bounds(a, cb, ce, off, bytes, kSiteTmaStore, t)) {
                    ctl->abort = 1;
                    break;
                }
                const uint32_t out_s = smem_addr(out_base + size_t(s) * TB);
                if constexpr (MODE == MODE_AR) {
                    for (int k = 0; k < p; ++k) bulk_store(static_cast<char *>(a.dst[k]) + off, out_s, bytes);
                } else {
                    bulk_store(static_cast<char *>(a.dst[c]) + (off - cb), out_s, bytes);
                }
                bulk_commit();
                // the stores of iterations up to i-(S-1) have read their out tiles
                bulk_wait_read(S - 1);
                if (i + 1 >= S) mbar_arrive(smem_addr(&out_free[(i + 1 - S) % S]));
            }
            bulk_wait_all();
        }
    } else {
        // ------------------------------ consumer warps ------------------------
        // Every lane waits on the stage's barriers itself; the vote makes the
        // warp leave together if any lane's wait gave up (so the __syncwarp
        // below is always reached by all of its lanes).
        const int cw = warp - 2;
        const int tid = threadIdx.x - 64;
        int c = 0;
        for (uint32_t i = 0;; ++i) {
            const uint32_t s = i % S;
            if (!__all_sync(0xffffffffu, bounded_wait(a, ctl, smem_addr(&full[s]), (i / S) & 1u, 1u, i))) break;
            const unsigned long long t = ctl->tile_of[s];
            // Out tile s must be free before this warp touches it or its
            // barrier -- also on the last visit: until the store warp has
            // read out_of[s] of tile i-S, a fast warp must neither overwrite
            // it nor arrive on folded[s] within that tile's phase.
            if (i >= S &&
                !__all_sync(0xffffffffu, bounded_wait(a, ctl, smem_addr(&out_free[s]), ((i / S) - 1) & 1u, 4u, i)))
                break;
            if (t == kNoTile) {
                // no more work: tell the store warp through the out tile's barrier
                if (cw == 0 && lane == 0) ctl->out_of[s] = kNoTile;
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&folded[s]));
                break;
            }
            while (t >= a.tstart[c + 1]) ++c;
            const uint64_t cb = a.bound[c] * S_ELEM, ce = a.bound[c + 1] * S_ELEM;
            const uint64_t off = cb + (t - a.tstart[c]) * TB;
            const uint32_t bytes = uint32_t(ce - off < TB ? ce - off : TB);
            const uint32_t in_s = smem_addr(in_base + size_t(s) * p * TB);
            const uint32_t out_s = smem_addr(out_base + size_t(s) * TB);
            for (uint32_t g = tid; g < bytes / 16; g += kTmaConsumers) {
                GroupFold<T, OP> acc;
                if constexpr (P > 0) {
                    uint4 r[P];
#pragma unroll
                    for (int k = 0; k < P; ++k) r[k] = lds_v4(in_s + k * TB + g * 16);
                    acc.first(r[0], a.scale);
#pragma unroll
                    for (int k = 1; k < P; ++k) acc.fold(r[k], a.scale);
                } else {
                    acc.first(lds_v4(in_s + g * 16), a.scale);
                    for (int k = 1; k < p; ++k) acc.fold(lds_v4(in_s + k * TB + g * 16), a.scale);
                }
                sts_v4(out_s + g * 16, acc.finish(p));
            }
            fence_proxy_async_smem();                          // out tile visible to the bulk stores
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_addr(&empty[s]));             // input slots of stage s are free
                if (cw == 0) ctl->out_of[s] = t;
                mbar_arrive(smem_addr(&folded[s]));            // this warp's part of out tile s is written
            }
        }
    }
    __syncthreads();
    // After an abort, wait (bounded) for loads still in flight into shared
    // memory -- at most the last S stages issued -- before the CTA gives its
    // shared memory back.
    if (threadIdx.x == 0 && ctl->abort) {
        const uint32_t issued = ctl->issued;
        for (uint32_t j = issued > S ? issued - S : 0; j < issued; ++j) {
            const uint32_t bar = smem_addr(&full[j % S]);
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(bar, (j / S) & 1u))
                if (global_ns() - t0 > uint64_t(a.wait_ns)) break;
        }
    }
    // The last CTA to finish takes no more tiles than any other; it returns
    // the tile counter to zero for the next launch on this status block.
    if (a.dynamic && threadIdx.x == 0) {
        if (atomicAdd(a.status + 6, 1u) == gridDim.x - 1) {
            atomicExch(reinterpret_cast<unsigned long long *>(a.status + 4), 0ull);
            atomicExch(a.status + 6, 0u);
        }
    }
}

// ---------------------------------------------------------------------------
// Wide variant: a tile's p ranks pass through the stages R at a time (8
// ranks of 8 KB, or 4 of 16 KB on small grids).  The
// producer loads ranks order[c][b*R ...] of tile t into a stage (one stage
// per batch b = 0 .. B-1, B = ceil(p/R)); each consumer thread keeps the fp32
// partial of its 16-byte groups of the tile in registers across the B
// batches, folding in the chunk's order exactly as the narrow kernel does,
// and after the last batch writes the tile to one of kTmaWideOut output
// tiles, from which the store warp issues the bulk fan-out stores.  The roles
// and their mbarriers are the narrow kernel's (producer warp, store warp,
// 8 consumer warps each waiting for itself), except that the output tiles
// are not tied to the stages: out tile k % kTmaWideOut holds the CTA's k-th
// finished tile.  Waits, abort, drain and the tile counter work as in the
// narrow kernel, with one tile per visit (a tile is B stages of work), or
// kTmaWideGrab on small grids.
// ---------------------------------------------------------------------------

constexpr unsigned kTmaWideGrab = 4;  // tiles per counter visit on small grids

// RM: the most ranks a stage holds (8, with tiles of at most 8 KB, or 4 with
// at most 16 KB: 64 KB per stage); each consumer thread folds the tile's
// 16-byte groups g = tid, tid + 256, ... -- at most G of them.  One
// instantiation per shape: the 8-rank shape compiled with room for 16 KB
// tiles ran 7 % slower on 16 SMs (99 registers against 79 and 80).
template <typename T, int OP, int MODE, int RM>
__global__ void __launch_bounds__(kTmaPipeThreads, 1)
    tma_wide_kernel(const __grid_constant__ TmaArgs<kMaxRanks> a)
{
    constexpr int G = RM <= 4 ? 4 : 2;                               // 16-byte groups per consumer thread
    using Tr = Traits<T>;
    constexpr int VEC = Tr::VEC;
    constexpr int S_ELEM = (VEC == 8) ? 2 : 4;
    constexpr uint32_t O = kTmaWideOut;
    extern __shared__ __align__(128) unsigned char smem[];

    const int p = a.p;
    const uint32_t TB = a.tile_bytes, S = a.stages, R = a.ranks_per_stage;
    const uint32_t B = (uint32_t(p) + R - 1) / R;                    // stages per tile
    unsigned char *in_base = smem;                                   // [S][R][TB]
    unsigned char *out_base = smem + size_t(S) * R * TB;             // [O][TB]
    uint64_t *full = reinterpret_cast<uint64_t *>(out_base + size_t(O) * TB);
    uint64_t *empty = full + S;        // the 8 consumer warps have read the stage's input slots
    uint64_t *folded = empty + S;      // the 8 consumer warps have written their parts of out tile o
    uint64_t *out_free = folded + O;   // the stores of out tile o have read it
    volatile TmaPipeCtl *ctl = reinterpret_cast<volatile TmaPipeCtl *>(out_free + O);

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < S; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), kTmaConsumerWarps);
        }
        for (uint32_t o = 0; o < O; ++o) {
            mbar_init(smem_addr(&folded[o]), kTmaConsumerWarps);
            mbar_init(smem_addr(&out_free[o]), 1);
        }
        ctl->abort = 0;
        ctl->issued = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async_smem();
    }
    __syncthreads();
    grid_dependency_wait();  // launched as a dependent: no global access before this

    const uint64_t ntiles = a.tstart[p];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            // Large messages (a.dynamic): each CTA's first grab of G tiles is
            // static (tiles blockIdx.x*G ...), the rest come from the tile
            // counter.  With G > 1 (small grids) the next grab is asked for
            // as the current one starts, so that the counter's round trip
            // overlaps this grab's stages.  Small messages: tile b, then
            // b + gridDim.x, ...
            unsigned long long *next = reinterpret_cast<unsigned long long *>(a.status + 4);
            int c = 0;
            uint32_t i = 0;
            bool stopped = false;
            const unsigned long long G = a.dynamic ? a.grab : 1ull;
            const bool early = G > 1;
            unsigned long long t = blockIdx.x * G, left = G;
            unsigned long long ahead = early ? atomicAdd(next, G) : 0ull;
            while (t < ntiles && !stopped) {
                while (t >= a.tstart[c + 1]) ++c;
                const uint64_t cb = a.bound[c] * S_ELEM, ce = a.bound[c + 1] * S_ELEM;
                const uint64_t off = cb + (t - a.tstart[c]) * TB;
                const uint32_t bytes = uint32_t(ce - off < TB ? ce - off : TB);
                for (uint32_t b = 0; b < B; ++b, ++i) {
                    const uint32_t s = i % S;
                    if (i >= S && !bounded_wait(a, ctl, smem_addr(&empty[s]), ((i / S) - 1) & 1u, 2u, i)) {
                        stopped = true;
                        break;
                    }
                    if (a.stall_test == 1 && i == 1) {  // withhold this stage: its consumers must time out
                        stopped = true;
                        break;
                    }
                    const uint32_t nb = uint32_t(p) - b * R < R ? uint32_t(p) - b * R : R;
                    if (!tile_in_bounds(a, cb, ce, off, bytes, kSiteTmaLoad, t, a.stall_test == 2 && i == 1)) {
                        ctl->abort = 1;
                        stopped = true;
                        break;
                    }
                    ctl->tile_of[s] = (t << 8) | b;
                    const uint32_t bar = smem_addr(&full[s]);
                    mbar_arrive_expect_tx(bar, nb * bytes);
                    unsigned char *slot = in_base + size_t(s) * R * TB;
                    for (uint32_t j = 0; j < nb; ++j)
                        bulk_load(smem_addr(slot + size_t(j) * TB),
                                  static_cast<const char *>(a.src[a.order[c][b * R + j]]) + off, bytes, bar);
                    ctl->issued = i + 1;
                }
                if (--left > 0) {
                    ++t;
                } else {
                    if (!a.dynamic) {
                        t += gridDim.x;
                    } else if (early) {
                        t = gridDim.x * G + ahead;
                        ahead = atomicAdd(next, G);
                    } else {
                        t = gridDim.x + atomicAdd(next, 1ull);
                    }
                    left = G;
                }
            }
            // The grab asked for ahead is never taken: storing its value waits
            // for that atomic to return, so that it has landed before this
            // CTA counts itself done and the last CTA resets the counter.
            if (early) ctl->unused_grab = ahead;
            if (!stopped) {
                // no more work: a stage with no bytes wakes the consumers
                const uint32_t s = i % S;
                if (i < S || bounded_wait(a, ctl, smem_addr(&empty[s]), ((i / S) - 1) & 1u, 2u, i)) {
                    ctl->tile_of[s] = kNoTile;
                    mbar_arrive(smem_addr(&full[s]));
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------ store warp ----------------------------
        if (lane == 0) {
            int c = 0;
            for (uint32_t k = 0;; ++k) {
                const uint32_t o = k % O;
                if (!bounded_wait(a, ctl, smem_addr(&folded[o]), (k / O) & 1u, 3u, k)) break;
                const unsigned long long t = ctl->out_of[o];
                if (t == kNoTile) break;
                while (t >= a.tstart[c + 1]) ++c;
                const uint64_t cb = a.bound[c] * S_ELEM, ce = a.bound[c + 1] * S_ELEM;
                const uint64_t off = cb + (t - a.tstart[c]) * TB;
                const uint32_t bytes = uint32_t(ce - off < TB ? ce - off : TB);
                if (!tile_in_bounds(a, cb, ce, off, bytes, kSiteTmaStore, t)) {
                    ctl->abort = 1;
                    break;
                }
                const uint32_t out_s = smem_addr(out_base + size_t(o) * TB);
                if constexpr (MODE == MODE_AR) {
                    for (int r = 0; r < p; ++r) bulk_store(static_cast<char *>(a.dst[r]) + off, out_s, bytes);
                } else {
                    bulk_store(static_cast<char *>(a.dst[c]) + (off - cb), out_s, bytes);
                }
                bulk_commit();
                // the stores of tiles up to k-(O-1) have read their out tiles
                bulk_wait_read(O - 1);
                if (k + 1 >= O) mbar_arrive(smem_addr(&out_free[(k + 1 - O) % O]));
            }
            bulk_wait_all();
        }
    } else {
        // ------------------------------ consumer warps ------------------------
        // As in the narrow kernel: every lane waits itself, and a vote makes
        // the warp leave together if any lane's wait gave up.
        const int cw = warp - 2;
        const int tid = threadIdx.x - 64;
        GroupFold<T, OP> acc[G];
        int c = 0;
        uint32_t k = 0;  // tiles finished by this CTA: the next goes to out tile k % O
        for (uint32_t i = 0;; ++i) {
            const uint32_t s = i % S;
            if (!__all_sync(0xffffffffu, bounded_wait(a, ctl, smem_addr(&full[s]), (i / S) & 1u, 1u, i))) break;
            const unsigned long long meta = ctl->tile_of[s];
            const uint32_t o = k % O;
            if (meta == kNoTile) {
                // no more work: once out tile o is free (its last tile's id
                // read), tell the store warp through its barrier
                if (k >= O &&
                    !__all_sync(0xffffffffu, bounded_wait(a, ctl, smem_addr(&out_free[o]), ((k / O) - 1) & 1u, 4u, k)))
                    break;
                if (cw == 0 && lane == 0) ctl->out_of[o] = kNoTile;
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&folded[o]));
                break;
            }
            const uint64_t t = meta >> 8;
            const uint32_t b = uint32_t(meta & 255u);
            while (t >= a.tstart[c + 1]) ++c;
            const uint64_t cb = a.bound[c] * S_ELEM, ce = a.bound[c + 1] * S_ELEM;
            const uint64_t off = cb + (t - a.tstart[c]) * TB;
            const uint32_t bytes = uint32_t(ce - off < TB ? ce - off : TB);
            const uint32_t nb = uint32_t(p) - b * R < R ? uint32_t(p) - b * R : R;
            const uint32_t in_s = smem_addr(in_base + size_t(s) * R * TB);
#pragma unroll
            for (int q = 0; q < G; ++q) {
                const uint32_t g = uint32_t(tid) + uint32_t(q) * kTmaConsumers;
                if (g * 16 >= bytes) continue;
                // the stage's loads in flight before their folds
                uint4 r[RM];
#pragma unroll
                for (uint32_t j = 0; j < uint32_t(RM); ++j)
                    if (j < nb) r[j] = lds_v4(in_s + j * TB + g * 16);
#pragma unroll
                for (uint32_t j = 0; j < uint32_t(RM); ++j) {
                    if (j < nb) {
                        if (b == 0 && j == 0) acc[q].first(r[j], a.scale);
                        else acc[q].fold(r[j], a.scale);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&empty[s]));  // this stage's input slots are free
            if (b + 1 == B) {
                // the tile is complete: write it to out tile o once the stores
                // of tile k - O have read it
                if (k >= O &&
                    !__all_sync(0xffffffffu, bounded_wait(a, ctl, smem_addr(&out_free[o]), ((k / O) - 1) & 1u, 4u, k)))
                    break;
                const uint32_t out_s = smem_addr(out_base + size_t(o) * TB);
#pragma unroll
                for (int q = 0; q < G; ++q) {
                    const uint32_t g = uint32_t(tid) + uint32_t(q) * kTmaConsumers;
                    if (g * 16 >= bytes) continue;
                    sts_v4(out_s + g * 16, acc[q].finish(p));
                }
                fence_proxy_async_smem();                      // out tile visible to the bulk stores
                __syncwarp();
                if (lane == 0) {
                    if (cw == 0) ctl->out_of[o] = t;
                    mbar_arrive(smem_addr(&folded[o]));        // this warp's part of out tile o is written
                }
                ++k;
            }
        }
    }
    __syncthreads();
    // After an abort, wait (bounded) for loads still in flight into shared
    // memory -- at most the last S stages issued -- before the CTA gives its
    // shared memory back.
    if (threadIdx.x == 0 && ctl->abort) {
        const uint32_t issued = ctl->issued;
        for (uint32_t j = issued > S ? issued - S : 0; j < issued; ++j) {
            const uint32_t bar = smem_addr(&full[j % S]);
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(bar, (j / S) & 1u))
                if (global_ns() - t0 > uint64_t(a.wait_ns)) break;
        }
    }
    // The last CTA to finish returns the tile counter to zero; the fence
    // orders this CTA's counter atomics before its count.
    if (a.dynamic && threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(a.status + 6, 1u) == gridDim.x - 1) {
            __threadfence();
            atomicExch(reinterpret_cast<unsigned long long *>(a.status + 4), 0ull);
            atomicExch(a.status + 6, 0u);
        }
    }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------

template <typename T, int OP, int P, int MODE>
static cudaError_t tma_launch_p(const Launch &L, LaunchInfo *info)
{
    constexpr int PM = P > 0 ? P : kMaxRanks;
    constexpr int S_ELEM = (Traits<T>::VEC == 8) ? 2 : 4;
    TmaArgs<PM> a;
    uint32_t tile = 0, stages = 0;
    size_t smem = 0;
    if (!tma_geometry(L.p, L.pipe_bytes, L.sm_budget, &tile, &stages, &smem)) return cudaErrorInvalidValue;
    static_assert(sizeof(TmaCtl) <= kTmaNarrowCtlBytes && sizeof(TmaPipeCtl) <= kTmaNarrowCtlBytes, "control block");
    for (int k = 0; k < L.p; ++k) {
        a.src[k] = L.src[k];
        a.dst[k] = L.dst[k];
    }
    uint64_t tiles = 0;
    for (int c = 0; c <= L.p; ++c) {
        a.bound[c] = L.table->bound[c];
        a.tstart[c] = tiles;
        if (c < L.p) {
            const uint64_t bytes = (L.table->bound[c + 1] - L.table->bound[c]) * S_ELEM;
            tiles += (bytes + tile - 1) / tile;
        }
    }
    for (int c = 0; c < L.p; ++c)
        for (int k = 0; k < L.p; ++k) a.order[c][k] = L.table->order[c * L.p + k];
    a.p = L.p;
    a.scale = 1.0f / float(L.p);
    a.tile_bytes = tile;
    a.stages = stages;
    a.status = L.status;
    a.wait_ns = L.wait_limit_ns;
    a.stall_test = L.stall_test;
    a.buf_bytes = uint64_t(L.n) * S_ELEM;
    a.ranks_per_stage = 0;  // wide kernel only

    void (*kern)(const TmaArgs<PM>) = tma_reduce_kernel<T, OP, P, MODE>;
    const int threads = kTmaPipeThreads;
    static std::atomic<unsigned long long> attr{0};  // devices on which the limit is raised
    {
        const cudaError_t err = allow_dynamic_smem(kern, kTmaSmemLimit, L.device, attr);
        if (err != cudaSuccess) return err;
    }
    uint64_t cap = uint64_t(L.num_sms);
    if (L.sm_budget > 0 && L.sm_budget < L.num_sms) cap = uint64_t(L.sm_budget);
    const int grid = int(tiles < cap ? (tiles ? tiles : 1) : cap);
    // the tile counter pays off once every CTA has many grabs to balance
    // kTmaGrab tiles per visit to the tile counter under an SM budget, one on
    // the whole GPU.  Measured on GB300 (AllReduce, bf16, 256 MiB per rank):
    // whole GPU p=2/4/8/12 6855/6936/6958/6843 -> 6955/7012/7030/6968 GB/s
    // with one; on 76 SMs one per visit lost 3-16 % at p <= 8.  The counter
    // takes over from 16 grabs per CTA (whole GPU, 32-64 MiB per rank: +8 to
    // +11 % against the static split, which smaller messages keep).
    a.grab = (L.sm_budget > 0 && L.sm_budget < L.num_sms) ? kTmaGrab : 1;
    a.dynamic = L.tile_counter && tiles >= 16ull * a.grab * uint64_t(grid) ? 1 : 0;
    cudaError_t err = launch_dependent(kern, unsigned(grid), unsigned(threads), smem, L.stream, a);
    if (err != cudaSuccess) return err;
    if (info) {
        info->kernel = MODE == MODE_AR ? "allreduce_tma" : "reduce_scatter_tma";
        info->grid = grid;
        info->block = threads;
        info->smem = smem;
        info->kernels = 1;
        info->counter = a.dynamic;
    }
    return cudaGetLastError();
}

template <typename T, int OP, int MODE>
static cudaError_t tma_wide_launch(const Launch &L, LaunchInfo *info)
{
    constexpr int S_ELEM = (Traits<T>::VEC == 8) ? 2 : 4;
    TmaArgs<kMaxRanks> a;
    uint32_t tile = 0, ranks = 0, stages = 0;
    size_t smem = 0;
    if (!tma_wide_geometry(L.p, L.pipe_bytes, L.sm_budget, &tile, &ranks, &stages, &smem)) return cudaErrorInvalidValue;
    for (int k = 0; k < L.p; ++k) {
        a.src[k] = L.src[k];
        a.dst[k] = L.dst[k];
    }
    uint64_t tiles = 0;
    for (int c = 0; c <= L.p; ++c) {
        a.bound[c] = L.table->bound[c];
        a.tstart[c] = tiles;
        if (c < L.p) tiles += ((L.table->bound[c + 1] - L.table->bound[c]) * S_ELEM + tile - 1) / tile;
    }
    for (int c = 0; c < L.p; ++c)
        for (int k = 0; k < L.p; ++k) a.order[c][k] = L.table->order[c * L.p + k];
    a.p = L.p;
    a.scale = 1.0f / float(L.p);
    a.tile_bytes = tile;
    a.stages = stages;
    a.ranks_per_stage = ranks;
    a.status = L.status;
    a.wait_ns = L.wait_limit_ns;
    a.stall_test = L.stall_test;
    a.buf_bytes = uint64_t(L.n) * S_ELEM;

    // devices on which each instantiation's shared-memory limit is raised
    static std::atomic<unsigned long long> attr4{0}, attr8{0};
    const bool four = ranks <= 4;
    void (*kern)(const TmaArgs<kMaxRanks>) = four ? tma_wide_kernel<T, OP, MODE, 4> : tma_wide_kernel<T, OP, MODE, 8>;
    {
        const cudaError_t err = allow_dynamic_smem(kern, kTmaSmemLimit, L.device, four ? attr4 : attr8);
        if (err != cudaSuccess) return err;
    }
    uint64_t cap = uint64_t(L.num_sms);
    if (L.sm_budget > 0 && L.sm_budget < L.num_sms) cap = uint64_t(L.sm_budget);
    const int grid = int(tiles < cap ? (tiles ? tiles : 1) : cap);
    // Grabs of kTmaWideGrab tiles on grids of at most kTmaSmallGrid CTAs,
    // one tile elsewhere.  Measured on GB300 (AllReduce, bf16, GB/s per SM):
    // p=16 on 8/16/32 SMs 89.0/89.8/89.7 -> 93.8/93.7/92.9 with grabs of four
    // asked for ahead, p=64 +2 %; on the whole GPU the coarser grabs cost 2 %.
    a.grab = (L.sm_budget > 0 && L.sm_budget <= kTmaSmallGrid) ? kTmaWideGrab : 1;
    // the counter pays off once every CTA has many grabs (a tile here is B stages of work)
    a.dynamic = L.tile_counter && tiles >= 16ull * a.grab * uint64_t(grid) ? 1 : 0;
    cudaError_t err = launch_dependent(kern, unsigned(grid), unsigned(kTmaPipeThreads), smem, L.stream, a);
    if (err != cudaSuccess) return err;
    if (info) {
        info->kernel = MODE == MODE_AR ? "allreduce_tma_wide" : "reduce_scatter_tma_wide";
        info->grid = grid;
        info->block = kTmaPipeThreads;
        info->smem = smem;
        info->kernels = 1;
        info->counter = a.dynamic;
    }
    return cudaGetLastError();
}

template <typename T, int OP, int MODE>
static cudaError_t tma_launch_op_mode(const Launch &L, LaunchInfo *info)
{
    switch (L.p) {
    case 2: return tma_launch_p<T, OP, 2, MODE>(L, info);
    case 3: return tma_launch_p<T, OP, 3, MODE>(L, info);
    case 4: return tma_launch_p<T, OP, 4, MODE>(L, info);
    case 8: return tma_launch_p<T, OP, 8, MODE>(L, info);
    default:
        return L.p > kTmaNarrowMaxRanks ? tma_wide_launch<T, OP, MODE>(L, info)
                                        : tma_launch_p<T, OP, 0, MODE>(L, info);
    }
}

template <typename T, int OP>
static cudaError_t tma_launch_op(const Launch &L, LaunchInfo *info)
{
    return L.mode == MODE_AR ? tma_launch_op_mode<T, OP, MODE_AR>(L, info)
                             : tma_launch_op_mode<T, OP, MODE_RS>(L, info);
}

template <typename T>
static cudaError_t launch_tma(const Launch &L, LaunchInfo *info)
{
    switch (L.op) {
    case OP_SUM: return tma_launch_op<T, OP_SUM>(L, info);
    case OP_PROD: return tma_launch_op<T, OP_PROD>(L, info);
    case OP_MIN: return tma_launch_op<T, OP_MIN>(L, info);
    case OP_MAX: return tma_launch_op<T, OP_MAX>(L, info);
    case OP_AVG: return tma_launch_op<T, OP_AVG>(L, info);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ccl
