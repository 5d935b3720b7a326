// Internal interface between the host front end (ccl.cpp) and the kernel
// translation units.  Not installed; the public interface is include/ccl.h.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ccl.h"

namespace ccl {

constexpr int kMaxRanks = 64;

enum Op : int { OP_SUM = 0, OP_PROD = 1, OP_MIN = 2, OP_MAX = 3, OP_AVG = 4 };
enum Dtype : int { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2, DT_I32 = 3 };
enum Mode : int { MODE_AR = 0, MODE_RS = 1 };

inline size_t elem_bytes(int dtype) { return (dtype == DT_F16 || dtype == DT_BF16) ? 2 : 4; }

// One chunk table: chunk c is elements [bound[c], bound[c+1]) and is folded
// in rank order order[c*p + 0], order[c*p + 1], ...
struct Table {
    int p = 0;
    uint64_t n = 0;
    uint64_t bound[kMaxRanks + 1];
    uint8_t order[kMaxRanks * kMaxRanks];
};

// What the front end decided; the kernel TUs turn it into a launch.
struct Launch {
    int p = 0;
    int op = 0;
    int dtype = 0;
    int mode = MODE_AR;
    uint64_t n = 0;
    const void *src[kMaxRanks];
    void *dst[kMaxRanks];
    const Table *table = nullptr;
    bool vec = false;          // 16-byte vector body allowed
    uint64_t self_mask = 0;    // AllGather: bit r set when dst[r] == src[r] (in place)
    bool alias = false;        // some output is (part of) an input: in-place loads, no ld.global.nc
    int device = 0;            // the current device while the kernel is launched
    int num_sms = 0;
    int sm_budget = 0;         // 0 = all SMs
    size_t pipe_bytes = 0;     // TMA stage bytes per rank
    unsigned *status = nullptr;  // device status block
    bool tile_counter = true;  // TMA: large messages may take tiles from a counter in the status block
    long long wait_limit_ns = 0;
    int stall_test = 0;
    cudaStream_t stream = nullptr;
};

// Filled by a launcher for diagnostics.
struct LaunchInfo {
    const char *kernel = "";
    int grid = 0;
    int block = 0;
    size_t smem = 0;
    int kernels = 0;           // kernels launched
    int counter = 0;           // 1: CTAs or warps took work from a device-wide counter
};

// Status-block code of an access outside a rank buffer that a kernel of the
// checked build computed and skipped (device.cuh, in_bounds).
constexpr unsigned kBoundsCode = 16;

// TMA variant geometry: tile bytes T per rank per stage and the stage count
// S for p ranks.  A stage holds p input tiles and one output tile; S fills
// the 227 KB of shared memory one CTA may address (one CTA per SM).  T-CCL
// ("Experimental Environment") uses 8 KB chunks.  want_tile != 0 forces T.
// False if no geometry fits.
constexpr size_t kTmaSmemLimit = 227 * 1024;
constexpr int kTmaMaxStages = 8;
constexpr size_t kTmaCtlBytes = 128;
constexpr size_t kTmaNarrowCtlBytes = 256;   // pipelined kernels: four barrier arrays and a larger control block

// Grids of at most this many CTAs (an SM budget) take larger narrow tiles.
constexpr int kTmaSmallGrid = 32;

// Default narrow tile.  Under a budget the kernel's rate per SM rises with
// the bytes per bulk copy until the SM's port to the crossbar bounds it near
// 100-105 GB/s; at a given tile, stages of two or three ranks are slower
// still (measured on GB300, AllReduce, bf16, GB/s per SM at 8 SMs: 8 KB
// tiles p=2 49, p=4 82, p=8 105; p=2 with 16 / 24 / 32 KB 79 / 103 / 92).
// Across many SMs more, smaller stages hide DRAM latency better and keep
// every SM busy on mid-size messages.  Chosen (8-32 SMs; whole GPU):
//   p=2:    24 KB on small grids (103 vs 79 with 16 KB), 16 KB otherwise
//           (whole GPU: 7112 vs 6712 with 8 KB; 4 MiB per rank: 3816 vs 3357
//           with 24 KB)
//   p=3:    16 KB (small grids: 105, 97 with 24 KB -- through its own
//           instantiation; the generic one moved 77-85)
//   p=4:    12 KB on small grids (105 vs 82 with 8 KB), 8 KB otherwise
//   p=5:    12 KB (101 vs 80; 76 SMs 85 vs 77; whole GPU within 0.4 %)
//   p=6:    12 KB on small grids (90 vs 82), 8 KB otherwise (76 SMs: 81 vs 72)
//   p=7-13: 8 KB (p=12: 99 vs 67 with 4 KB; p=7 with 12 KB: +3 % on 8 SMs, -10 % on 76)
inline size_t tma_default_tile(int p, int sm_budget)
{
    const bool small = sm_budget > 0 && sm_budget <= kTmaSmallGrid;
    if (small) return p == 2 ? 24576 : p == 3 ? 16384 : p <= 6 ? 12288 : 8192;
    return p <= 3 ? 16384 : p == 5 ? 12288 : 8192;
}

inline bool tma_geometry(int p, size_t want_tile, int sm_budget, uint32_t *tile, uint32_t *stages, size_t *smem)
{
    size_t T = want_tile ? want_tile : tma_default_tile(p, sm_budget);
    for (; T >= 1024; T /= 2) {
        const size_t per_stage = size_t(p + 1) * T;
        size_t S = (kTmaSmemLimit - 4 * kTmaMaxStages * 8 - kTmaNarrowCtlBytes) / per_stage;
        if (S > size_t(kTmaMaxStages)) S = kTmaMaxStages;
        if (S >= 2) {
            *tile = uint32_t(T);
            *stages = uint32_t(S);
            *smem = S * per_stage + 4 * S * 8 + kTmaNarrowCtlBytes;
            return true;
        }
        if (want_tile) return false;
    }
    return false;
}

// Above kTmaNarrowMaxRanks ranks a stage holding one tile of every rank
// would force tiles below 8 KB (p+1 of them per stage, two stages), and
// smaller bulk copies cost more per byte.  The wide geometry keeps 8 or
// 16 KB per copy and brings the p ranks through the stages R at a time (a
// tile takes ceil(p/R) stages); kTmaWideOut output tiles sit beside the
// stages.  T <= 16 KB so that each consumer thread folds at most four 16-byte
// groups per tile in registers.  Measured on GB300 (AllReduce, bf16), wide
// (8 ranks of 8 KB) against narrow: p=14 on 16 SMs 84 vs 84 GB/s per SM (6 KB
// tiles), on 76 SMs 81 vs 77, whole GPU +1 %; p=16 90 vs 78 (4 KB tiles); p=24
// 93 vs 77; p=32 93 vs 48 (2 KB); p=13 83 vs 99 (narrow, 8 KB tiles) -- so
// the wide kernel from 14 ranks.  Stages of 4 ranks of 16 KB (half the
// copies per byte) against 8 of 8 KB: on 8-16 SMs p=16 95-96 vs 94, p=24 98-99
// vs 95, p=64 99 vs 95; on 76 SMs -1 to -3 %, on the whole GPU -0.5 % and up
// to -7 % at 4-16 MiB per rank -- so 4 x 16 KB on grids of at most
// kTmaSmallGrid CTAs, 8 x 8 KB otherwise.  More output tiles (3 or 4)
// measured the same as two.
constexpr int kTmaNarrowMaxRanks = 13;
constexpr int kTmaWideRanks = 8;          // the most ranks a stage holds
constexpr int kTmaWideOut = 2;            // output tiles
constexpr size_t kTmaWideMaxTile = 16384;

inline bool tma_wide_geometry(int p, size_t want_tile, int sm_budget, uint32_t *tile, uint32_t *ranks,
                              uint32_t *stages, size_t *smem)
{
    const bool small = sm_budget > 0 && sm_budget <= kTmaSmallGrid;
    const size_t T = want_tile ? want_tile : (small ? 16384 : 8192);
    if (T > kTmaWideMaxTile || T < 1024) return false;
    const size_t per = T > 8192 ? 4 : size_t(kTmaWideRanks);  // ranks per stage: 64 KB stages at most
    const size_t R = size_t(p) < per ? size_t(p) : per;
    // out tiles, four barrier arrays (full/empty per stage, folded/out_free per out tile), control block
    const size_t fixed = kTmaWideOut * T + 2 * (kTmaMaxStages + kTmaWideOut) * 8 + kTmaNarrowCtlBytes;
    size_t S = (kTmaSmemLimit - fixed) / (R * T);
    if (S > size_t(kTmaMaxStages)) S = kTmaMaxStages;
    if (S < 2) return false;
    *tile = uint32_t(T);
    *ranks = uint32_t(R);
    *stages = uint32_t(S);
    *smem = S * R * T + kTmaWideOut * T + 2 * (S + kTmaWideOut) * 8 + kTmaNarrowCtlBytes;
    return true;
}

// Bulk-reduce variant: the reductions the PTX bulk-reduce instruction
// provides (sum on f32/f16/bf16/i32, min/max on f16/bf16/i32), and its
// geometry: two stages of p tiles, small enough for several CTAs per SM.
inline bool bulkred_supported(int dtype, int op)
{
    if (op == OP_SUM) return true;
    if (op == OP_MIN || op == OP_MAX) return dtype != DT_F32;
    return false;
}

inline bool bulkred_geometry(int p, size_t want_tile, uint32_t *tile, uint32_t *ranks, uint32_t *stages,
                             size_t *smem)
{
    // Up to 16 ranks a stage holds a tile of every rank, about 64 KB per
    // pipe (three pipes per SM).  Above 16 the ranks pass through the stages
    // eight at a time with 4 KB tiles, instead of shrinking the tiles to 1 KB.
    // tile measured on GB300 (AllReduce, every SM): p=2 16 KB 5510 vs 8 KB 4914 GB/s (the same at 16 SMs);
    // p=4 8 KB (16 KB: +2.5 % on every SM, -10 % at 16 SMs); p=8 4 KB; p=16 2 KB
    const size_t R = p <= 16 ? size_t(p) : 8;
    size_t T = want_tile ? want_tile : (p <= 2 ? 16384 : p <= 4 ? 8192 : p <= 8 ? 4096 : p <= 16 ? 2048 : 4096);
    const uint32_t S = 2;
    for (; T >= 1024; T /= 2) {
        const size_t bytes = size_t(S) * R * T + 2 * S * 8 + kTmaCtlBytes;
        if (bytes <= kTmaSmemLimit) {
            *tile = uint32_t(T);
            *ranks = uint32_t(R);
            *stages = S;
            *smem = bytes;
            return true;
        }
        if (want_tile) return false;
    }
    return false;
}

// Per-dtype AllReduce / ReduceScatter launchers (ld/st variant).  They pick
// the in-place instantiation (coherent loads, reduce_{dtype}_inplace.cu)
// when L.alias is set.
cudaError_t launch_reduce_f32(const Launch &L, LaunchInfo *info);
cudaError_t launch_reduce_f16(const Launch &L, LaunchInfo *info);
cudaError_t launch_reduce_bf16(const Launch &L, LaunchInfo *info);
cudaError_t launch_reduce_i32(const Launch &L, LaunchInfo *info);
cudaError_t launch_reduce_inplace_f32(const Launch &L, LaunchInfo *info);
cudaError_t launch_reduce_inplace_f16(const Launch &L, LaunchInfo *info);
cudaError_t launch_reduce_inplace_bf16(const Launch &L, LaunchInfo *info);
cudaError_t launch_reduce_inplace_i32(const Launch &L, LaunchInfo *info);

// Per-dtype AllReduce / ReduceScatter launchers (TMA variant).
cudaError_t launch_tma_f32(const Launch &L, LaunchInfo *info);
cudaError_t launch_tma_f16(const Launch &L, LaunchInfo *info);
cudaError_t launch_tma_bf16(const Launch &L, LaunchInfo *info);
cudaError_t launch_tma_i32(const Launch &L, LaunchInfo *info);

// Per-dtype bulk-reduce launchers: the ReduceScatter core (for MODE_AR chunk c
// is written into rank c's output at the chunk's offset; the caller then runs
// the in-place AllGather).
cudaError_t launch_bulkred_f32(const Launch &L, LaunchInfo *info);
cudaError_t launch_bulkred_f16(const Launch &L, LaunchInfo *info);
cudaError_t launch_bulkred_bf16(const Launch &L, LaunchInfo *info);
cudaError_t launch_bulkred_i32(const Launch &L, LaunchInfo *info);

// AllGather (broadcast store), dtype-agnostic beyond the element size.
cudaError_t launch_gather(const Launch &L, LaunchInfo *info);

// Comparison executors: the ring run hop by hop (stepwise = true) or the
// one-phase all-pairs reduction (stepwise = false); AllReduce only.
cudaError_t launch_compare(const Launch &L, LaunchInfo *info, bool stepwise);

// AllReduce fused with the residual merge and RMSNorm (rmsnorm.cu).
struct NormLaunch {
    const void *residual = nullptr;
    void *residual_out = nullptr;
    const void *gamma = nullptr;
    uint64_t rows = 0;
    uint64_t hidden = 0;
    float eps = 0.0f;
};
cudaError_t launch_allreduce_rmsnorm(const Launch &L, const NormLaunch &N, LaunchInfo *info);

// The measured launch table (launch_table.cpp): the estimated per-call time
// (us) of an AllReduce with the ld/st or TMA kernel, and AUTO's choice.
// num_sms 0 = the SM count of the device the table was measured on.
bool launch_table_estimate(int p, int elem_bytes, int sm_budget, int num_sms, double bytes_per_rank, int variant,
                           double *us);
bool launch_table_prefers_tma(int p, int elem_bytes, int sm_budget, int num_sms, double bytes_per_rank);
int launch_table_points();

// Sets the message ccl_last_error() returns on this host thread; returns st.
ccl_status_t record_error(ccl_status_t st, const char *msg);

}  // namespace ccl
