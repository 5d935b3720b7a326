// AllReduce fused with the residual merge and RMSNorm.
//
// "Inside NCCL AllReduce", last section: in Kimi's decoding path the
// residual merge and the RMSNorm after the all-reduce run inside the
// all-reduce kernel, one kernel fewer per layer.  Per row of a [rows, hidden] buffer:
//   y   = sum AllReduce of the p rank rows (schedule order, fp32, rounded)
//   h   = round(y + residual)                     written to residual_out
//   out = round(h * (1 / sqrt(mean(h^2) + eps)) * gamma)   written to every rank
// A thread-block cluster of C CTAs per row, each CTA a slice of the columns
// (for decode, C up to 8 so that a row of 8192 columns is spread over 1024
// threads; for many rows, one CTA per row).  Pass 1 folds the p inputs, merges the residual, stores h and
// accumulates the slice's sum of squares of the rounded h; the C partial sums
// are exchanged through distributed shared memory -- each CTA pushes its sum
// into every CTA of the row with st.async and waits on its own mbarrier for
// the C sums (every CTA adds the same C values in the same order, so all
// slices use one bit-identical 1/rms) -- and pass 2 normalises the h values
// the same thread produced (kept in registers, with gamma, for the first few
// units of each thread) and writes the slice to all p outputs.  The exchange
// wait is bounded by the communicator's wait limit; on expiry the CTA records
// it in the status block (ccl_comm_check reports CCL_ERR_TIMEOUT), waits once
// more, bounded, for late writes into its shared memory, and finishes.  The
// only barrier is the cluster barrier before the first remote write, which
// every CTA of the row reaches.  Each element
// is read from the rank inputs once; all arithmetic is fp32 with explicit
// round-to-nearest operations (1/sqrtf is IEEE-rounded under the default
// flags).  Bytes: (2p + 2) n s + hidden s.  Loads are coherent (no
// ld.global.nc): the residual is usually updated in place, and the rank
// outputs may be the inputs.
#include <cooperative_groups.h>

#include "device.cuh"

namespace ccl {

namespace cg = cooperative_groups;

constexpr int kNormDecodeThreads = 128;
constexpr int kNormMidThreads = 1024;
constexpr int kNormPrefillThreads = 256;
constexpr int kNormMaxCluster = 8;

template <int PM>
struct NormArgs {
    const void *src[PM];
    void *dst[PM];
    uint64_t bound[PM + 1];
    uint8_t order[PM][PM];
    const void *residual;
    void *residual_out;
    const void *gamma;
    uint64_t rows;
    uint64_t hidden;
    int p;
    int vec;        // 16-byte groups: pointers aligned, hidden and every chunk boundary multiples of VEC
    float eps;
    unsigned *status;   // the communicator's status block: a wait that gave up is recorded here
    long long wait_ns;  // bound on the exchange wait
    int stall_test;     // 1: cluster rank 1 withholds its slice sum, so the exchange wait runs out (tests)
};

__device__ __forceinline__ uint32_t cl_map(uint32_t local, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

__device__ __forceinline__ bool cl_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

template <typename T, int PM>
__device__ __forceinline__ float fold_one(const NormArgs<PM> &a, int p, uint64_t e)
{
    using Tr = Traits<T>;
    using F = Fold<T, OP_SUM>;
    int c = 0;
    while (e >= a.bound[c + 1]) ++c;
    float acc = Tr::load1(a.src[a.order[c][0]], e);
    for (int k = 1; k < p; ++k) acc = F::fold(acc, Tr::load1(a.src[a.order[c][k]], e), 1.0f);
    return acc;
}

template <typename T>
__device__ __forceinline__ float round_to(float v)
{
    alignas(4) unsigned char tmp[4];
    Traits<T>::store1(tmp, 0, v);
    return Traits<T>::load1(tmp, 0);
}

__device__ __forceinline__ float block_sum(float v, float *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = lane < int(blockDim.x / 32) ? red[lane] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[0] = v;
    }
    __syncthreads();
    v = red[0];
    __syncthreads();
    return v;
}

template <typename T, int P, int THREADS>
__global__ void __launch_bounds__(THREADS) ar_rmsnorm_kernel(const __grid_constant__ NormArgs<(P > 0 ? P : kMaxRanks)> a)
{
    using Tr = Traits<T>;
    using F = Fold<T, OP_SUM>;
    constexpr int VEC = Tr::VEC;
    constexpr int S = (VEC == 8) ? 2 : 4;
    __shared__ float red[32];
    __shared__ float parts[kNormMaxCluster];
    __shared__ __align__(8) uint64_t xbar;
    cg::cluster_group cluster = cg::this_cluster();
    const int C = int(cluster.num_blocks());
    const int q = int(cluster.block_rank());
    if (C > 1) {
        // the exchange barrier must be initialised before any peer signals it:
        // arrive now, wait just before the first remote write (pass 1 hides it)
        if (threadIdx.x == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(uint32_t(__cvta_generic_to_shared(&xbar))) : "memory");
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    }
    grid_dependency_wait();
    grid_dependents_launch();
    const int p = P > 0 ? P : a.p;
    const uint64_t H = a.hidden;
    const uint64_t row = blockIdx.x / C;
    const uint64_t base = row * H;
    // this CTA's slice: units are 16-byte groups (vec) or elements
    const uint64_t units = a.vec ? H / VEC : H;
    const uint64_t u0 = units * q / C, u1 = units * (q + 1) / C;

    // The decode and mid shapes (one unit per thread at hidden 8192) keep h
    // and gamma in registers between the passes: 3.43 vs 3.79 us per decode
    // call, 4.59 vs 5.31 at 32 tokens.  The prefill shape re-reads them from
    // L2: keeping four units' worth doubles its registers, halves the CTAs
    // per SM and costs 1.5 % at 4096 tokens.  Units beyond KEEP re-read.
    constexpr int KEEP = THREADS == kNormPrefillThreads ? 0 : 1;
    uint4 hkeep[KEEP > 0 ? KEEP : 1], gkeep[KEEP > 0 ? KEEP : 1];

    float ss = 0.0f;
    // pass 1: fold, merge, keep h, sum of squares
    if (a.vec) {
        auto pass1 = [&](uint64_t g, uint4 *hk, uint4 *gk) {
            const uint64_t e = base + g * VEC;
            // rank buffers hold rows * hidden elements, gamma hidden
            if (!in_bounds(e + VEC <= a.rows * H && (g + 1) * VEC <= H, a.status, kSiteNorm, e)) return;
            if (gk) *gk = *reinterpret_cast<const uint4 *>(static_cast<const char *>(a.gamma) + g * VEC * S);
            int c = 0;
            while (e >= a.bound[c + 1]) ++c;
            float acc[VEC], v[VEC];
            if constexpr (P > 0) {
                uint4 r[P];
                if constexpr (THREADS <= 128) {
                    // decode (few rows): all p loads in flight before the first
                    // fold -- 3.89 vs 4.03 us per decode call on GB300
                    const char *sp[P];
#pragma unroll
                    for (int k = 0; k < P; ++k) sp[k] = static_cast<const char *>(a.src[a.order[c][k]]) + e * S;
#pragma unroll
                    for (int k = 0; k < P; ++k) r[k] = ld_coherent_v4(sp[k]);
                    hold_batch(r);
                } else {
                    // many rows: the compiler's interleaved schedule uses fewer
                    // registers and keeps more CTAs resident (measured with
                    // 512-thread CTAs: 193 vs 202 us at 4096 tokens)
#pragma unroll
                    for (int k = 0; k < P; ++k)
                        r[k] = ld_coherent_v4(static_cast<const char *>(a.src[a.order[c][k]]) + e * S);
                }
                Tr::unpack(r[0], acc);
#pragma unroll
                for (int k = 1; k < P; ++k) {
                    Tr::unpack(r[k], v);
#pragma unroll
                    for (int i = 0; i < VEC; ++i) acc[i] = F::fold(acc[i], v[i], 1.0f);
                }
            } else {
                Tr::unpack(ld_coherent_v4(static_cast<const char *>(a.src[a.order[c][0]]) + e * S), acc);
                for (int k = 1; k < p; ++k) {
                    Tr::unpack(ld_coherent_v4(static_cast<const char *>(a.src[a.order[c][k]]) + e * S), v);
#pragma unroll
                    for (int i = 0; i < VEC; ++i) acc[i] = F::fold(acc[i], v[i], 1.0f);
                }
            }
            Tr::unpack(Tr::pack(acc), acc);                                  // y, rounded
            Tr::unpack(ld_coherent_v4(static_cast<const char *>(a.residual) + e * S), v);
#pragma unroll
            for (int i = 0; i < VEC; ++i) acc[i] = __fadd_rn(acc[i], v[i]);   // the merge
            const uint4 hq = Tr::pack(acc);
            st_v4(static_cast<char *>(a.residual_out) + e * S, hq);
            if (hk) *hk = hq;
            Tr::unpack(hq, acc);                                             // h, rounded
#pragma unroll
            for (int i = 0; i < VEC; ++i) ss = __fadd_rn(ss, __fmul_rn(acc[i], acc[i]));
        };
#pragma unroll
        for (int j = 0; j < KEEP; ++j) {
            const uint64_t g = u0 + threadIdx.x + uint64_t(j) * blockDim.x;
            if (g < u1) pass1(g, &hkeep[j], &gkeep[j]);
        }
        for (uint64_t g = u0 + threadIdx.x + uint64_t(KEEP) * blockDim.x; g < u1; g += blockDim.x)
            pass1(g, nullptr, nullptr);
    } else {
        for (uint64_t j = u0 + threadIdx.x; j < u1; j += blockDim.x) {
            const uint64_t e = base + j;
            if (!in_bounds(e < a.rows * H && j < H, a.status, kSiteNorm, e)) continue;
            const float y = round_to<T>(fold_one<T>(a, p, e));
            const float h = round_to<T>(__fadd_rn(y, Tr::load1(a.residual, e)));
            Tr::store1(a.residual_out, e, h);
            ss = __fadd_rn(ss, __fmul_rn(h, h));
        }
    }
    const float part = block_sum(ss, red);
    float total = part;
    if (C > 1) {
        bool gave_up = false;
        // push: every CTA writes its slice sum into parts[q] of every CTA of the
        // row (itself included) and waits for the C sums to land in its own
        // shared memory -- no cluster barrier round trip, no remote reads.  A
        // CTA leaves only after all C writes into it have landed, so none is
        // written after it has gone.  Measured on GB300 (p=8 bf16, hidden 8192,
        // per call in a CUDA graph) against a cluster barrier followed by C
        // remote reads: 1 token 3.20 -> 2.67 us, 32 tokens 3.60 -> 3.07, 128
        // tokens 6.58 -> 6.00, 256 and 4096 tokens unchanged; the same bits.
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
        const uint32_t lbar = uint32_t(__cvta_generic_to_shared(&xbar));
        if (threadIdx.x == 0)
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(lbar), "r"(uint32_t(C * 4)) : "memory");
        if (int(threadIdx.x) < C && !(a.stall_test == 1 && q == 1)) {
            const uint32_t k = threadIdx.x;
            const uint32_t raddr = cl_map(uint32_t(__cvta_generic_to_shared(&parts[q])), k);
            const uint32_t rbar = cl_map(lbar, k);
            asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
                         ::"r"(raddr), "r"(__float_as_uint(part)), "r"(rbar) : "memory");
        }
        if (!cl_try_wait(lbar, 0)) {
            const uint64_t t0 = [] { uint64_t t; asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)); return t; }();
            for (;;) {
                if (cl_try_wait(lbar, 0)) break;
                uint64_t t;
                asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
                if (t - t0 > uint64_t(a.wait_ns)) {
                    if (a.status && atomicCAS(&a.status[0], 0u, 5u) == 0u) {
                        a.status[1] = blockIdx.x;
                        a.status[2] = unsigned(row);
                        a.status[3] = threadIdx.x;
                    }
                    gave_up = true;
                    break;
                }
            }
        }
        if (gave_up) {
            // A sum is missing (recorded above; this call's outputs are
            // wrong).  Wait once more, again bounded, so that a late peer's
            // write is not left to land after this CTA has gone, then go on.
            uint64_t t1;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
            for (;;) {
                if (cl_try_wait(lbar, 0)) break;
                uint64_t t;
                asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
                if (t - t1 > uint64_t(a.wait_ns)) break;
            }
        }
        total = 0.0f;
        for (int k = 0; k < C; ++k) total = __fadd_rn(total, parts[k]);
    }
    const float inv = 1.0f / sqrtf(__fadd_rn(__fdiv_rn(total, float(H)), a.eps));

    // pass 2: normalise the h this thread stored, broadcast to every rank
    if (a.vec) {
        auto pass2 = [&](uint64_t g, const uint4 &hq, const uint4 &gq) {
            const uint64_t e = base + g * VEC;
            if (!in_bounds(e + VEC <= a.rows * H && (g + 1) * VEC <= H, a.status, kSiteNorm, e)) return;
            float h[VEC], gm[VEC];
            Tr::unpack(hq, h);
            Tr::unpack(gq, gm);
#pragma unroll
            for (int i = 0; i < VEC; ++i) h[i] = __fmul_rn(__fmul_rn(h[i], inv), gm[i]);
            const uint4 out = Tr::pack(h);
            if constexpr (P > 0) {
#pragma unroll
                for (int k = 0; k < P; ++k) st_stream_v4(static_cast<char *>(a.dst[k]) + e * S, out);
            } else {
                for (int k = 0; k < p; ++k) st_stream_v4(static_cast<char *>(a.dst[k]) + e * S, out);
            }
        };
#pragma unroll
        for (int j = 0; j < KEEP; ++j) {
            const uint64_t g = u0 + threadIdx.x + uint64_t(j) * blockDim.x;
            if (g < u1) pass2(g, hkeep[j], gkeep[j]);
        }
        for (uint64_t g = u0 + threadIdx.x + uint64_t(KEEP) * blockDim.x; g < u1; g += blockDim.x) {
            const uint64_t e = base + g * VEC;
            if (!in_bounds(e + VEC <= a.rows * H && (g + 1) * VEC <= H, a.status, kSiteNorm, e)) continue;
            pass2(g, *reinterpret_cast<const uint4 *>(static_cast<const char *>(a.residual_out) + e * S),
                  *reinterpret_cast<const uint4 *>(static_cast<const char *>(a.gamma) + g * VEC * S));
        }
    } else {
        for (uint64_t j = u0 + threadIdx.x; j < u1; j += blockDim.x) {
            const uint64_t e = base + j;
            if (!in_bounds(e < a.rows * H && j < H, a.status, kSiteNorm, e)) continue;
            const float o = __fmul_rn(__fmul_rn(Tr::load1(a.residual_out, e), inv), Tr::load1(a.gamma, j));
            for (int k = 0; k < p; ++k) Tr::store1(a.dst[k], e, o);
        }
    }
}

template <typename T, int P>
static cudaError_t norm_launch(const Launch &L, const NormLaunch &N, LaunchInfo *info)
{
    constexpr int PM = P > 0 ? P : kMaxRanks;
    NormArgs<PM> a;
    for (int k = 0; k < L.p; ++k) {
        a.src[k] = L.src[k];
        a.dst[k] = L.dst[k];
    }
    for (int c = 0; c <= L.p; ++c) a.bound[c] = L.table->bound[c];
    for (int c = 0; c < L.p; ++c)
        for (int k = 0; k < L.p; ++k) a.order[c][k] = L.table->order[c * L.p + k];
    a.residual = N.residual;
    a.residual_out = N.residual_out;
    a.gamma = N.gamma;
    a.rows = N.rows;
    a.hidden = N.hidden;
    a.p = L.p;
    a.vec = L.vec ? 1 : 0;
    a.eps = N.eps;
    a.status = L.status;
    a.wait_ns = L.wait_limit_ns > 0 ? L.wait_limit_ns : 2000000000LL;
    a.stall_test = L.stall_test;
    // CTA shape by rows against the SM count; a row takes a cluster of C CTAs
    // only when it needs more than one.  Measured on GB300 (p=8 bf16, hidden
    // 8192, per call, CUDA-graph replay):
    //   rows < SMs (decode): 128 threads, one unit each, up to 8 CTAs a row --
    //     latency rules;
    //   SMs <= rows < 2 SMs: 1024 threads, one unit each -- 256 tokens
    //     12.96 us against 16.13 with 512 threads x 2 units;
    //   rows >= 2 SMs (prefill): 256 threads, four units each, so more and
    //     smaller CTAs per SM overlap one another's block reductions -- 4096
    //     tokens 188 vs 194 us, 8192 tokens 367 vs 384.
    const uint64_t units = L.vec ? N.hidden / Traits<T>::VEC : N.hidden;
    const uint64_t sms = uint64_t(L.num_sms);
    const int threads = N.rows < sms ? kNormDecodeThreads : N.rows < 2 * sms ? kNormMidThreads : kNormPrefillThreads;
    const uint64_t per_cta = uint64_t(threads) * (N.rows < 2 * sms ? 1 : 4);
    const uint64_t want = (units + per_cta - 1) / per_cta;
    const int C = int(want < 1 ? 1 : want > uint64_t(kNormMaxCluster) ? kNormMaxCluster : want);
    if (N.rows * uint64_t(C) > 0x7fffffffull) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(N.rows * C));
    cfg.blockDim = dim3(unsigned(threads));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // launched as a dependent
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = unsigned(C);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = C > 1 ? 2 : 1;  // one CTA per row: no cluster needed
    cudaError_t err = threads == kNormDecodeThreads ? cudaLaunchKernelEx(&cfg, ar_rmsnorm_kernel<T, P, kNormDecodeThreads>, a)
                      : threads == kNormMidThreads  ? cudaLaunchKernelEx(&cfg, ar_rmsnorm_kernel<T, P, kNormMidThreads>, a)
                                                    : cudaLaunchKernelEx(&cfg, ar_rmsnorm_kernel<T, P, kNormPrefillThreads>, a);
    if (err != cudaSuccess) return err;
    const int grid = int(N.rows * C);
    if (info) {
        info->kernel = "allreduce_residual_rmsnorm";
        info->grid = grid;
        info->block = threads;
        info->smem = 0;
        info->kernels = 1;
    }
    return cudaGetLastError();
}

template <typename T>
static cudaError_t norm_dtype(const Launch &L, const NormLaunch &N, LaunchInfo *info)
{
    return L.p == 8 ? norm_launch<T, 8>(L, N, info) : norm_launch<T, 0>(L, N, info);
}

cudaError_t launch_allreduce_rmsnorm(const Launch &L, const NormLaunch &N, LaunchInfo *info)
{
    switch (L.dtype) {
    case DT_F32: return norm_dtype<F32>(L, N, info);
    case DT_F16: return norm_dtype<F16>(L, N, info);
    case DT_BF16: return norm_dtype<BF16>(L, N, info);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ccl
