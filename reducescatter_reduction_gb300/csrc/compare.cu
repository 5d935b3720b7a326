// Comparison executors for the pages' other AllReduce algorithms, run on one
// GPU so that their cost can be measured against the fused kernel.
//
// Stepwise ring ("Inside NCCL AllReduce", section "The ring, exactly as the
// kernel runs it"): 2(p-1) launches, one per hop.  Reduce-scatter hop h
// (1 <= h < p): for every chunk c, rank d = (c+1+h) mod p receives the
// partial held by rank (c+h) mod p (at h = 1, that rank's own contribution),
// adds its contribution in fp32 and keeps the result, rounded to the element
// type, in its output buffer at the chunk's place -- the partial lives in a
// buffer between hops, as it does in a ring of GPUs.  All-gather hop h: rank
// (c+h) mod p copies the finished chunk from rank (c+h-1) mod p.  Bytes:
// 3(p-1) n s for the reduce-scatter hops + 2(p-1) n s for the all-gather hops,
// against 2 p n s for the fused kernel.
//
// One-phase all-pairs (MSCCL++, section on the 1PA algorithm: every rank
// reads every peer's data and reduces all of it itself): each rank's output is
// computed independently from all p inputs, in the chunk's order -- the fused
// kernel's bits with p times its reads (p^2 n s read + p n s written).
//
// Loads are coherent (no ld.global.nc): in place, a reduce-scatter hop reads
// a rank's contribution and overwrites it with the partial.
#include "device.cuh"

namespace ccl {

constexpr int kCmpThreads = 256;

struct CmpArgs {
    const void *src[kMaxRanks];
    void *dst[kMaxRanks];
    uint64_t bound[kMaxRanks + 1];
    uint8_t order[kMaxRanks][kMaxRanks];
    uint64_t n;
    int p;
    int hop;        // stepwise: 1 .. p-1
    int vec;        // 16-byte groups (every chunk boundary and pointer aligned)
    float scale;
};

template <int VEC>
__device__ __forceinline__ int chunk_of(const CmpArgs &a, uint64_t e, int c)
{
    while (e >= a.bound[c + 1]) ++c;
    return c;
}

// ---------------------------------------------------------------------------
// Stepwise ring: one reduce-scatter hop.
// ---------------------------------------------------------------------------

template <typename T, int OP>
__device__ __forceinline__ void rs_hop_one(const CmpArgs &a, int c, uint64_t e)
{
    using Tr = Traits<T>;
    using F = Fold<T, OP>;
    const int p = a.p, h = a.hop;
    const int d = (c + 1 + h) % p;
    typename Tr::Acc held;
    if (h == 1) {
        // the first rank's contribution as it would be sent: scaled (avg), in the element type
        auto v = F::first(Tr::load1(a.src[(c + 1) % p], e), a.scale);
        alignas(4) unsigned char tmp[4];
        Tr::store1(tmp, 0, v);
        held = Tr::load1(tmp, 0);
    } else {
        held = Tr::load1(a.dst[(c + h) % p], e);
    }
    auto acc = F::fold(held, Tr::load1(a.src[d], e), a.scale);
    if (h == p - 1) acc = F::finish(acc, p);
    Tr::store1(a.dst[d], e, acc);
}

template <typename T, int OP>
__global__ void __launch_bounds__(kCmpThreads) ring_rs_hop_kernel(const __grid_constant__ CmpArgs a)
{
    using Tr = Traits<T>;
    using F = Fold<T, OP>;
    using Acc = typename Tr::Acc;
    constexpr int VEC = Tr::VEC;
    constexpr int S = (VEC == 8) ? 2 : 4;
    const uint64_t tid = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
    const int p = a.p, h = a.hop;
    const uint64_t ngroups = a.vec ? a.n / VEC : 0;
    for (uint64_t g = tid; g < ngroups; g += stride) {
        const uint64_t e = g * VEC;
        const int c = chunk_of<VEC>(a, e, 0);
        const int d = (c + 1 + h) % p;
        Acc held[VEC], v[VEC];
        if (h == 1) {
            Tr::unpack(ld_coherent_v4(static_cast<const char *>(a.src[(c + 1) % p]) + e * S), v);
#pragma unroll
            for (int i = 0; i < VEC; ++i) v[i] = F::first(v[i], a.scale);
            Tr::unpack(Tr::pack(v), held);              // held in the element type
        } else {
            Tr::unpack(ld_coherent_v4(static_cast<const char *>(a.dst[(c + h) % p]) + e * S), held);
        }
        Tr::unpack(ld_coherent_v4(static_cast<const char *>(a.src[d]) + e * S), v);
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            held[i] = F::fold(held[i], v[i], a.scale);
            if (h == p - 1) held[i] = F::finish(held[i], p);
        }
        st_stream_v4(static_cast<char *>(a.dst[d]) + e * S, Tr::pack(held));
    }
    for (uint64_t e = ngroups * VEC + tid; e < a.n; e += stride) rs_hop_one<T, OP>(a, chunk_of<VEC>(a, e, 0), e);
}

// All-gather hop: copy each finished chunk one rank further along the ring.
template <int U>
__global__ void __launch_bounds__(kCmpThreads) ring_ag_hop_kernel(const __grid_constant__ CmpArgs a, int vec_units)
{
    const uint64_t tid = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
    const int p = a.p, h = a.hop;
    const uint64_t nunits = a.n / vec_units;
    for (uint64_t u = tid; u < nunits; u += stride) {
        const uint64_t e = u * vec_units;
        const int c = chunk_of<1>(a, e, 0);
        const char *from = static_cast<const char *>(a.dst[(c + h - 1) % p]) + e * (U / vec_units);
        char *to = static_cast<char *>(a.dst[(c + h) % p]) + e * (U / vec_units);
        if constexpr (U == 16) st_stream_v4(to, ld_coherent_v4(from));
        else if constexpr (U == 4) *reinterpret_cast<uint32_t *>(to) = *reinterpret_cast<const uint32_t *>(from);
        else *reinterpret_cast<uint16_t *>(to) = *reinterpret_cast<const uint16_t *>(from);
    }
}

// ---------------------------------------------------------------------------
// One-phase all-pairs: blockIdx.y is the output rank.
// ---------------------------------------------------------------------------

template <typename T, int OP>
__global__ void __launch_bounds__(kCmpThreads) one_phase_kernel(const __grid_constant__ CmpArgs a)
{
    using Tr = Traits<T>;
    using F = Fold<T, OP>;
    using Acc = typename Tr::Acc;
    constexpr int VEC = Tr::VEC;
    constexpr int S = (VEC == 8) ? 2 : 4;
    const uint64_t tid = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
    const int p = a.p, r = blockIdx.y;
    const uint64_t ngroups = a.vec ? a.n / VEC : 0;
    for (uint64_t g = tid; g < ngroups; g += stride) {
        const uint64_t e = g * VEC;
        const int c = chunk_of<VEC>(a, e, 0);
        Acc acc[VEC];
        for (int k0 = 0; k0 < p; k0 += 8) {
            uint4 rv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (k0 + j < p) rv[j] = ld_coherent_v4(static_cast<const char *>(a.src[a.order[c][k0 + j]]) + e * S);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (k0 + j < p) {
                    Acc v[VEC];
                    Tr::unpack(rv[j], v);
#pragma unroll
                    for (int i = 0; i < VEC; ++i) acc[i] = (k0 + j == 0) ? F::first(v[i], a.scale) : F::fold(acc[i], v[i], a.scale);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < VEC; ++i) acc[i] = F::finish(acc[i], p);
        st_stream_v4(static_cast<char *>(a.dst[r]) + e * S, Tr::pack(acc));
    }
    for (uint64_t e = ngroups * VEC + tid; e < a.n; e += stride) {
        const int c = chunk_of<VEC>(a, e, 0);
        auto acc = F::first(Tr::load1(a.src[a.order[c][0]], e), a.scale);
        for (int k = 1; k < p; ++k) acc = F::fold(acc, Tr::load1(a.src[a.order[c][k]], e), a.scale);
        Tr::store1(a.dst[r], e, F::finish(acc, p));
    }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------

static void fill_args(const Launch &L, CmpArgs &a)
{
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
}

static int cmp_grid(uint64_t units)
{
    uint64_t g = (units + kCmpThreads - 1) / kCmpThreads;
    if (g < 1) g = 1;
    if (g > 0x7fffffff) g = 0x7fffffff;
    return int(g);
}

template <typename T, int OP>
static cudaError_t stepwise_op(const Launch &L, LaunchInfo *info)
{
    constexpr int VEC = Traits<T>::VEC;
    constexpr int S = (VEC == 8) ? 2 : 4;
    CmpArgs a;
    fill_args(L, a);
    const int grid = cmp_grid(L.vec ? L.n / VEC + L.n % VEC : L.n);
    int launched = 0;
    for (int h = 1; h < L.p; ++h) {
        a.hop = h;
        ring_rs_hop_kernel<T, OP><<<grid, kCmpThreads, 0, L.stream>>>(a);
        ++launched;
        cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    for (int h = 1; h < L.p; ++h) {
        a.hop = h;
        if (L.vec) ring_ag_hop_kernel<16><<<cmp_grid(L.n / VEC), kCmpThreads, 0, L.stream>>>(a, VEC);
        else if (S == 2) ring_ag_hop_kernel<2><<<cmp_grid(L.n), kCmpThreads, 0, L.stream>>>(a, 1);
        else ring_ag_hop_kernel<4><<<cmp_grid(L.n), kCmpThreads, 0, L.stream>>>(a, 1);
        ++launched;
        cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    if (info) {
        info->kernel = "allreduce_ring_stepwise";
        info->grid = grid;
        info->block = kCmpThreads;
        info->smem = 0;
        info->kernels = launched;
    }
    return cudaSuccess;
}

template <typename T, int OP>
static cudaError_t one_phase_op(const Launch &L, LaunchInfo *info)
{
    constexpr int VEC = Traits<T>::VEC;
    CmpArgs a;
    fill_args(L, a);
    a.hop = 0;
    const int grid = cmp_grid(L.vec ? L.n / VEC + L.n % VEC : L.n);
    one_phase_kernel<T, OP><<<dim3(grid, L.p), kCmpThreads, 0, L.stream>>>(a);
    if (info) {
        info->kernel = "allreduce_one_phase";
        info->grid = grid * L.p;
        info->block = kCmpThreads;
        info->smem = 0;
        info->kernels = 1;
    }
    return cudaGetLastError();
}

template <typename T>
static cudaError_t compare_dtype(const Launch &L, LaunchInfo *info, bool stepwise)
{
    switch (L.op) {
    case OP_SUM: return stepwise ? stepwise_op<T, OP_SUM>(L, info) : one_phase_op<T, OP_SUM>(L, info);
    case OP_PROD: return stepwise ? stepwise_op<T, OP_PROD>(L, info) : one_phase_op<T, OP_PROD>(L, info);
    case OP_MIN: return stepwise ? stepwise_op<T, OP_MIN>(L, info) : one_phase_op<T, OP_MIN>(L, info);
    case OP_MAX: return stepwise ? stepwise_op<T, OP_MAX>(L, info) : one_phase_op<T, OP_MAX>(L, info);
    case OP_AVG: return stepwise ? stepwise_op<T, OP_AVG>(L, info) : one_phase_op<T, OP_AVG>(L, info);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_compare(const Launch &L, LaunchInfo *info, bool stepwise)
{
    switch (L.dtype) {
    case DT_F32: return compare_dtype<F32>(L, info, stepwise);
    case DT_F16: return compare_dtype<F16>(L, info, stepwise);
    case DT_BF16: return compare_dtype<BF16>(L, info, stepwise);
    default: return compare_dtype<I32>(L, info, stepwise);
    }
}

}  // namespace ccl
