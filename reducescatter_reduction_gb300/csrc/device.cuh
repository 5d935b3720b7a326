// Device-side helpers: 128-bit global loads/stores with cache hints, and the
// per-element-type arithmetic of the reduction (widen to fp32, fold in order,
// round once to the element type).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <atomic>
#include <type_traits>
#include <utility>

#include "internal.h"

namespace ccl {

// ---------------------------------------------------------------------------
// Checked build (compiled with -DCCL_BOUNDS_CHECK; see build.build_checked):
// before each global access a kernel computes, it tests that the access lies
// inside the rank buffer it addresses.  A violation records kBoundsCode, the
// block, the (low 32 bits of the) index and the site in the launch's status
// block -- the first record wins -- and the access is not made.  The host
// reports it as CCL_ERR_BOUNDS.  Nothing traps.  In the default build the
// tests compile away.
// ---------------------------------------------------------------------------
#ifdef CCL_BOUNDS_CHECK
constexpr bool kBoundsCheck = true;
#else
constexpr bool kBoundsCheck = false;
#endif

// Sites named in the record (word 3).
enum BoundsSite : unsigned {
    kSiteReduceGroup = 1,   // ld/st kernel, a 16-byte group
    kSiteReduceElem = 2,    // ld/st kernel, one element
    kSiteTmaLoad = 3,       // TMA kernels, bulk loads of a stage
    kSiteTmaStore = 4,      // TMA kernels, bulk stores of an out tile
    kSiteGather = 5,        // AllGather kernel
    kSiteBulkred = 6,       // bulk-reduce kernel
    kSiteNorm = 7,          // fused AllReduce + residual + RMSNorm
};

__device__ __forceinline__ bool in_bounds(bool ok, unsigned *status, unsigned site, uint64_t index)
{
    if constexpr (!kBoundsCheck) {
        (void)ok;
        (void)status;
        (void)site;
        (void)index;
        return true;
    } else {
        if (ok) return true;
        if (status != nullptr && atomicCAS(&status[0], 0u, kBoundsCode) == 0u) {
            status[1] = blockIdx.x;
            status[2] = unsigned(index);
            status[3] = site;
        }
        return false;
    }
}

// ---------------------------------------------------------------------------
// Memory access.  Inputs are streamed once: read without allocating in L1,
// with a 256-byte L2 prefetch hint.  ld_stream_v4 reads through the
// non-coherent path, which PTX defines only for data that no thread writes
// while the kernel runs: it serves launches where no output overlaps an
// input.  ld_coherent_v4 is the same load without .nc, for in-place launches
// (an output is an input), where each element is read and then written by
// the same thread.  Measured on GB300 (AllReduce p=8/16 bf16, p=5/8 fp32, in
// place and out of place): the two loads run at the same speed within
// 0.05 %; ReduceScatter p=8 bf16 0.2-0.3 % slower with the coherent load.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint4 ld_stream_v4(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ld_coherent_v4(const void *p)
{
    uint4 r;
    asm volatile("ld.global.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p)
                 : "memory");
    return r;
}

// NC: the launch's outputs overlap none of its inputs.
template <bool NC>
__device__ __forceinline__ uint4 ld_in_v4(const void *p)
{
    if constexpr (NC) return ld_stream_v4(p);
    else return ld_coherent_v4(p);
}

__device__ __forceinline__ void st_v4(void *p, const uint4 &v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Keeps a batch of loads in flight: an empty volatile asm that "modifies"
// every loaded register.  Volatile asm statements keep their order, so all of
// the batch's loads are issued before the first value is consumed (without
// it the compiler may interleave each load with its fold and keep only one or
// two loads outstanding).
template <int N>
__device__ __forceinline__ void hold_batch(uint4 (&r)[N])
{
#pragma unroll
    for (int k = 0; k < N; ++k) asm volatile("" : "+r"(r[k].x), "+r"(r[k].y), "+r"(r[k].z), "+r"(r[k].w));
}

// Results are written once and not read again by this kernel: streaming
// (evict-first) stores.  Measured on GB300 with one 16-byte group per
// thread: p=8 bf16 AllReduce 6.86 -> 7.03 TB/s, p=16 6.40 -> 7.05 TB/s.
__device__ __forceinline__ void st_stream_v4(void *p, const uint4 &v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch (sm_90 and later).  A kernel launched with
// launch_dependent may be scheduled while the kernel before it in the stream
// is still draining; before its first global memory access it waits, with
// grid_dependency_wait, until that kernel has completed and its writes are
// visible.  grid_dependents_launch lets the next such kernel be scheduled
// once every CTA of this grid has issued it (or exited); it changes only
// when the next kernel is scheduled, never what it may read.  Both
// instructions do nothing in a kernel launched the ordinary way.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
static cudaError_t launch_dependent(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem,
                                    cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// cudaFuncSetAttribute acts on the kernel as loaded for the current device,
// so a raised dynamic shared-memory limit is set once per device: bit d of
// `done` records device d (a device numbered 64 or more sets it every call).
template <typename... KArgs>
static cudaError_t allow_dynamic_smem(void (*kern)(KArgs...), size_t bytes, int device,
                                      std::atomic<unsigned long long> &done)
{
    const unsigned long long bit = (device >= 0 && device < 64) ? (1ull << device) : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    const cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
    if (err == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return err;
}

// ---------------------------------------------------------------------------
// Element types.  Each traits class gives: the accumulator type, VEC =
// elements per 16 bytes, unpacking a 16-byte vector into VEC accumulator
// values, packing VEC finished values back, and single-element load/store.
// ---------------------------------------------------------------------------

struct F32 {};
struct F16 {};
struct BF16 {};
struct I32 {};

template <typename T> struct Traits;

template <> struct Traits<F32> {
    using Acc = float;
    static constexpr int VEC = 4;
    static constexpr int kDtype = DT_F32;
    __device__ static void unpack(const uint4 &v, float (&f)[VEC])
    {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ static uint4 pack(const float (&f)[VEC])
    {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
    __device__ static float load1(const void *base, uint64_t e)
    {
        return static_cast<const float *>(base)[e];
    }
    __device__ static void store1(void *base, uint64_t e, float v)
    {
        static_cast<float *>(base)[e] = v;
    }
};

// bf16 is the upper half of an fp32 word: widening is a 16-bit shift.
template <> struct Traits<BF16> {
    using Acc = float;
    static constexpr int VEC = 8;
    static constexpr int kDtype = DT_BF16;
    __device__ static void unpack(const uint4 &v, float (&f)[VEC])
    {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static uint32_t pack2(float lo, float hi)
    {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ static uint4 pack(const float (&f)[VEC])
    {
        return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]),
                          pack2(f[6], f[7]));
    }
    __device__ static float load1(const void *base, uint64_t e)
    {
        return __uint_as_float(uint32_t(static_cast<const uint16_t *>(base)[e]) << 16);
    }
    __device__ static void store1(void *base, uint64_t e, float v)
    {
        __nv_bfloat16 h = __float2bfloat16_rn(v);
        static_cast<uint16_t *>(base)[e] = *reinterpret_cast<uint16_t *>(&h);
    }
};

template <> struct Traits<F16> {
    using Acc = float;
    static constexpr int VEC = 8;
    static constexpr int kDtype = DT_F16;
    __device__ static void unpack(const uint4 &v, float (&f)[VEC])
    {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
            float2 t = __half22float2(h);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
    __device__ static uint32_t pack2(float lo, float hi)
    {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ static uint4 pack(const float (&f)[VEC])
    {
        return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]),
                          pack2(f[6], f[7]));
    }
    __device__ static float load1(const void *base, uint64_t e)
    {
        return __half2float(static_cast<const __half *>(base)[e]);
    }
    __device__ static void store1(void *base, uint64_t e, float v)
    {
        static_cast<__half *>(base)[e] = __float2half_rn(v);
    }
};

// int32 accumulates in uint32 so that sum and prod wrap modulo 2^32.
template <> struct Traits<I32> {
    using Acc = uint32_t;
    static constexpr int VEC = 4;
    static constexpr int kDtype = DT_I32;
    __device__ static void unpack(const uint4 &v, uint32_t (&f)[VEC])
    {
        f[0] = v.x;
        f[1] = v.y;
        f[2] = v.z;
        f[3] = v.w;
    }
    __device__ static uint4 pack(const uint32_t (&f)[VEC]) { return make_uint4(f[0], f[1], f[2], f[3]); }
    __device__ static uint32_t load1(const void *base, uint64_t e)
    {
        return static_cast<const uint32_t *>(base)[e];
    }
    __device__ static void store1(void *base, uint64_t e, uint32_t v)
    {
        static_cast<uint32_t *>(base)[e] = v;
    }
};

// ---------------------------------------------------------------------------
// The fold.  `first` turns the first contribution into the accumulator,
// `fold` adds one more (acc = acc (+) v), `finish` produces the stored value.
// Floating point: explicit round-to-nearest intrinsics, so no multiply-add
// is ever contracted; min/max by compare-and-select (earlier operand wins
// ties, exactly as written, not fminf/fmaxf).
// ---------------------------------------------------------------------------

template <int OP> struct FoldF {
    __device__ static __forceinline__ float first(float v, float scale)
    {
        return OP == OP_AVG ? __fmul_rn(v, scale) : v;
    }
    __device__ static __forceinline__ float fold(float acc, float v, float scale)
    {
        if constexpr (OP == OP_SUM) return __fadd_rn(acc, v);
        else if constexpr (OP == OP_AVG) return __fadd_rn(acc, __fmul_rn(v, scale));
        else if constexpr (OP == OP_PROD) return __fmul_rn(acc, v);
        else if constexpr (OP == OP_MIN) return (v < acc) ? v : acc;
        else return (v > acc) ? v : acc;
    }
    __device__ static __forceinline__ float finish(float acc, int) { return acc; }
};

template <int OP> struct FoldI {
    __device__ static __forceinline__ uint32_t first(uint32_t v, float) { return v; }
    __device__ static __forceinline__ uint32_t fold(uint32_t acc, uint32_t v, float)
    {
        if constexpr (OP == OP_SUM || OP == OP_AVG) return acc + v;
        else if constexpr (OP == OP_PROD) return acc * v;
        else if constexpr (OP == OP_MIN) return (int32_t(v) < int32_t(acc)) ? v : acc;
        else return (int32_t(v) > int32_t(acc)) ? v : acc;
    }
    // int avg: the wrapped sum divided once by p, truncating toward zero
    __device__ static __forceinline__ uint32_t finish(uint32_t acc, int p)
    {
        if constexpr (OP == OP_AVG) return uint32_t(int32_t(acc) / p);
        else return acc;
    }
};

template <typename T, int OP>
using Fold = typename std::conditional<std::is_same<T, I32>::value, FoldI<OP>, FoldF<OP>>::type;

// ---------------------------------------------------------------------------
// The fold of one 16-byte group per rank: `first` takes the first rank's
// group, `fold` each later one in order, `finish` returns the packed result.
// In general the lanes are widened to fp32 (or uint32) and folded with Fold.
// ---------------------------------------------------------------------------

template <typename T, int OP, typename Enable = void>
struct GroupFold {
    using Tr = Traits<T>;
    using F = Fold<T, OP>;
    typename Tr::Acc acc[Tr::VEC];

    __device__ __forceinline__ void first(const uint4 &r, float scale)
    {
        typename Tr::Acc v[Tr::VEC];
        Tr::unpack(r, v);
#pragma unroll
        for (int i = 0; i < Tr::VEC; ++i) acc[i] = F::first(v[i], scale);
    }
    __device__ __forceinline__ void fold(const uint4 &r, float scale)
    {
        typename Tr::Acc v[Tr::VEC];
        Tr::unpack(r, v);
#pragma unroll
        for (int i = 0; i < Tr::VEC; ++i) acc[i] = F::fold(acc[i], v[i], scale);
    }
    __device__ __forceinline__ uint4 finish(int p)
    {
#pragma unroll
        for (int i = 0; i < Tr::VEC; ++i) acc[i] = F::finish(acc[i], p);
        return Tr::pack(acc);
    }
};

// min/max of fp16 or bf16: the result is one of the inputs, so no lane needs
// widening or rounding.  Pairs of lanes are compared in place with the
// ordered IEEE comparison (false for NaN; -0 equals +0) and the later rank's
// lane replaces the accumulator's only where it compares strictly less
// (min) or greater (max) -- the operand the fp32 compare-and-select keeps,
// bit for bit, since the widening is exact and preserves order.  Measured on
// GB300 (ld/st AllReduce, fp16 and bf16 alike): p=8 over 64 Mi elements
// 6.04 -> 6.67 TB/s, p=16 over 112 Mi 5.89 -> 6.72 TB/s.  The rest of the
// gap to sum (7.04) is the compare -> select dependency chain, which keeps
// each CTA resident longer with no loads in flight; issuing every load before
// the first compare changed nothing, more CTAs per SM recover part of it at
// p = 8 (reduce_kernel_occ5).
template <typename T> struct Pair16;
template <> struct Pair16<F16> {
    __device__ static __forceinline__ uint32_t lt(uint32_t a, uint32_t b)
    {
        return __hlt2_mask(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&b));
    }
    __device__ static __forceinline__ uint32_t gt(uint32_t a, uint32_t b)
    {
        return __hgt2_mask(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&b));
    }
};
template <> struct Pair16<BF16> {
    __device__ static __forceinline__ uint32_t lt(uint32_t a, uint32_t b)
    {
        return __hlt2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&a), *reinterpret_cast<const __nv_bfloat162 *>(&b));
    }
    __device__ static __forceinline__ uint32_t gt(uint32_t a, uint32_t b)
    {
        return __hgt2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&a), *reinterpret_cast<const __nv_bfloat162 *>(&b));
    }
};

template <typename T, int OP>
constexpr bool kSelect16 = (std::is_same<T, F16>::value || std::is_same<T, BF16>::value) &&
                           (OP == OP_MIN || OP == OP_MAX);

template <typename T, int OP>
struct GroupFold<T, OP, typename std::enable_if<kSelect16<T, OP>>::type> {
    uint32_t w[4];

    __device__ static __forceinline__ uint32_t pick(uint32_t acc, uint32_t v)
    {
        const uint32_t m = OP == OP_MIN ? Pair16<T>::lt(v, acc) : Pair16<T>::gt(v, acc);
        return (v & m) | (acc & ~m);
    }
    __device__ __forceinline__ void first(const uint4 &r, float)
    {
        w[0] = r.x;
        w[1] = r.y;
        w[2] = r.z;
        w[3] = r.w;
    }
    __device__ __forceinline__ void fold(const uint4 &r, float)
    {
        w[0] = pick(w[0], r.x);
        w[1] = pick(w[1], r.y);
        w[2] = pick(w[2], r.z);
        w[3] = pick(w[3], r.w);
    }
    __device__ __forceinline__ uint4 finish(int) { return make_uint4(w[0], w[1], w[2], w[3]); }
};

}  // namespace ccl
