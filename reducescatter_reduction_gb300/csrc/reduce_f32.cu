// AllReduce / ReduceScatter kernels for f32 rank buffers (see reduce.cuh).
#include "reduce.cuh"

namespace ccl {

cudaError_t launch_reduce_f32(const Launch &L, LaunchInfo *info)
{
    return L.alias ? launch_reduce_inplace_f32(L, info) : launch_reduce<F32, true>(L, info);
}

}  // namespace ccl
