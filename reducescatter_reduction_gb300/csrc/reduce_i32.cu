// AllReduce / ReduceScatter kernels for i32 rank buffers (see reduce.cuh).
#include "reduce.cuh"

namespace ccl {

cudaError_t launch_reduce_i32(const Launch &L, LaunchInfo *info)
{
    return L.alias ? launch_reduce_inplace_i32(L, info) : launch_reduce<I32, true>(L, info);
}

}  // namespace ccl
