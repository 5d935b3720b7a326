// AllReduce / ReduceScatter kernels for f16 rank buffers (see reduce.cuh).
#include "reduce.cuh"

namespace ccl {

cudaError_t launch_reduce_f16(const Launch &L, LaunchInfo *info)
{
    return L.alias ? launch_reduce_inplace_f16(L, info) : launch_reduce<F16, true>(L, info);
}

}  // namespace ccl
