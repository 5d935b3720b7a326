// AllReduce / ReduceScatter kernels for bf16 rank buffers (see reduce.cuh).
#include "reduce.cuh"

namespace ccl {

cudaError_t launch_reduce_bf16(const Launch &L, LaunchInfo *info)
{
    return L.alias ? launch_reduce_inplace_bf16(L, info) : launch_reduce<BF16, true>(L, info);
}

}  // namespace ccl
