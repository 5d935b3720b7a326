// AllReduce / ReduceScatter kernels for bf16 rank buffers (see reduce.cuh).
#include "reduce.cuh"

namespace ccl {

cudaError_t launch_reduce_bf16(const Launch &L, LaunchInfo *info) { return launch_reduce<BF16>(L, info); }

}  // namespace ccl
