// AllReduce / ReduceScatter kernels for i32 rank buffers (see reduce.cuh).
#include "reduce.cuh"

namespace ccl {

cudaError_t launch_reduce_i32(const Launch &L, LaunchInfo *info) { return launch_reduce<I32>(L, info); }

}  // namespace ccl
