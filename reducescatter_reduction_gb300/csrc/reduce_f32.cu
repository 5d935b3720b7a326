// AllReduce / ReduceScatter kernels for f32 rank buffers (see reduce.cuh).
#include "reduce.cuh"

namespace ccl {

cudaError_t launch_reduce_f32(const Launch &L, LaunchInfo *info) { return launch_reduce<F32>(L, info); }

}  // namespace ccl
