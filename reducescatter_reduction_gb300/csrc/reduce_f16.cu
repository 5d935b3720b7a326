// AllReduce / ReduceScatter kernels for f16 rank buffers (see reduce.cuh).
#include "reduce.cuh"

namespace ccl {

cudaError_t launch_reduce_f16(const Launch &L, LaunchInfo *info) { return launch_reduce<F16>(L, info); }

}  // namespace ccl
