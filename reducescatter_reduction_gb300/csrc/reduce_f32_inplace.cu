// AllReduce / ReduceScatter kernels for f32 rank buffers whose outputs are
// their inputs (in place): coherent loads (see reduce.cuh, device.cuh).
#include "reduce.cuh"

namespace ccl {

cudaError_t launch_reduce_inplace_f32(const Launch &L, LaunchInfo *info) { return launch_reduce<F32, false>(L, info); }

}  // namespace ccl
