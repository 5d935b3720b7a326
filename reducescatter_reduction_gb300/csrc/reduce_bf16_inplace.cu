// AllReduce / ReduceScatter kernels for bf16 rank buffers whose outputs are
// their inputs (in place): coherent loads (see reduce.cuh, device.cuh).
#include "reduce.cuh"

namespace ccl {

cudaError_t launch_reduce_inplace_bf16(const Launch &L, LaunchInfo *info) { return launch_reduce<BF16, false>(L, info); }

}  // namespace ccl
