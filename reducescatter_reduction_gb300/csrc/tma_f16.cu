// TMA-variant AllReduce / ReduceScatter kernels for f16 rank buffers (see tma.cuh).
#include "tma.cuh"

namespace ccl {

cudaError_t launch_tma_f16(const Launch &L, LaunchInfo *info) { return launch_tma<F16>(L, info); }

}  // namespace ccl
