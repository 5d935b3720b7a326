// TMA-variant AllReduce / ReduceScatter kernels for i32 rank buffers (see tma.cuh).
#include "tma.cuh"

namespace ccl {

cudaError_t launch_tma_i32(const Launch &L, LaunchInfo *info) { return launch_tma<I32>(L, info); }

}  // namespace ccl
