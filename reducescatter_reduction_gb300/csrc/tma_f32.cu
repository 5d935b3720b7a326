// TMA-variant AllReduce / ReduceScatter kernels for f32 rank buffers (see tma.cuh).
#include "tma.cuh"

namespace ccl {

cudaError_t launch_tma_f32(const Launch &L, LaunchInfo *info) { return launch_tma<F32>(L, info); }

}  // namespace ccl
