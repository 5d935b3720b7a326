// TMA-variant AllReduce / ReduceScatter kernels for bf16 rank buffers (see tma.cuh).
#include "tma.cuh"

namespace ccl {

cudaError_t launch_tma_bf16(const Launch &L, LaunchInfo *info) { return launch_tma<BF16>(L, info); }

}  // namespace ccl
