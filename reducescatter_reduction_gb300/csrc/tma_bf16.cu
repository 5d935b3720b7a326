// TMA and TMA bulk-reduce AllReduce / ReduceScatter kernels for bf16 rank buffers (see tma.cuh, bulkred.cuh).
#include "bulkred.cuh"

namespace ccl {

cudaError_t launch_tma_bf16(const Launch &L, LaunchInfo *info) { return launch_tma<BF16>(L, info); }

cudaError_t launch_bulkred_bf16(const Launch &L, LaunchInfo *info) { return launch_bulkred<BF16>(L, info); }

}  // namespace ccl
