// TMA and TMA bulk-reduce AllReduce / ReduceScatter kernels for i32 rank buffers (see tma.cuh, bulkred.cuh).
#include "bulkred.cuh"

namespace ccl {

cudaError_t launch_tma_i32(const Launch &L, LaunchInfo *info) { return launch_tma<I32>(L, info); }

cudaError_t launch_bulkred_i32(const Launch &L, LaunchInfo *info) { return launch_bulkred<I32>(L, info); }

}  // namespace ccl
