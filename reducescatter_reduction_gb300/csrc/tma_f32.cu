// TMA and TMA bulk-reduce AllReduce / ReduceScatter kernels for f32 rank buffers (see tma.cuh, bulkred.cuh).
#include "bulkred.cuh"

namespace ccl {

cudaError_t launch_tma_f32(const Launch &L, LaunchInfo *info) { return launch_tma<F32>(L, info); }

cudaError_t launch_bulkred_f32(const Launch &L, LaunchInfo *info) { return launch_bulkred<F32>(L, info); }

}  // namespace ccl
