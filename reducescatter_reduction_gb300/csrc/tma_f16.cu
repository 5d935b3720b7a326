// TMA and TMA bulk-reduce AllReduce / ReduceScatter kernels for f16 rank buffers (see tma.cuh, bulkred.cuh).
#include "bulkred.cuh"

namespace ccl {

cudaError_t launch_tma_f16(const Launch &L, LaunchInfo *info) { return launch_tma<F16>(L, info); }

cudaError_t launch_bulkred_f16(const Launch &L, LaunchInfo *info) { return launch_bulkred<F16>(L, info); }

}  // namespace ccl
