// tcgen05 varlen kernel: placeholder until the tensor-core path lands.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
bool varlen_tc_supported(int, int, int) { return false; }
cudaError_t launch_varlen_tc(const VarlenParams&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                             cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace pa
