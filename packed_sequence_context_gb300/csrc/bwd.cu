// Backward attention (placeholder until the tcgen05 kernel lands).
#include "common.cuh"
namespace thd {
cudaError_t launch_bwd(const BwdParams&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                       const CUtensorMap&, int, int, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace thd
