// Backward kernels (placeholder until the dK/dV and dQ kernels land).
#include "common.cuh"

namespace dma {
cudaError_t launch_bwd(const dma_plan_s&, const dma_bf16*, const dma_bf16*, const float*,
                       const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                       const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, dma_bf16*,
                       float*, float*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace dma
