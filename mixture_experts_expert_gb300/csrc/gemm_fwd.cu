// Forward grouped GEMMs: gate/up projection with the fused SwiGLU epilogue, and the
// down projection.
#include "gemm.cuh"

namespace moe {
template cudaError_t launch_gemm_kind<GemmKind::GateUp>(const GemmParams&, int, int, cudaStream_t);
template cudaError_t launch_gemm_kind<GemmKind::Down>(const GemmParams&, int, int, cudaStream_t);
}  // namespace moe
