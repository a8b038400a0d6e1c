// Backward grouped GEMMs on token rows: dA (router-weighted, fp16), the gate/up
// recompute with the fused SwiGLU' epilogue, and the input gradient.
#include "gemm.cuh"

namespace moe {
template cudaError_t launch_gemm_kind<GemmKind::DA>(const GemmParams&, int, int, cudaStream_t);
template cudaError_t launch_gemm_kind<GemmKind::BwdGU>(const GemmParams&, int, int, cudaStream_t);
template cudaError_t launch_gemm_kind<GemmKind::Dx>(const GemmParams&, int, int, cudaStream_t);
}  // namespace moe
