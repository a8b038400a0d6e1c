// Backward weight-gradient grouped GEMMs (K = the expert's token rows, fp32 out,
// split experts reduce-added through TMA).
#include "gemm.cuh"

namespace moe {
template cudaError_t launch_gemm_kind<GemmKind::DwGU>(const GemmParams&, int, int, cudaStream_t);
template cudaError_t launch_gemm_kind<GemmKind::DwD>(const GemmParams&, int, int, cudaStream_t);
}  // namespace moe
