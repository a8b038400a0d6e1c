// Host-side declarations shared by the translation units of libmoe_gb300.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// Device-side error codes written to the first word of the workspace.
enum DevErr : int {
  kDevOk = 0,
  kDevBadExpertId = 1,      // a topk id outside [0, E)
  kDevTimeoutProducer = 2,  // TMA producer gave up waiting on a free stage
  kDevTimeoutMma = 3,       // MMA issuer gave up waiting on data or TMEM
  kDevTimeoutEpilogue = 4,  // epilogue gave up waiting on an accumulator
  kDevTimeoutRoute = 6,     // the fused routing kernel gave up at a grid barrier
  kDevFp16Range = 7,        // x or dY holds inf / NaN or a magnitude of 2^60 or more, or a
                            // scaled fp16 intermediate of the backward overflowed
};

// Power-of-two scales of the backward's fp16 operands.  The backward first reduces
// max|x| and max|dY| (their fp32 bit patterns, in the workspace header at kMaxAbsOffset);
// with ex = floor(log2 max|x|), ey = floor(log2 max|dY|) (each clamped to [-59, 59]) the
// fp16 tensors hold
//   x16    = x      * 2^(kX16Exp - ex)            dy16 = dY * 2^(kDy16Exp - ey)
//   dA16   = w dA   * 2^(kDAExp - ey)             dH16 = [dG dU] * 2^(kDHExp - ey - ex)
//   wact16 = w act  * 2^(kActExp - 2 ex)
// and the weight-gradient epilogues multiply by the inverse powers.  Multiplying by 2^k
// changes only the exponent, so the scaling itself is exact; it keeps the largest x and
// dY values just below 2^15 and the intermediates (linear in dY; dG, dU also in x; act
// quadratic in x) near 2^8 - 2^10, far from both ends of fp16's range, for max|x| and
// max|dY| anywhere in [2^-59, 2^60).
constexpr int kX16Exp = 14;
constexpr int kDy16Exp = 14;
constexpr int kDAExp = 8;
constexpr int kDHExp = 8;
constexpr int kActExp = 8;
constexpr size_t kMaxAbsOffset = 256;   // two uint32 in the workspace header

// Identifiers of every kernel the library launches (for launch counting and timing).
enum KernelId : int {
  kKRouteCount = 0,
  kKRouteScan,
  kKRouteScatter,
  kKGatherX,
  kKGemmGateUp,
  kKGemmDown,
  kKCombine,
  kKBwdPrepRows,
  kKGemmDA,
  kKGemmBwdGU,
  kKGemmDx,
  kKDwPrep,
  kKGemmDwGU,
  kKGemmDwD,
  kKRouterTopk,
  kKRouterWGrad,
  kKRouterBwd,
  kKRouteFused,
  kKBwdPrepPad,
  kKCombineDx,     // the backward's dX reduction (the combine kernel, run inside the backward)
  kNumKernelIds
};

const char* kernel_name(int id);

// Argument checks shared by the entry points (moe_api.cu).
bool basic_sizes_ok(int T, int K, int E, int align);   // T, K, E, align and the sizes they imply
size_t capacity_of(int T, int K, int E, int align);    // moe_capacity without the checks
bool aligned16(const void* p);
int check_device();   // MOE_OK, MOE_ERR_UNSUPPORTED (not sm_103) or MOE_ERR_CUDA

// Brackets one launch with timing events when timing is on; counts launches.
struct LaunchScope {
  LaunchScope(int id, cudaStream_t s);
  ~LaunchScope();
  int id;
  cudaStream_t stream;
  int slot;
};

// Grouped-GEMM variants (one tcgen05 kernel template, one instantiation each).
enum class GemmKind : int { GateUp = 0, Down = 1, DA = 2, BwdGU = 3, Dx = 4, DwGU = 5, DwD = 6 };

// Tile sizes shared by host and device.
constexpr int kBM = 128;        // token rows (or feature rows for dW) per tile
constexpr int kBK = 64;         // K per pipeline stage (one 128-byte swizzle row of bf16)
// Default dW chunk: an expert with more padded rows than the chunk size is split into equal
// dW chunks of at most that many rows (reduce-added) and gets the compensated
// (value + residual) fp16 operands.  The per-shape tuning may choose another multiple of 64.
constexpr int kDwChunkRows = 4096;
// Experts with more real rows than this take compensated (value + residual) fp16 operands
// in their weight gradients: the error of one fp16 pass grows with the square root of the
// rows summed, and above this count it would approach the tolerance.  Independent of the
// chunking, which only spreads an expert's rows over more tiles.
constexpr int kDwCompRows = 4096;
constexpr int kMaxExperts = 1024;   // largest E the entry points accept

struct GemmParams {
  CUtensorMap mapA0;
  CUtensorMap mapA1;
  CUtensorMap mapB0;
  CUtensorMap mapB1;
  CUtensorMap mapB2;
  CUtensorMap mapB3;
  CUtensorMap mapO0;
  CUtensorMap mapO1;
  CUtensorMap mapO2;
  CUtensorMap mapO3;
  CUtensorMap mapO4;
  const int* offsets;      // [E+1] padded expert offsets (device)
  const int* counts;       // [E] real rows per expert (device) or null: all rows are real
  const int* dw_prefix;    // [E+1] dW split-K chunk prefix over experts (device), dW kinds only
  const float* w_perm;     // [cap] router weight per sorted row (DA, BwdGU)
  const uint16_t* dA;      // [cap, I] router-weighted dA, fp16 (BwdGU reads it)
  const uint16_t* dA_lo;   // [cap, I] its fp16 residual (rows of compensated experts)
  const uint32_t* maxabs;  // backward kinds: {max|x|, max|dY|} as fp32 bits (scales)
  int* err;                // device error word
  int E, D, I;
  int n_tiles;             // N tiles per M tile
  int m_tiles;             // M tiles per expert (dW kinds)
  int tile_n;              // DA: output columns per tile (256, or 128 when I % 256 != 0)
  int order;               // pair kinds: 0 = an expert's tiles row pair by row pair (N tiles
                           // consecutive), 1 = N tile by N tile (row pairs consecutive)
  int swap_tails;          // pair kinds: odd last row tiles computed transposed (else a ghost half)
  int dw_chunk_rows;       // dW split threshold / chunk size (multiple of 64)
  int drop_loads;          // test hook: the producer issues nothing, so the waits expire
};

// Launch one grouped GEMM; `max_tiles` bounds the device-side tile count.
template <GemmKind KIND>
cudaError_t launch_gemm_kind(const GemmParams& p, int max_tiles, int num_sms, cudaStream_t s);

// Route / movement kernels.
cudaError_t launch_route(const int32_t* ids, const float* w, const uint16_t* x, int T, int K,
                         int E, int D, int align, int cap, int32_t* counts, int32_t* offsets,
                         int32_t* perm_src, int32_t* inv_perm, float* w_perm, uint16_t* x_perm,
                         int32_t* chunk_counts, int* err, unsigned* sync, cudaStream_t s);

cudaError_t launch_gather_rows(const uint16_t* src, const int32_t* perm_src, const float* w_perm,
                               const int32_t* offsets, int E, int K, int D, int cap,
                               uint16_t* dst, int kernel_id, cudaStream_t s);

// Backward operand preparation for every sorted row s < offsets[E]:
//   dy_perm[s] = dy[perm_src[s] / K] (bf16, unscaled), dy16[s] = fp16 of the same row
//   scaled by 2^(kDy16Exp - ey), x16[s] = fp16(x[perm_src[s] / K] * 2^(kX16Exp - ex))
//   (from x_perm[s] when x is null); zero rows on padding.
// A first kernel reduces max|x| (x, or x_perm's routed rows) and max|dY| into `maxabs`
// (zeroed here first) and records each routed slot's sorted row in `inv` ([T*K] scratch).
cudaError_t launch_bwd_prep_rows(const uint16_t* dy, const uint16_t* x, const uint16_t* x_perm,
                                 const int32_t* perm_src, const int32_t* offsets, int T, int E,
                                 int K, int D, int cap, int32_t* inv, uint16_t* dy_perm,
                                 uint16_t* dy16, uint16_t* x16, uint32_t* maxabs, int* err,
                                 cudaStream_t s);

cudaError_t launch_combine(const uint16_t* src_perm, const int32_t* inv_perm, const float* w,
                           int T, int K, int D, uint16_t* out, cudaStream_t s,
                           int kernel_id = kKCombine);

cudaError_t launch_dw_prep(const int32_t* offsets, int E, int chunk_rows, int* dw_prefix,
                           float* dw_gate, float* dw_up, float* dw_down, int D, int I,
                           cudaStream_t s);

int route_num_chunks(int R);

// Router step (router: 0 = softmax top-K renormalised, 1 = sigmoid of the top-1 logit).
cudaError_t launch_router_topk(const float* logits, int T, int E, int K, int router, int32_t* ids,
                               float* w, cudaStream_t s);
cudaError_t launch_router_backward(const int32_t* ids, const float* w, const float* dw, int T,
                                   int E, int K, int router, float* dz, cudaStream_t s);
cudaError_t launch_router_weight_grad(const uint16_t* dy, const uint16_t* y_perm,
                                      const int32_t* inv, int T, int K, int D, float* dw,
                                      cudaStream_t s);

}  // namespace moe
