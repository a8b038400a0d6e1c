/*
 * moe_gb300.h -- C ABI of libmoe_gb300: the routed Mixture-of-Experts expert-MLP
 * layer (forward and backward) on one NVIDIA GB300 (sm_103a).
 *
 * Source of the method: "LigerCute -- native CUTLASS + NVSHMEM kernels" (the
 * liger-cute-kernels 0.8.3 package README), sections "Overview" and
 * "LigerMoE design" (Forward pass, Backward pass).  The expert MLP is SwiGLU:
 *   f_e(x) = (silu(x W_gate[e]) * (x W_up[e])) W_down[e],  silu(z) = z / (1 + e^-z).
 * The layer output is Y[t] = sum_k topk_w[t,k] * f_{topk_ids[t,k]}(x[t]).
 *
 * Conventions shared by every entry point
 *   - All tensors are dense and row-major.  bf16 tensors are passed as raw 16-bit
 *     storage (moe_bf16_t).  Sizes are element counts.
 *   - Device pointers point to memory of the current CUDA device.  The library
 *     allocates no memory and never synchronises the host (except
 *     moe_get_device_error and moe_timing_collect); every call enqueues its kernels
 *     on `stream` (a cudaStream_t, NULL = legacy default stream) and returns
 *     (moe_expert_mlp_bwd also uses a side stream of its own, joined before it returns).
 *   - The caller owns every buffer.  Buffers must not alias unless stated.
 *   - Arguments are validated on the host before anything is launched; a failed
 *     check returns a negative moe_status_t and launches nothing.  Conditions only
 *     the GPU can see (an expert id outside [0,E), a bounded wait that gave up) are
 *     recorded in the first word of `workspace` and read with moe_get_device_error.
 *   - Notation: T tokens, K experts per token, E experts, D hidden size,
 *     I expert intermediate size, R = T*K routed slots, cap = moe_capacity(T,K,E,align).
 *   - Entry points that run GEMMs (moe_expert_mlp_fwd / _bwd) need D % 256 == 0,
 *     I % 128 == 0 and align % 128 == 0; every pointer they read through TMA must be
 *     16-byte aligned.  Launch shapes depend only on sizes, never on the routing, so
 *     a fixed-size call sequence can be captured once in a CUDA graph and replayed
 *     with new routings.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 5

typedef uint16_t moe_bf16_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,   /* a size, pointer or alignment check failed */
  MOE_ERR_UNSUPPORTED = -2,   /* not an sm_103 device, or a shape the kernels do not cover */
  MOE_ERR_CUDA = -3,          /* a CUDA runtime / driver call failed */
  MOE_ERR_DEVICE_TIMEOUT = -4,/* (device error word) a kernel's bounded wait gave up */
  MOE_ERR_BAD_INDEX = -5,     /* (device error word) an expert id outside [0, E) */
  MOE_ERR_FP16_RANGE = -6     /* (device error word) moe_expert_mlp_bwd met inf / NaN or a
                                 magnitude of 2^60 or more in x or dy, or one of its scaled
                                 fp16 intermediates overflowed (see moe_expert_mlp_bwd) */
} moe_status_t;

/* Version of this ABI (MOE_ABI_VERSION). */
int moe_abi_version(void);

/* Static, human-readable text for a moe_status_t value. */
const char* moe_status_string(int status);

/*
 * Rows of every expert-sorted ("perm") buffer: R + E*(align-1), rounded up to a
 * multiple of `align`.  Sized from the total routed-token count rather than a
 * per-expert capacity ("Overview": symmetric buffers sized from the total
 * routed-token capacity keep execution CUDA-Graph compatible under dynamic
 * routing).  Returns 0 for invalid arguments.
 */
size_t moe_capacity(int T, int K, int E, int align);

/*
 * Bytes of scratch the layer needs: a 1 KB header (device error word), routing
 * chunk counters, the dW split schedule, each routed slot's sorted row [T*K], the
 * activation act [cap, I], the hidden gradient [cap, 2I] (bf16 and fp16), the routed
 * output gradient [cap, D] (bf16 and fp16), an fp16 copy of x_perm [cap, D], fp16
 * residuals of the weight-gradient operands and dA [cap, I] (fp16, with its residual).  One
 * workspace may serve the forward and the backward of the same sizes, but not
 * two calls running concurrently.  Returns 0 for invalid arguments.
 */
size_t moe_workspace_bytes(int T, int K, int E, int D, int I, int align);

/*
 * Zeroes the workspace header (the device error word).  Call once after
 * allocating a workspace.  Asynchronous on `stream`.
 */
int moe_workspace_init(void* workspace, void* stream);

/*
 * Expert sort ("LigerMoE design / Forward pass": routed tokens are sorted by
 * expert before the main loop).  A slot is the flat index j = t*K + k.
 *
 *   topk_ids [T,K] int32 (device)  expert of each slot, in [0, E); a token may repeat an expert
 *   topk_w   [T,K] fp32  (device)  router weight of each slot
 *   x        [T,D] bf16  (device)  token activations; NULL skips the row gather
 * Outputs (device):
 *   counts   [E]     int32  slots per expert
 *   offsets  [E+1]   int32  offsets[0] = 0, offsets[e+1] = offsets[e] + ceil(counts[e]/align)*align
 *   perm_src [cap]   int32  the slot j stored at sorted row s; -1 on padding and beyond offsets[E]
 *   inv_perm [R]     int32  sorted row of slot j (perm_src[inv_perm[j]] == j)
 *   w_perm   [cap]   fp32   router weight at sorted row s; 0 on padding
 *   x_perm   [cap,D] bf16   x[perm_src[s] / K] at sorted row s, zero rows on padding;
 *                           rows at and beyond offsets[E] are not written (ignored if x is NULL)
 * Within an expert, slots keep ascending j, so the result is unique and matches the
 * oracle bit for bit.  Constraints: T >= 0, 1 <= K <= 32, 1 <= E <= 1024, align >= 1,
 * D % 8 == 0 (when x is given), R and cap < 2^31.  Uses the workspace's routing counters.
 */
int moe_route_permute(const int32_t* topk_ids, const float* topk_w, const moe_bf16_t* x,
                      int T, int K, int E, int D, int align,
                      int32_t* counts, int32_t* offsets, int32_t* perm_src, int32_t* inv_perm,
                      float* w_perm, moe_bf16_t* x_perm, void* workspace, void* stream);

/*
 * Expert MLP forward on the sorted rows ("LigerMoE design / Forward pass": the MMA
 * warps execute the expert MLP).  For every row s of expert e (offsets[e] <= s < offsets[e+1]):
 *   act[s]    = bf16( silu(x_perm[s] W_gate[e]) * (x_perm[s] W_up[e]) )   (fp32 accumulate)
 *   y_perm[s] = bf16( act[s] W_down[e] )                                  (fp32 accumulate)
 *   x_perm [cap,D] bf16, w_gate [E,D,I] bf16, w_up [E,D,I] bf16, w_down [E,I,D] bf16,
 *   offsets [E+1] int32 (from moe_route_permute with the same align) -- all device.
 *   counts [E] int32 (device) or NULL: the real rows of each expert (moe_route_permute's
 *   counts).  Rows of expert e at and past offsets[e] + counts[e] are padding; with counts
 *   the GEMMs skip most of the padding of an expert's last row tile.  With NULL every row
 *   below offsets[e+1] is computed (padding rows of x_perm are zero, so they give zero).
 *   y_perm [cap,D] bf16 (device): rows < offsets[E] written; padding rows come out zero.
 * act is kept in the workspace.  Needs D % 256 == 0, I % 128 == 0, align % 128 == 0.
 */
int moe_expert_mlp_fwd(const moe_bf16_t* x_perm, const moe_bf16_t* w_gate,
                       const moe_bf16_t* w_up, const moe_bf16_t* w_down,
                       const int32_t* offsets, const int32_t* counts, int T, int K, int E,
                       int D, int I, int align, moe_bf16_t* y_perm, void* workspace,
                       void* stream);

/*
 * Token combine ("LigerMoE design": the forward's final local combine applies the
 * router weights; the backward's final local dispatch reduces the routed dX back to
 * the original tokens):
 *   out[t] = bf16( sum_k w[t,k] * src_perm[inv_perm[t*K+k]] ),  fp32 sum, k ascending.
 *   src_perm [rows,D] bf16, inv_perm [T*K] int32, topk_w [T,K] fp32 or NULL (weight 1),
 *   out [T,D] bf16 -- all device; out must not alias src_perm.
 * Constraints: T >= 0, 1 <= K <= 32, D % 8 == 0.
 */
int moe_combine(const moe_bf16_t* src_perm, const int32_t* inv_perm, const float* topk_w,
                int T, int K, int D, moe_bf16_t* out, void* stream);

/*
 * Expert MLP backward on the sorted rows ("LigerMoE design / Backward pass"):
 *   1. routed expert-output gradient: the rows dy[perm_src[s] / K] (zero on padding); the
 *      router weight w_perm[s] is applied in fp32 inside step 2
 *   2. recompute G = x_perm W_gate[e], U = x_perm W_up[e]; dA = w_perm[s] * dy_row W_down[e]^T
 *      (fp32, kept in fp16);
 *      dG = dA U silu'(G), dU = dA silu(G)  (bf16 for step 3, fp16 copies for step 4),
 *      and w_perm[s] * silu(G) U (fp16, for step 4)
 *   3. input gradient  dx_perm[s] = bf16( dG[s] W_gate[e]^T + dU[s] W_up[e]^T )
 *   4. weight gradients (fp32), summed over all of the expert's rows:
 *        dw_down[e] = sum_s (w act)_s^T dy_row_s,  dw_gate[e] = x_perm_e^T dG_e,
 *        dw_up[e] = x_perm_e^T dU_e
 *      computed from fp16 operands (x and dy convert exactly; the intermediates keep 10
 *      mantissa bits) with fp32 accumulation; an expert with more than 4096 real rows
 *      also runs the fp16 residuals of the rounded intermediates (compensated operands),
 *      and one with more padded rows than the shape's dW chunk (moe_tuning_t, default
 *      4096) is split over several tiles whose parts are TMA reduce-added.  Experts with
 *      no rows get exactly zero.
 *   Range of the fp16 operands: every fp16 tensor is scaled by a power of two chosen on
 *   the GPU from max|x| and max|dy| (ex, ey = their floor(log2), reduced first in the
 *   workspace): x by 2^(14-ex), dy by 2^(14-ey), w*dA by 2^(8-ey), dG and dU by
 *   2^(8-ey-ex), w*act by 2^(8-2ex); the weight-gradient epilogues multiply by the
 *   inverse powers in fp32.  Scaling by 2^k is exact, so the results do not depend on the
 *   scale of dy (scaling dy by 2^k scales every gradient by exactly 2^k) and fp16's narrow
 *   exponent range costs nothing for max|x|, max|dy| in [2^-59, 2^60).  Reported in the
 *   device error word as MOE_ERR_FP16_RANGE (the results of that call are then not
 *   meaningful): inf / NaN or a magnitude of 2^60 or more in x or dy, and a scaled
 *   intermediate that overflows fp16 (the scales leave about 2^6 of headroom over the
 *   magnitudes of dy, x * dy and x^2 respectively, i.e. weights with row norms up to
 *   about 64).
 *   dy [T,D] bf16, x_perm/perm_src/w_perm/offsets/counts (counts may be NULL) from
 *   moe_route_permute, weights as in the forward -- all device.  x [T,D] bf16 (device) or
 *   NULL: the unsorted input of the forward; when given, step 4's fp16 copy of the sorted
 *   rows is gathered from it (each token row is read K times, mostly from cache) instead
 *   of being read from x_perm.  Outputs (device): dx_perm [cap,D] bf16 (rows < offsets[E]),
 *   dw_gate [E,D,I] fp32, dw_up [E,D,I] fp32, dw_down [E,I,D] fp32 (fully overwritten).
 *   inv_perm [T*K] int32 (moe_route_permute's) and dx [T,D] bf16 (device), both or neither:
 *   when given, the call also reduces dx_perm to tokens, dx = moe_combine(dx_perm,
 *   inv_perm, NULL) bit for bit, beside its weight-gradient GEMMs; when NULL, reduce
 *   dx_perm with moe_combine(dx_perm, inv_perm, NULL, ...) afterwards.
 * Concurrency: with dx given, the dx reduction runs on a second, low-priority stream of
 * the library's own, beside the weight-gradient GEMMs (its blocks share each SM with a GEMM
 * CTA); that stream forks from and joins back into `stream` within the call, so the call
 * behaves as if everything ran on `stream`, also inside a stream capture.  The first such
 * call on a device creates that stream and its events: make it before any capture.
 * Needs D % 256 == 0, I % 128 == 0, align % 128 == 0.
 */
int moe_expert_mlp_bwd(const moe_bf16_t* dy, const moe_bf16_t* x, const moe_bf16_t* x_perm,
                       const int32_t* perm_src,
                       const float* w_perm, const int32_t* offsets, const int32_t* counts,
                       const moe_bf16_t* w_gate, const moe_bf16_t* w_up,
                       const moe_bf16_t* w_down, int T, int K, int E, int D, int I, int align,
                       moe_bf16_t* dx_perm, float* dw_gate, float* dw_up, float* dw_down,
                       const int32_t* inv_perm, moe_bf16_t* dx, void* workspace, void* stream);

/* ---- router step ------------------------------------------------------------
 * The pages have the forward's final combine apply the router weights ("LigerMoE
 * design / Forward pass"); how the weights arise is fixed by the workloads the layer
 * is measured on.  These calls produce the routing that moe_route_permute consumes and
 * the gradients that flow back into the router. */
typedef enum {
  MOE_ROUTER_SOFTMAX_TOPK = 0,  /* softmax over all E logits, the K largest, renormalised */
  MOE_ROUTER_SIGMOID_TOP1 = 1   /* the largest logit's expert, weight sigmoid(logit); K = 1 */
} moe_router_t;

/*
 * For every token t: the K experts of largest logits[t,:] (equal logits: the lower
 * expert index first; slot k = 0 holds the largest), and their weights:
 *   SOFTMAX_TOPK  topk_w[t,k] = softmax(logits[t,:])_{e_k} / sum_j softmax(logits[t,:])_{e_j}
 *                 (= the softmax over the K chosen logits), fp32
 *   SIGMOID_TOP1  topk_w[t,0] = 1 / (1 + exp(-logits[t,e_0]))
 *   logits [T,E] fp32 -> topk_ids [T,K] int32, topk_w [T,K] fp32, all device.
 * Constraints: T >= 0, 1 <= K <= 32, K <= E <= 1024, SIGMOID_TOP1 needs K == 1.
 * The expert choice is made on the fp32 logits exactly (bit-reproducible).
 */
int moe_router_topk(const float* logits, int T, int E, int K, int router, int32_t* topk_ids,
                    float* topk_w, void* stream);

/*
 * Router-weight gradient of L = sum(Y * dY), Y[t] = sum_k topk_w[t,k] f_{e_k}(x[t]):
 *   d_topk_w[t,k] = sum_d dy[t,d] * y_perm[inv_perm[t*K+k], d]     (fp32 sum)
 * where y_perm is moe_expert_mlp_fwd's output (the unweighted expert outputs, in
 * sorted order) and inv_perm moe_route_permute's.  dy [T,D] bf16, y_perm [cap,D] bf16,
 * inv_perm [T*K] int32 -> d_topk_w [T,K] fp32, all device.  D % 8 == 0.
 */
int moe_router_weight_grad(const moe_bf16_t* dy, const moe_bf16_t* y_perm,
                           const int32_t* inv_perm, int T, int K, int D, float* d_topk_w,
                           void* stream);

/*
 * Logit gradient through the router weights (the expert choice is piecewise constant in
 * the logits and contributes nothing):
 *   SOFTMAX_TOPK  d_logits[t,e_k] = w_k (dw_k - sum_j w_j dw_j), zero for unchosen experts
 *   SIGMOID_TOP1  d_logits[t,e_0] = dw_0 w_0 (1 - w_0), zero elsewhere
 *   topk_ids, topk_w from moe_router_topk; d_topk_w [T,K] fp32 -> d_logits [T,E] fp32
 *   (fully overwritten), all device.  Constraints as moe_router_topk.
 */
int moe_router_backward(const int32_t* topk_ids, const float* topk_w, const float* d_topk_w,
                        int T, int E, int K, int router, float* d_logits, void* stream);

/*
 * moe_route_permute without a workspace, for callers that cannot allocate device
 * memory: code that only receives pointers to its tensors (a plugin or operator
 * interface whose host framework owns every allocation), or an engine whose device
 * memory is carved out once up front.  This entry point has no counterpart on the
 * pages the library follows; it is an interface convenience.
 *
 * Arguments, outputs and results are exactly those of moe_route_permute (bit for bit)
 * minus `workspace`.  The per-chunk expert counters live instead in one fixed 1 MiB
 * array inside the library (every GPU that loads the library keeps it until the
 * process exits), so E * ceil(T*K / 256) must not exceed 262144; larger sizes return
 * MOE_ERR_UNSUPPORTED before anything is launched.  Nothing is allocated: no
 * cudaMalloc, cudaFree or allocating library call.
 *
 * Every call looks up the array's device address on the current device (with
 * cudaGetSymbolAddress), so the address stays right across a cudaDeviceReset.  The
 * first call on each device also loads the library's device code; make that first call
 * before any stream capture.  All calls share the one array, whose counters every call
 * rewrites before reading them, so two calls whose kernels overlap on the GPU (different
 * streams, or different host threads) race and corrupt each other's result; serialise
 * them.  Expert ids outside [0, E) are skipped without being reported
 * (moe_route_permute reports them in its workspace's error word).
 */
int moe_route_permute_noalloc(const int32_t* topk_ids, const float* topk_w,
                              const moe_bf16_t* x, int T, int K, int E, int D, int align,
                              int32_t* counts, int32_t* offsets, int32_t* perm_src,
                              int32_t* inv_perm, float* w_perm, moe_bf16_t* x_perm,
                              void* stream);

/*
 * Reads and clears the device error word of `workspace` (synchronises `stream`).
 * *code receives MOE_OK, MOE_ERR_BAD_INDEX, MOE_ERR_FP16_RANGE or MOE_ERR_DEVICE_TIMEOUT;
 * *detail the raw device code (which role timed out).  After an error it also zeroes the rest of the
 * workspace header (counters a kernel that gave up may leave set): call it, or
 * moe_workspace_init, before reusing a workspace after an error.  For tests and debugging.
 */
int moe_get_device_error(void* workspace, int* code, int* detail, void* stream);

/* ---- per-shape tuning -------------------------------------------------------
 * Launch choices of the grouped GEMMs that change their speed, not what they compute
 * (results stay within the same tolerance of the exact values; the tile order changes no
 * bit at all).  A table compiled into the library, written by the package's tuner from
 * measurements on a GB300, picks them per layer shape; shapes it does not hold get the
 * defaults.  The pages rely on tuned per-shape configurations in the same way
 * ("LigerCute -- native CUTLASS + NVSHMEM kernels", the tuned kernel-configuration tables
 * of the grouped GEMMs). */

/* Token-row grouped GEMMs, as indices of moe_tuning_t.order. */
typedef enum {
  MOE_GEMM_GATE_UP = 0,      /* forward gate/up + SwiGLU */
  MOE_GEMM_DOWN = 1,         /* forward down projection */
  MOE_GEMM_DA = 2,           /* backward dA = w * dY W_down^T */
  MOE_GEMM_BWD_GATE_UP = 3,  /* backward gate/up recompute + SwiGLU' */
  MOE_GEMM_DX = 4            /* backward dX */
} moe_tuned_gemm_t;

typedef struct {
  /* Per token-row GEMM: the order of an expert's tiles.  0 (default): row pair by row
   * pair, its N tiles consecutive (they share the token rows); 1: N tile by N tile, its
   * row pairs consecutive (they share each weight tile; pays when an expert's weights are
   * large and it has several 256-row pairs). */
  int order[5];
  /* 1 (default): an expert's odd last 128-row tile is computed transposed, over its real
   * rows only; 0: as half of a 256-row pair whose other half idles. */
  int swap_tails;
  /* dA GEMM output columns per tile: 256 (the default when I % 256 == 0) or 128.  256 on
   * a shape with I % 256 != 0 runs as 128. */
  int da_tile_n;
  /* An expert with more padded rows than this has its weight gradient split into equal
   * chunks of at most this many rows, reduce-added in fp32.  A multiple of 64 in
   * [256, 65536]; default 4096.  (Independently, an expert with more than 4096 real rows
   * takes compensated value + residual fp16 operands in its weight gradients.) */
  int dw_chunk_rows;
} moe_tuning_t;

/*
 * The choices moe_expert_mlp_fwd / moe_expert_mlp_bwd make for this shape.  Host only
 * (needs no GPU).  *source (if not NULL) receives 0 = defaults, 1 = the compiled table
 * (the entry with the same K, E, D, I and the nearest T), 2 = the override.
 * MOE_ERR_INVALID_ARG for a NULL `out` or sizes outside the entry points' ranges.
 */
int moe_tuning_get(int T, int K, int E, int D, int I, moe_tuning_t* out, int* source);

/*
 * Process-wide override: every later moe_expert_mlp_fwd / _bwd call, of any shape, uses
 * `t` until a call with NULL returns to the table.  For tuners and tests.  A value out of
 * range returns MOE_ERR_INVALID_ARG and leaves the previous state.  Calls read the
 * setting once, when they launch: change it only between calls.
 */
int moe_tuning_override(const moe_tuning_t* t);

/* ---- diagnostics ---------------------------------------------------------- */

/*
 * Test hook for the failure path.  Makes the next grouped-GEMM launch of the calling
 * host thread (the gate/up GEMM of the next moe_expert_mlp_fwd) issue no loads.  Its
 * MMA and epilogue warps then wait on barriers nothing completes; each wait gives up
 * after about one second, the kernel lets in-flight work drain, frees its tensor memory
 * and returns, and the workspace error word reads MOE_ERR_DEVICE_TIMEOUT.  Nothing
 * faults, traps or hangs, and the context stays usable.  The outputs of that call are
 * undefined.
 */
int moe_debug_drop_next_loads(void);

/* Number of distinct kernels; kernel ids are 0 .. moe_num_kernels()-1. */
int moe_num_kernels(void);

/* Static name of kernel `id`, or NULL. */
const char* moe_kernel_name(int id);

/* Kernels launched by this library since it was loaded (all ids; per id if counts != NULL,
 * counts has moe_num_kernels() entries). */
long long moe_launch_count(long long* counts);

/*
 * Per-kernel timing.  While enabled, every launch is bracketed by two CUDA events
 * recorded on its own stream.  Not for use inside stream capture.
 */
int moe_timing_enable(int on);

/* The same for the kernels whose bit (1 << id) is set in kernel_mask only (0 = off), so
 * that timing one kernel adds two events per launch of it and nothing elsewhere. */
int moe_timing_enable_mask(unsigned long long kernel_mask);

/* Waits for the recorded events, adds each launch's duration to ms[id] and 1 to
 * launches[id] (arrays of moe_num_kernels() entries, zeroed by the caller), and
 * forgets the records. */
int moe_timing_collect(double* ms, long long* launches);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
