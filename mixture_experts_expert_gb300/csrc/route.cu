// Routing and data-movement kernels (HBM-bound): expert histogram, prefix scan,
// stable scatter into expert-sorted order, the token-order copies into sorted rows
// (x for the forward; dY and the fp16 dW operands for the backward), the weighted
// combine back to tokens, and the dW split-K preparation.
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kChunk = 256;           // flat routed slots per chunk (one warp each)
constexpr int kRouteWarps = 8;        // warps per block in the count / scatter kernels
constexpr int kPadSlices = 8;         // token-order copies: padding-zeroing blocks per expert

__global__ void k_gather_tokens(const uint16_t* __restrict__ x,
                                const int32_t* __restrict__ perm_src,
                                const int32_t* __restrict__ inv,
                                const int32_t* __restrict__ offsets, int T, int E, int K, int D,
                                int token_blocks, uint16_t* __restrict__ x_perm);

int route_num_chunks(int R) { return (R + kChunk - 1) / kChunk; }

// Per-chunk expert histogram into chunk_counts[e][c]; also marks every sorted row as
// padding (perm_src = -1, w_perm = 0) before the scatter fills the real ones.
__global__ void __launch_bounds__(kRouteWarps * 32) k_route_count(
    const int32_t* __restrict__ ids, int R, int E, int nchunks, int cap,
    int32_t* __restrict__ chunk_counts, int32_t* __restrict__ perm_src,
    float* __restrict__ w_perm, int* err) {
  extern __shared__ int sh_hist[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < cap; i += gridDim.x * blockDim.x) {
    perm_src[i] = -1;
    w_perm[i] = 0.f;
  }
  int* h = sh_hist + warp * E;
  for (int e = lane; e < E; e += 32) h[e] = 0;
  __syncwarp();
  const int c = blockIdx.x * kRouteWarps + warp;
  if (c >= nchunks) return;
  for (int i = lane; i < kChunk; i += 32) {
    const int j = c * kChunk + i;
    if (j < R) {
      const int e = __ldg(ids + j);
      if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) atomicAdd(&h[e], 1);
      else report_error(err, kDevBadExpertId);
    }
  }
  __syncwarp();
  for (int e = lane; e < E; e += 32) chunk_counts[static_cast<size_t>(e) * nchunks + c] = h[e];
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// One warp per expert: exclusive prefix over its chunk counts (in place, giving each
// chunk's first rank inside the expert) and the expert's total count.
__global__ void __launch_bounds__(kRouteWarps * 32) k_route_scan(int E, int nchunks,
                                                               int32_t* __restrict__ chunk_counts,
                                                               int32_t* __restrict__ counts) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouteWarps + warp;
  if (e >= E) return;
  int32_t* row = chunk_counts + static_cast<size_t>(e) * nchunks;
  int running = 0;
  for (int cb = 0; cb < nchunks; cb += 32) {
    const int c = cb + lane;
    const int v = c < nchunks ? row[c] : 0;
    const int incl = warp_incl_scan(v, lane);
    if (c < nchunks) row[c] = running + incl - v;
    running += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) counts[e] = running;
}

// Exclusive scan of the padded expert counts into s_off[0..E] (one block; every thread
// takes part).  Each block of the scatter kernel computes it for itself; block 0 also
// publishes it as `offsets`.
__device__ __forceinline__ void block_padded_offsets(const int32_t* __restrict__ counts, int E,
                                                     int align, int* s_off, int* s_warp) {
  const int nthr = blockDim.x;
  const int per = (E + nthr - 1) / nthr;   // consecutive experts per thread
  const int e0 = threadIdx.x * per;
  int local = 0;
  for (int i = 0; i < per; ++i) {
    const int e = e0 + i;
    if (e < E) local += (__ldg(counts + e) + align - 1) / align * align;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int incl = warp_incl_scan(local, lane);
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = nthr >> 5;
    const int v = lane < nw ? s_warp[lane] : 0;
    s_warp[lane] = warp_incl_scan(v, lane) - v;
  }
  __syncthreads();
  int run = s_warp[warp] + incl - local;
  for (int i = 0; i < per; ++i) {
    const int e = e0 + i;
    if (e < E) {
      s_off[e] = run;
      run += (__ldg(counts + e) + align - 1) / align * align;
    }
  }
  if (threadIdx.x == nthr - 1) s_off[E] = run;
  __syncthreads();
}

// Stable scatter: each warp walks its chunk in slot order; equal experts inside a
// 32-slot step are ranked by lane, and a per-warp running row per expert carries the
// order across steps.  Slot j lands on row offsets[e] + (rank of j among e's slots).
__global__ void __launch_bounds__(kRouteWarps * 32) k_route_scatter(
    const int32_t* __restrict__ ids, const float* __restrict__ w, int R, int E, int nchunks,
    int align, const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ perm_src,
    int32_t* __restrict__ inv_perm, float* __restrict__ w_perm) {
  extern __shared__ int sh_run[];
  __shared__ int s_off[1025];
  __shared__ int s_warp[32];
  block_padded_offsets(counts, E, align, s_off, s_warp);
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = s_off[e];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * kRouteWarps + warp;
  if (c >= nchunks) return;
  int* run = sh_run + warp * E;
  for (int e = lane; e < E; e += 32)
    run[e] = s_off[e] + chunk_base[static_cast<size_t>(e) * nchunks + c];
  __syncwarp();
  const unsigned lt = (1u << lane) - 1u;
  for (int it = 0; it < kChunk / 32; ++it) {
    const int j = c * kChunk + it * 32 + lane;
    int e = j < R ? __ldg(ids + j) : -1;
    if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt);
    const int s = e >= 0 ? run[e] + rank : 0;
    __syncwarp();
    if (e >= 0 && rank == 0) run[e] += __popc(peers);
    __syncwarp();
    if (e >= 0) {
      perm_src[s] = j;
      inv_perm[j] = s;
      w_perm[s] = __ldg(w + j);
    }
  }
}

// ------------------------------------------------------------------ fused routing
// The routing phases in one cooperative launch (every block resident), separated by
// grid barriers: (A) padding marks and per-chunk expert histograms, (B) per-expert scan
// over the chunks, (C) padded offsets and the stable scatter.  One launch instead of
// three saves their launch gaps and tails.  The gather of the token rows stays a
// separate kernel: folded into this launch as a fourth phase it ran slower (measured
// 107 us for the four phases against 24.5 us for these three plus 60 us for the gather).

// Waits until `target` blocks have arrived at *ctr (a counter that only grows during the
// launch).  Bounded: after kWaitLimitNs it records a timeout and returns false.
__device__ __forceinline__ bool grid_barrier(unsigned* ctr, unsigned target, int* err,
                                             int* s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(ctr, 1u);
    int ok = 1;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
      if (v >= target) break;
      __nanosleep(64);   // back off: every block polls the same counter
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        report_error(err, kDevTimeoutRoute);
        ok = 0;
        break;
      }
    }
    __threadfence();
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

__global__ void __launch_bounds__(kRouteWarps * 32) k_route_fused(
    const int32_t* __restrict__ ids, const float* __restrict__ w, int R, int E, int align,
    int nchunks, int cap, int32_t* __restrict__ chunk_counts, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ perm_src,
    int32_t* __restrict__ inv_perm, float* __restrict__ w_perm, unsigned* sync, int* err) {
  extern __shared__ int sh[];          // per warp: E ints (histogram, then running rows)
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_warp[32];
  __shared__ int s_ok;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kRouteWarps + warp;          // global warp
  const int nw = gridDim.x * kRouteWarps;
  const unsigned nb = gridDim.x;
  int* h = sh + warp * E;

  // (A) every sorted row starts as padding; per-chunk histograms
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < cap; i += gridDim.x * blockDim.x) {
    perm_src[i] = -1;
    w_perm[i] = 0.f;
  }
  for (int c = gw; c < nchunks; c += nw) {
    for (int e = lane; e < E; e += 32) h[e] = 0;
    __syncwarp();
    for (int i = lane; i < kChunk; i += 32) {
      const int j = c * kChunk + i;
      if (j < R) {
        const int e = __ldg(ids + j);
        if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) atomicAdd(&h[e], 1);
        else report_error(err, kDevBadExpertId);
      }
    }
    __syncwarp();
    for (int e = lane; e < E; e += 32) chunk_counts[static_cast<size_t>(e) * nchunks + c] = h[e];
    __syncwarp();
  }
  if (!grid_barrier(sync, nb, err, &s_ok)) return;

  // (B) per expert: each chunk's first rank inside the expert, and the expert's count
  for (int e = gw; e < E; e += nw) {
    int32_t* row = chunk_counts + static_cast<size_t>(e) * nchunks;
    int running = 0;
    for (int cb = 0; cb < nchunks; cb += 32) {
      const int c = cb + lane;
      const int v = c < nchunks ? __ldcg(row + c) : 0;   // written by other blocks in (A)
      const int incl = warp_incl_scan(v, lane);
      if (c < nchunks) row[c] = running + incl - v;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) counts[e] = running;
  }
  if (!grid_barrier(sync, 2 * nb, err, &s_ok)) return;

  // (C) padded offsets (every block, from the counts) and the stable scatter
  {
    const int nthr = blockDim.x;
    const int per = (E + nthr - 1) / nthr;
    const int e0 = threadIdx.x * per;
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int e = e0 + i;
      if (e < E) local += (__ldcg(counts + e) + align - 1) / align * align;
    }
    const int incl = warp_incl_scan(local, lane);
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int v = lane < (nthr >> 5) ? s_warp[lane] : 0;
      s_warp[lane] = warp_incl_scan(v, lane) - v;
    }
    __syncthreads();
    int run = s_warp[warp] + incl - local;
    for (int i = 0; i < per; ++i) {
      const int e = e0 + i;
      if (e < E) {
        s_off[e] = run;
        run += (__ldcg(counts + e) + align - 1) / align * align;
      }
    }
    if (threadIdx.x == nthr - 1) s_off[E] = run;
    __syncthreads();
  }
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = s_off[e];
  const unsigned lt = (1u << lane) - 1u;
  for (int c = gw; c < nchunks; c += nw) {
    for (int e = lane; e < E; e += 32)
      h[e] = s_off[e] + __ldcg(chunk_counts + static_cast<size_t>(e) * nchunks + c);
    __syncwarp();
    for (int it = 0; it < kChunk / 32; ++it) {
      const int j = c * kChunk + it * 32 + lane;
      int e = j < R ? __ldg(ids + j) : -1;
      if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) e = -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(peers & lt);
      const int s = e >= 0 ? h[e] + rank : 0;
      __syncwarp();
      if (e >= 0 && rank == 0) h[e] += __popc(peers);
      __syncwarp();
      if (e >= 0) {
        perm_src[s] = j;
        inv_perm[j] = s;
        w_perm[s] = __ldg(w + j);
      }
    }
    __syncwarp();
  }
  // the last block out resets the barrier counter for the next launch
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(sync + 1, 1u) == nb - 1) {
      atomicExch(sync, 0u);
      atomicExch(sync + 1, 0u);
    }
  }
}

cudaError_t launch_route(const int32_t* ids, const float* w, const uint16_t* x, int T, int K,
                         int E, int D, int align, int cap, int32_t* counts, int32_t* offsets,
                         int32_t* perm_src, int32_t* inv_perm, float* w_perm, uint16_t* x_perm,
                         int32_t* chunk_counts, int* err, unsigned* sync, cudaStream_t s) {
  const int R = T * K;
  if (sync != nullptr) {
    // one cooperative launch: a warp per chunk (count, scatter) or per expert (scan),
    // no more blocks than fit on the GPU at once
    const int nch = route_num_chunks(R);
    const size_t shf = static_cast<size_t>(kRouteWarps) * E * sizeof(int);
    static bool configured_fused[64] = {};
    int dev = 0, sms = 0, per_sm = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured_fused[dev]) {
      cudaFuncSetAttribute(k_route_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
      configured_fused[dev] = true;
    }
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_route_fused, kRouteWarps * 32, shf);
    const int resident = (per_sm < 1 ? 1 : per_sm) * (sms < 1 ? 1 : sms);
    const int want = ((nch > E ? nch : E) + kRouteWarps - 1) / kRouteWarps;
    const int blocks = want < 1 ? 1 : (want < resident ? want : resident);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kRouteWarps * 32);
    cfg.dynamicSmemBytes = shf;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    {
      LaunchScope ls(kKRouteFused, s);
      e = cudaLaunchKernelEx(&cfg, k_route_fused, ids, w, R, E, align, nch, cap, chunk_counts,
                             counts, offsets, perm_src, inv_perm, w_perm, sync, err);
    }
    if (e == cudaSuccess && x != nullptr && R > 0) {
      const int token_blocks = (R / K + 7) / 8;
      LaunchScope ls(kKGatherX, s);
      k_gather_tokens<<<token_blocks + E * kPadSlices, 256, 0, s>>>(
          x, perm_src, inv_perm, offsets, R / K, E, K, D, token_blocks, x_perm);
      e = cudaGetLastError();
    }
    return e;
  }
  const int nchunks = route_num_chunks(R);
  const int blocks = nchunks > 0 ? (nchunks + kRouteWarps - 1) / kRouteWarps : 1;
  const size_t sh = static_cast<size_t>(kRouteWarps) * E * sizeof(int);
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaFuncSetAttribute(k_route_count, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
    cudaFuncSetAttribute(k_route_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
    configured[dev] = true;
  }
  {
    LaunchScope ls(kKRouteCount, s);
    k_route_count<<<blocks, kRouteWarps * 32, sh, s>>>(ids, R, E, nchunks, cap, chunk_counts,
                                                       perm_src, w_perm, err);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    LaunchScope ls(kKRouteScan, s);
    k_route_scan<<<(E + kRouteWarps - 1) / kRouteWarps, kRouteWarps * 32, 0, s>>>(
        E, nchunks, chunk_counts, counts);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  {
    // (with no routed slots the scatter still runs one block, to publish the offsets)
    LaunchScope ls(kKRouteScatter, s);
    k_route_scatter<<<blocks, kRouteWarps * 32, sh, s>>>(ids, w, R, E, nchunks, align,
                                                         chunk_counts, counts, offsets,
                                                         perm_src, inv_perm, w_perm);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (x != nullptr && R > 0) {
    e = launch_gather_rows(x, perm_src, nullptr, offsets, E, K, D, cap, x_perm, kKGatherX, s);
  }
  return e;
}

// ------------------------------------------------------------------ row gather
// Token-order copies: each routed token row is read once and written to its K sorted
// rows; blocks past the token blocks zero the padding rows, kPadSlices blocks per expert.

// [*lo, *end): the padding rows of expert e (its real rows come first in its segment).
__device__ __forceinline__ void padding_rows(const int32_t* __restrict__ perm_src,
                                             const int32_t* __restrict__ offsets, int e,
                                             int* lo_out, int* end_out) {
  int lo = __ldg(offsets + e), hi = __ldg(offsets + e + 1);
  *end_out = hi;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(perm_src + mid) >= 0) lo = mid + 1; else hi = mid;
  }
  *lo_out = lo;
}

// Sorted row of slot j held by lane k = j - t*K of the warp of token t, or -1.  An entry
// of a slot that reached no row (an expert id outside [0, E)) is stale, so it counts only
// when perm_src points back at it.
__device__ __forceinline__ int slot_row(const int32_t* __restrict__ inv,
                                        const int32_t* __restrict__ perm_src, int rows, int t,
                                        int K, int lane) {
  if (lane >= K) return -1;
  const int j = t * K + lane;
  const int s = __ldg(inv + j);
  return (s >= 0 && s < rows && __ldg(perm_src + s) == j) ? s : -1;
}

// x_perm[s] = x[t] for every sorted row s of token t; zero padding rows.
__global__ void __launch_bounds__(256) k_gather_tokens(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ perm_src,
    const int32_t* __restrict__ inv, const int32_t* __restrict__ offsets, int T, int E, int K,
    int D, int token_blocks, uint16_t* __restrict__ x_perm) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nvec = D >> 3;
  if (static_cast<int>(blockIdx.x) >= token_blocks) {
    const int b = blockIdx.x - token_blocks;
    const int e = b / kPadSlices, slice = b - e * kPadSlices;
    if (e >= E) return;
    int lo, end;
    padding_rows(perm_src, offsets, e, &lo, &end);
    for (int r = lo + slice * (blockDim.x >> 5) + warp; r < end;
         r += kPadSlices * (blockDim.x >> 5)) {
      uint4* d = reinterpret_cast<uint4*>(x_perm) + static_cast<size_t>(r) * nvec;
      for (int v = lane; v < nvec; v += 32) __stcs(d + v, make_uint4(0, 0, 0, 0));
    }
    return;
  }
  const int rows = __ldg(offsets + E);
  const int wpg = (token_blocks * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += wpg) {
    const int my_s = slot_row(inv, perm_src, rows, t, K, lane);
    if (!__ballot_sync(0xffffffffu, my_s >= 0)) continue;
    const uint4* sp = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * D);
    // warp-uniform trip count: every lane takes part in the shuffles of every step
    for (int vb = 0; vb < nvec; vb += 32 * 8) {
      const int v0 = vb + lane;
      uint4 q[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (v0 + 32 * u < nvec) q[u] = __ldg(sp + v0 + 32 * u);
      for (int k = 0; k < K; ++k) {
        const int s = __shfl_sync(0xffffffffu, my_s, k);
        if (s < 0) continue;   // warp-uniform
        uint4* d = reinterpret_cast<uint4*>(x_perm) + static_cast<size_t>(s) * nvec;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (v0 + 32 * u < nvec) __stcs(d + v0 + 32 * u, q[u]);
      }
    }
  }
}

__device__ __forceinline__ uint4 scale_bf16x8(uint4 q, float sc) {
  uint32_t* w = reinterpret_cast<uint32_t*>(&q);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&w[i]);
    const float2 f = __bfloat1622float2(b);
    w[i] = pack_bf16x2(f.x * sc, f.y * sc);
  }
  return q;
}

// dst[s] = src[perm_src[s] / K] (times w_perm[s] when SCALE), zero on padding rows,
// for s < offsets[E].  One warp per sorted row, 16-byte vectors.
template <bool SCALE>
__global__ void __launch_bounds__(256) k_gather_rows(const uint16_t* __restrict__ src,
                                                     const int32_t* __restrict__ perm_src,
                                                     const float* __restrict__ w_perm,
                                                     const int32_t* __restrict__ offsets, int E,
                                                     int K, int D, uint16_t* __restrict__ dst) {
  const int rows = __ldg(offsets + E);
  const int lane = threadIdx.x & 31;
  const int nvec = D >> 3;
  const int wpg = (gridDim.x * blockDim.x) >> 5;
  for (int s = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; s < rows; s += wpg) {
    const int j = __ldg(perm_src + s);
    uint4* d = reinterpret_cast<uint4*>(dst + static_cast<size_t>(s) * D);
    // the sorted rows are written once and not read again here: streaming stores keep
    // them from evicting the token rows, which K slots each read from cache
    if (j < 0) {
      for (int v = lane; v < nvec; v += 32) __stcs(d + v, make_uint4(0, 0, 0, 0));
      continue;
    }
    const uint4* sp = reinterpret_cast<const uint4*>(src + static_cast<size_t>(j / K) * D);
    const float sc = SCALE ? __ldg(w_perm + s) : 1.0f;
    int v = lane;
    for (; v + 96 < nvec; v += 128) {
      uint4 q0 = __ldg(sp + v), q1 = __ldg(sp + v + 32), q2 = __ldg(sp + v + 64),
            q3 = __ldg(sp + v + 96);
      if (SCALE) {
        q0 = scale_bf16x8(q0, sc); q1 = scale_bf16x8(q1, sc);
        q2 = scale_bf16x8(q2, sc); q3 = scale_bf16x8(q3, sc);
      }
      __stcs(d + v, q0); __stcs(d + v + 32, q1); __stcs(d + v + 64, q2); __stcs(d + v + 96, q3);
    }
    for (; v < nvec; v += 32) {
      uint4 q = __ldg(sp + v);
      if (SCALE) q = scale_bf16x8(q, sc);
      __stcs(d + v, q);
    }
  }
}

cudaError_t launch_gather_rows(const uint16_t* src, const int32_t* perm_src, const float* w_perm,
                               const int32_t* offsets, int E, int K, int D, int cap,
                               uint16_t* dst, int kernel_id, cudaStream_t s) {
  int blocks = (cap + 7) / 8;
  if (blocks < 1) blocks = 1;
  LaunchScope ls(kernel_id, s);
  if (w_perm) k_gather_rows<true><<<blocks, 256, 0, s>>>(src, perm_src, w_perm, offsets, E, K, D, dst);
  else k_gather_rows<false><<<blocks, 256, 0, s>>>(src, perm_src, nullptr, offsets, E, K, D, dst);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ backward row prep
// fp16 copy of eight bf16 values times 2^k (f = 2^k, exact: only the exponent moves).
__device__ __forceinline__ uint4 bf16x8_to_f16x8_scaled(uint4 q, float f) {
  uint32_t* w = reinterpret_cast<uint32_t*>(&q);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w[i]));
    w[i] = pack_f16x2(v.x * f, v.y * f);
  }
  return q;
}

// Largest magnitude among eight bf16 values, as bf16 bits in both halves of the result
// (non-negative bf16 bit patterns order like their values).
__device__ __forceinline__ uint32_t bf16x8_absmax_bits(uint4 q, uint32_t m) {
  m = __vmaxu2(m, q.x & 0x7fff7fffu);
  m = __vmaxu2(m, q.y & 0x7fff7fffu);
  m = __vmaxu2(m, q.z & 0x7fff7fffu);
  m = __vmaxu2(m, q.w & 0x7fff7fffu);
  return m;
}

// max over both 16-bit halves, widened to the fp32 bit pattern of the same value
__device__ __forceinline__ uint32_t bf16_pair_max_to_f32_bits(uint32_t m2) {
  const uint32_t a = m2 & 0xffffu, b = m2 >> 16;
  return (a > b ? a : b) << 16;
}

// Block-wide max of v (every thread of the block calls it), then one atomicMax.
__device__ __forceinline__ void block_atomic_max(uint32_t v, uint32_t* dst, uint32_t* s_red) {
  v = __reduce_max_sync(0xffffffffu, v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < static_cast<int>(blockDim.x >> 5) ? s_red[lane] : 0u;
    w = __reduce_max_sync(0xffffffffu, w);
    if (lane == 0 && w != 0u) atomicMax(dst, w);
  }
  __syncthreads();
}

// Two kernels.  The first records each routed slot's sorted row (inv[j] = s; a slot that
// reached no row, an expert id outside [0, E), keeps whatever its entry held, so the second
// kernel accepts inv[j] = s only when perm_src[s] == j) and reduces max|x| (x, or the routed
// rows of x_perm when x is not given) and max|dY| into maxabs[0], maxabs[1] (fp32 bits;
// zeroed before the launch).  Inputs with inf / NaN or a magnitude of 2^60 or more are
// reported: the scales cover finite magnitudes below 2^60.
// In the second, one warp per token reads the token's dY and x rows once and writes them
// to its K sorted rows: dy_perm[s] = dy[t] (bf16), dy16[s] = fp16(dy[t] * 2^(kDy16Exp - ey)),
// x16[s] = fp16(x[t] * 2^(kX16Exp - ex)) (from the sorted copy of the row when x is not
// given); its last E * kPadSlices blocks zero the three copies' padding rows.  In sorted
// order the token rows would be re-read K times, mostly from DRAM once the copies being
// written have pushed them out of L2.
__global__ void __launch_bounds__(256) k_bwd_prep_pad(const int32_t* __restrict__ perm_src,
                                                      const int32_t* __restrict__ offsets, int E,
                                                      int32_t* __restrict__ inv,
                                                      const uint16_t* __restrict__ x,
                                                      const uint16_t* __restrict__ x_perm,
                                                      const uint16_t* __restrict__ dy, int T,
                                                      int D, uint32_t* maxabs, int* err) {
  __shared__ uint32_t s_red[32];
  const int rows = __ldg(offsets + E);
  const int gtid = blockIdx.x * blockDim.x + threadIdx.x;
  const int gthreads = gridDim.x * blockDim.x;
  for (int s = gtid; s < rows; s += gthreads) {
    const int j = __ldg(perm_src + s);
    if (j >= 0) inv[j] = s;
  }
  const size_t nvec_y = static_cast<size_t>(T) * D / 8;
  const size_t nvec_x = x ? nvec_y : static_cast<size_t>(rows) * D / 8;
  const uint4* px = reinterpret_cast<const uint4*>(x ? x : x_perm);
  const uint4* py = reinterpret_cast<const uint4*>(dy);
  uint32_t mx = 0, my = 0;
  // four independent 16-byte loads in flight per thread and step
  const size_t step = static_cast<size_t>(gthreads);
  size_t v = gtid;
  for (; v + 3 * step < nvec_x; v += 4 * step) {
    const uint4 a = __ldg(px + v), b = __ldg(px + v + step), c = __ldg(px + v + 2 * step),
                d = __ldg(px + v + 3 * step);
    mx = bf16x8_absmax_bits(d, bf16x8_absmax_bits(c, bf16x8_absmax_bits(b,
             bf16x8_absmax_bits(a, mx))));
  }
  for (; v < nvec_x; v += step) mx = bf16x8_absmax_bits(__ldg(px + v), mx);
  v = gtid;
  for (; v + 3 * step < nvec_y; v += 4 * step) {
    const uint4 a = __ldg(py + v), b = __ldg(py + v + step), c = __ldg(py + v + 2 * step),
                d = __ldg(py + v + 3 * step);
    my = bf16x8_absmax_bits(d, bf16x8_absmax_bits(c, bf16x8_absmax_bits(b,
             bf16x8_absmax_bits(a, my))));
  }
  for (; v < nvec_y; v += step) my = bf16x8_absmax_bits(__ldg(py + v), my);
  mx = bf16_pair_max_to_f32_bits(mx);
  my = bf16_pair_max_to_f32_bits(my);
  // 2^60 = 0x5d800000: inf / NaN and magnitudes beyond the scales' range
  if (mx >= 0x5d800000u || my >= 0x5d800000u) report_error(err, kDevFp16Range);
  block_atomic_max(mx, maxabs, s_red);
  block_atomic_max(my, maxabs + 1, s_red);
}

__global__ void __launch_bounds__(256) k_bwd_prep_rows(
    const uint16_t* __restrict__ dy, const uint16_t* __restrict__ x,
    const uint16_t* __restrict__ x_perm, const int32_t* __restrict__ perm_src,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ inv, int T, int E, int K,
    int D, int token_blocks, uint16_t* __restrict__ dy_perm, uint16_t* __restrict__ dy16,
    uint16_t* __restrict__ x16, const uint32_t* __restrict__ maxabs) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nvec = D >> 3;
  if (static_cast<int>(blockIdx.x) >= token_blocks) {
    // padding rows of expert e: its real rows come first in its segment
    const int b = blockIdx.x - token_blocks;
    const int e = b / kPadSlices, slice = b - e * kPadSlices;
    if (e >= E) return;
    int lo, end;
    padding_rows(perm_src, offsets, e, &lo, &end);
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int r = lo + slice * (blockDim.x >> 5) + warp; r < end;
         r += kPadSlices * (blockDim.x >> 5)) {
      const size_t off = static_cast<size_t>(r) * nvec;
      uint4* dp = reinterpret_cast<uint4*>(dy_perm) + off;
      uint4* d16 = reinterpret_cast<uint4*>(dy16) + off;
      uint4* x16p = reinterpret_cast<uint4*>(x16) + off;
      for (int v = lane; v < nvec; v += 32) {
        __stcs(dp + v, z);
        __stcs(d16 + v, z);
        __stcs(x16p + v, z);
      }
    }
    return;
  }
  const int wpg = (token_blocks * blockDim.x) >> 5;
  const int rows = __ldg(offsets + E);
  const BwdExps sc = load_bwd_exps(maxabs);
  const float fx = pow2f(kX16Exp - sc.ex), fy = pow2f(kDy16Exp - sc.ey);
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += wpg) {
    const int my_s = slot_row(inv, perm_src, rows, t, K, lane);   // lane k: slot (t, k)
    const unsigned valid = __ballot_sync(0xffffffffu, my_s >= 0);
    if (!valid) continue;
    const int s_first = __shfl_sync(0xffffffffu, my_s, __ffs(valid) - 1);
    const uint4* sp = reinterpret_cast<const uint4*>(dy + static_cast<size_t>(t) * D);
    const uint4* xp = reinterpret_cast<const uint4*>(
        x ? x + static_cast<size_t>(t) * D : x_perm + static_cast<size_t>(s_first) * D);
    // warp-uniform trip count: every lane takes part in the shuffles of every step
    for (int vb = 0; vb < nvec; vb += 32 * 4) {
      const int v0 = vb + lane;
      uint4 q[4], h[4], xh[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = v0 + 32 * u;
        if (v < nvec) {
          q[u] = __ldg(sp + v);
          xh[u] = bf16x8_to_f16x8_scaled(__ldg(xp + v), fx);
          h[u] = bf16x8_to_f16x8_scaled(q[u], fy);
        }
      }
      for (int k = 0; k < K; ++k) {
        const int s = __shfl_sync(0xffffffffu, my_s, k);
        if (s < 0) continue;   // warp-uniform
        const size_t off = static_cast<size_t>(s) * nvec;
        uint4* dp = reinterpret_cast<uint4*>(dy_perm) + off;
        uint4* d16 = reinterpret_cast<uint4*>(dy16) + off;
        uint4* x16p = reinterpret_cast<uint4*>(x16) + off;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int v = v0 + 32 * u;
          if (v < nvec) {
            __stcs(dp + v, q[u]);   // streaming stores: written once, read by later kernels
            __stcs(d16 + v, h[u]);
            __stcs(x16p + v, xh[u]);
          }
        }
      }
    }
  }
}

cudaError_t launch_bwd_prep_rows(const uint16_t* dy, const uint16_t* x, const uint16_t* x_perm,
                                 const int32_t* perm_src, const int32_t* offsets, int T, int E,
                                 int K, int D, int cap, int32_t* inv, uint16_t* dy_perm,
                                 uint16_t* dy16, uint16_t* x16, uint32_t* maxabs, int* err,
                                 cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(maxabs, 0, 2 * sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  if (T > 0) {
    // enough blocks to stream x and dY (T * D values each) at full bandwidth: about four
    // 16-byte vectors per thread and tensor, at most 2048 blocks
    const long long vec = static_cast<long long>(T) * D / 8;
    long long want = (vec + 1023) / 1024;
    const long long rows_blocks = (static_cast<long long>(cap) + 255) / 256;
    if (rows_blocks > want) want = rows_blocks;
    const int blocks = static_cast<int>(want < 1 ? 1 : (want > 2048 ? 2048 : want));
    LaunchScope ls(kKBwdPrepPad, s);
    k_bwd_prep_pad<<<blocks, 256, 0, s>>>(perm_src, offsets, E, inv, x, x_perm, dy, T, D, maxabs,
                                          err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int token_blocks = (T + 7) / 8;
  LaunchScope ls(kKBwdPrepRows, s);
  k_bwd_prep_rows<<<token_blocks + E * kPadSlices, 256, 0, s>>>(
      dy, x, x_perm, perm_src, offsets, inv, T, E, K, D, token_blocks, dy_perm, dy16, x16,
      maxabs);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ combine
// out[t] = sum_k w[t,k] * src[inv[t*K+k]] in fp32, k ascending, one warp per token.
__global__ void __launch_bounds__(256) k_combine(const uint16_t* __restrict__ src,
                                                 const int32_t* __restrict__ inv,
                                                 const float* __restrict__ w, int T, int K,
                                                 int D, uint16_t* __restrict__ out) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int my_row = lane < K ? __ldg(inv + static_cast<size_t>(t) * K + lane) : 0;
  const float my_w = lane < K ? (w ? __ldg(w + static_cast<size_t>(t) * K + lane) : 1.0f) : 0.f;
  const int nvec = D >> 3;
  uint4* o = reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * D);
  // warp-uniform trip count: every lane takes part in the shuffles of every step; two
  // vector columns per step keep 2 x 8 row loads in flight per lane
  for (int vb = 0; vb < nvec; vb += 64) {
    int vv[2];
    bool act[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      vv[h] = vb + 32 * h + lane;
      act[h] = vv[h] < nvec;
    }
    float acc[2][8];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[h][i] = 0.f;
    for (int k0 = 0; k0 < K; k0 += 8) {
      uint4 q[2][8];
      float wk[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int k = k0 + u;
        const int row = __shfl_sync(0xffffffffu, my_row, k & 31);
        wk[u] = __shfl_sync(0xffffffffu, my_w, k & 31);
        const uint4* rp = reinterpret_cast<const uint4*>(src + static_cast<size_t>(row) * D);
#pragma unroll
        for (int h = 0; h < 2; ++h)
          q[h][u] = (act[h] && k < K) ? __ldcs(rp + vv[h]) : make_uint4(0, 0, 0, 0);   // read once
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (k0 + u >= K) break;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t* qw = reinterpret_cast<const uint32_t*>(&q[h][u]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qw[i]));
            acc[h][2 * i] = fmaf(wk[u], f.x, acc[h][2 * i]);
            acc[h][2 * i + 1] = fmaf(wk[u], f.y, acc[h][2 * i + 1]);
          }
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
      if (act[h])
        o[vv[h]] = make_uint4(pack_bf16x2(acc[h][0], acc[h][1]), pack_bf16x2(acc[h][2], acc[h][3]),
                              pack_bf16x2(acc[h][4], acc[h][5]), pack_bf16x2(acc[h][6], acc[h][7]));
  }
}

cudaError_t launch_combine(const uint16_t* src_perm, const int32_t* inv_perm, const float* w,
                           int T, int K, int D, uint16_t* out, cudaStream_t s, int kernel_id) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + 7) / 8;
  LaunchScope ls(kernel_id, s);
  k_combine<<<blocks, 256, 0, s>>>(src_perm, inv_perm, w, T, K, D, out);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ dW split-K preparation
// Block (0,0) writes dw_prefix[e] = sum_{e' < e} chunks(e'), chunks(e) = max(1, ceil(rows_e / chunk)).
// Block e zeroes dW[e] when expert e is split (its tiles reduce-add into it).
__global__ void __launch_bounds__(256) k_dw_prep(const int32_t* __restrict__ offsets, int E,
                                                 int chunk, int* __restrict__ dw_prefix,
                                                 float* __restrict__ dwg,
                                                 float* __restrict__ dwu,
                                                 float* __restrict__ dwd, int D, int I) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    // chunks(e) = max(1, ceil(rows_e / chunk)); each thread sums a run of experts
    __shared__ int s_warp[32];
    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int e0 = threadIdx.x * per;
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int e = e0 + i;
      if (e < E) {
        const int rows = __ldg(offsets + e + 1) - __ldg(offsets + e);
        const int ch = (rows + chunk - 1) / chunk;
        local += ch < 1 ? 1 : ch;
      }
    }
    const int incl = warp_incl_scan(local, lane);
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int v = lane < static_cast<int>(blockDim.x >> 5) ? s_warp[lane] : 0;
      s_warp[lane] = warp_incl_scan(v, lane) - v;
    }
    __syncthreads();
    int run = s_warp[warp] + incl - local;
    for (int i = 0; i < per; ++i) {
      const int e = e0 + i;
      if (e < E) {
        dw_prefix[e] = run;
        const int rows = __ldg(offsets + e + 1) - __ldg(offsets + e);
        const int ch = (rows + chunk - 1) / chunk;
        run += ch < 1 ? 1 : ch;
      }
    }
    if (threadIdx.x == blockDim.x - 1) dw_prefix[E] = run;
  }
  const int e = blockIdx.x;
  if (e >= E) return;
  const int rows = __ldg(offsets + e + 1) - __ldg(offsets + e);
  if (rows <= chunk) return;
  // a split expert's three dW tensors are zeroed by gridDim.y blocks, one slice each
  const size_t n4 = static_cast<size_t>(D) * I / 4;
  float4* g4 = reinterpret_cast<float4*>(dwg + static_cast<size_t>(e) * D * I);
  float4* u4 = reinterpret_cast<float4*>(dwu + static_cast<size_t>(e) * D * I);
  float4* d4 = reinterpret_cast<float4*>(dwd + static_cast<size_t>(e) * D * I);
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  const size_t step = static_cast<size_t>(blockDim.x) * gridDim.y;
  for (size_t i = static_cast<size_t>(blockIdx.y) * blockDim.x + threadIdx.x; i < n4; i += step) {
    g4[i] = z;
    u4[i] = z;
    d4[i] = z;
  }
}

cudaError_t launch_dw_prep(const int32_t* offsets, int E, int chunk_rows, int* dw_prefix,
                           float* dw_gate, float* dw_up, float* dw_down, int D, int I,
                           cudaStream_t s) {
  LaunchScope ls(kKDwPrep, s);
  // ~2048 blocks in all, so that one split expert's zeroing still spans the GPU while a
  // launch with no split expert stays cheap
  const int slices = E >= 2048 ? 1 : 2048 / E;
  k_dw_prep<<<dim3(E, slices), 256, 0, s>>>(offsets, E, chunk_rows, dw_prefix, dw_gate, dw_up,
                                             dw_down, D, I);
  return cudaGetLastError();
}

}  // namespace moe

// ------------------------------------------------------------------ routing without a workspace
// moe_route_permute needs a caller-provided workspace for its per-chunk expert counters.
// Some callers have no way to obtain device memory for it: code that only receives
// pointers to its tensors (a plugin or operator ABI whose host framework owns every
// allocation), or an engine whose device memory is carved out once up front and may not
// grow afterwards.  moe_route_permute_noalloc serves them: its counters live in a
// fixed array compiled into this library, so the caller passes only inputs and outputs.
#include "moe_gb300.h"

namespace moe {
namespace {

// 1 MiB: the chunk counters need E * ceil(T*K / 256) ints.
constexpr int kNoAllocScratchInts = 1 << 18;
static __device__ __align__(256) int32_t g_route_scratch[kNoAllocScratchInts];

// Host code cannot use g_route_scratch's name as a device pointer: its device address is
// looked up on the current device at every call (cheap once the library's device code is
// loaded), so that a context torn down and made again (cudaDeviceReset) never leaves a
// stale address behind.
int32_t* noalloc_scratch_for_current_device(cudaError_t* err) {
  void* p = nullptr;
  *err = cudaGetSymbolAddress(&p, g_route_scratch);
  return *err == cudaSuccess ? static_cast<int32_t*>(p) : nullptr;
}

}  // namespace
}  // namespace moe

extern "C" __attribute__((visibility("default"))) int moe_route_permute_noalloc(
    const int32_t* topk_ids, const float* topk_w, const uint16_t* x, int T, int K, int E, int D,
    int align, int32_t* counts, int32_t* offsets, int32_t* perm_src, int32_t* inv_perm,
    float* w_perm, uint16_t* x_perm, void* stream) {
  using namespace moe;
  // the same argument rules as moe_route_permute (minus the workspace)
  if (!basic_sizes_ok(T, K, E, align)) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets || !perm_src || !w_perm) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_ids || !topk_w || !inv_perm)) return MOE_ERR_INVALID_ARG;
  if (x && (!x_perm || D <= 0 || D % 8 != 0 || !aligned16(x) || !aligned16(x_perm)))
    return MOE_ERR_INVALID_ARG;
  // the counters must fit the fixed array
  const long long need = static_cast<long long>(E) * route_num_chunks(T * K);
  if (need > kNoAllocScratchInts) return MOE_ERR_UNSUPPORTED;
  const int st = check_device();
  if (st != MOE_OK) return st;
  cudaError_t e = cudaSuccess;
  int32_t* scratch = noalloc_scratch_for_current_device(&e);
  if (!scratch) return MOE_ERR_CUDA;
  // every chunk counter is rewritten by each call before it is read, so nothing needs
  // clearing; expert ids outside [0, E) are skipped without being reported (no error slot)
  e = launch_route(topk_ids, topk_w, x, T, K, E, D, align,
                   static_cast<int>(capacity_of(T, K, E, align)), counts, offsets, perm_src,
                   inv_perm, w_perm, x_perm, scratch, nullptr, nullptr,
                   static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
