// Router step on both sides of the expert-MLP layer.
//
// The pages ("LigerCute -- native CUTLASS + NVSHMEM kernels", LigerMoE design, Forward
// pass) have the final combine apply the router weights; how the weights arise is fixed
// by the workloads: a softmax over all E logits, the K largest (equal values: the lower
// expert index), renormalised over those K; or, for the Llama-4-Scout shape, the sigmoid
// of the single largest logit.  The backward gives the router-weight gradient
// dL/dw[t,k] = <dY[t], f_e(x[t])> from the forward's unweighted expert output y_perm,
// and the logit gradient through the weights.
//
// All three kernels run one warp per token; they are HBM- or latency-bound and small
// next to the expert GEMMs (logits are [T, E] fp32, at most a few MB).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <type_traits>

#include "internal.h"

namespace moe {
namespace {

constexpr int kRouterWarps = 8;            // tokens per 256-thread block
constexpr int kMaxPerLane = kMaxExperts / 32;

// (v, i) beats (w, j): larger value, or equal value and lower index.
__device__ __forceinline__ bool better(float v, int i, float w, int j) {
  return v > w || (v == w && i < j);
}

// Softmax over all E logits, top-K, renormalised == softmax over the K chosen logits
// (the full normaliser cancels); the choice is made on the logits themselves, which
// order exactly as the probabilities do.
template <int kRouter, int kPerLane>
__global__ void __launch_bounds__(32 * kRouterWarps) k_router_topk(
    const float* __restrict__ logits, int T, int E, int K, int32_t* __restrict__ ids,
    float* __restrict__ w) {
  const int t = blockIdx.x * kRouterWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* z = logits + static_cast<size_t>(t) * E;
  float v[kPerLane];   // lane holds logits lane, lane + 32, ... (E <= 32 * kPerLane)
#pragma unroll
  for (int j = 0; j < kPerLane; ++j) {
    const int e = lane + 32 * j;
    v[j] = e < E ? __ldg(z + e) : -INFINITY;
  }
  bool taken[kPerLane];
#pragma unroll
  for (int j = 0; j < kPerLane; ++j) taken[j] = lane + 32 * j >= E;
  float my_val = 0.f;   // lane k keeps the k-th chosen logit and expert
  int my_idx = 0;
  for (int k = 0; k < K; ++k) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
      const int e = lane + 32 * j;
      if (!taken[j] && better(v[j], e, bv, bi)) { bv = v[j]; bi = e; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if ((bi & 31) == lane) {
#pragma unroll
      for (int j = 0; j < kPerLane; ++j)
        if (lane + 32 * j == bi) taken[j] = true;
    }
    if (lane == k) { my_val = bv; my_idx = bi; }
  }
  float wk;
  if (kRouter == 0) {
    const float m = __shfl_sync(0xffffffffu, my_val, 0);   // the largest chosen logit
    const float ex = lane < K ? expf(my_val - m) : 0.f;
    float s = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    wk = ex / s;
  } else {
    wk = 1.0f / (1.0f + expf(-my_val));
  }
  if (lane < K) {
    ids[static_cast<size_t>(t) * K + lane] = my_idx;
    w[static_cast<size_t>(t) * K + lane] = wk;
  }
}

// d_logits: the chosen experts' entries from the weights' gradient, zero elsewhere.
// Softmax router: w = softmax over the chosen logits, so dz_k = w_k (dw_k - <w, dw>).
// Sigmoid router: dz = dw * w * (1 - w).
template <int kRouter>
__global__ void __launch_bounds__(32 * kRouterWarps) k_router_backward(
    const int32_t* __restrict__ ids, const float* __restrict__ w, const float* __restrict__ dw,
    int T, int E, int K, float* __restrict__ dz) {
  const int t = blockIdx.x * kRouterWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  float* row = dz + static_cast<size_t>(t) * E;
  for (int e = lane; e < E; e += 32) row[e] = 0.f;
  const size_t o = static_cast<size_t>(t) * K + lane;
  const float wk = lane < K ? __ldg(w + o) : 0.f;
  const float gk = lane < K ? __ldg(dw + o) : 0.f;
  float g;
  if (kRouter == 0) {
    float s = wk * gk;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    g = wk * (gk - s);
  } else {
    g = gk * wk * (1.0f - wk);
  }
  __syncwarp();
  if (lane < K) row[__ldg(ids + o)] = g;
}

// d_topk_w[t,k] = <dy[t], y_perm[inv[t*K+k]]>: one warp per routed slot streams its
// sorted expert-output row against the token's dY row (read K times, from cache),
// 16-byte loads, two vectors in flight per lane, fp32 sums.
__global__ void __launch_bounds__(32 * kRouterWarps) k_router_weight_grad(
    const uint16_t* __restrict__ dy, const uint16_t* __restrict__ y_perm,
    const int32_t* __restrict__ inv, int T, int K, int D, float* __restrict__ dw) {
  const long long j = static_cast<long long>(blockIdx.x) * kRouterWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (j >= static_cast<long long>(T) * K) return;
  const int t = static_cast<int>(j / K);
  const int nvec = D >> 3;
  const uint4* d = reinterpret_cast<const uint4*>(dy + static_cast<size_t>(t) * D);
  const uint4* y = reinterpret_cast<const uint4*>(y_perm + static_cast<size_t>(__ldg(inv + j)) * D);
  float acc = 0.f;
  for (int vi = lane; vi < nvec; vi += 64) {
    uint4 dq[2], yq[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int v = vi + 32 * h;
      dq[h] = v < nvec ? __ldg(d + v) : make_uint4(0, 0, 0, 0);
      yq[h] = v < nvec ? __ldg(y + v) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __nv_bfloat162* dh = reinterpret_cast<const __nv_bfloat162*>(&dq[h]);
      const __nv_bfloat162* yh = reinterpret_cast<const __nv_bfloat162*>(&yq[h]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 a = __bfloat1622float2(dh[i]);
        const float2 b = __bfloat1622float2(yh[i]);
        acc += a.x * b.x + a.y * b.y;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) dw[j] = acc;
}

}  // namespace

cudaError_t launch_router_topk(const float* logits, int T, int E, int K, int router, int32_t* ids,
                               float* w, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + kRouterWarps - 1) / kRouterWarps;
  LaunchScope ls(kKRouterTopk, s);
  // the fewest logits per lane that hold a row
  auto go = [&](auto per_lane) {
    constexpr int P = decltype(per_lane)::value;
    if (router == 0) k_router_topk<0, P><<<blocks, 32 * kRouterWarps, 0, s>>>(logits, T, E, K, ids, w);
    else k_router_topk<1, P><<<blocks, 32 * kRouterWarps, 0, s>>>(logits, T, E, K, ids, w);
  };
  if (E <= 32) go(std::integral_constant<int, 1>());
  else if (E <= 64) go(std::integral_constant<int, 2>());
  else if (E <= 128) go(std::integral_constant<int, 4>());
  else if (E <= 256) go(std::integral_constant<int, 8>());
  else if (E <= 512) go(std::integral_constant<int, 16>());
  else go(std::integral_constant<int, kMaxPerLane>());
  return cudaGetLastError();
}

cudaError_t launch_router_backward(const int32_t* ids, const float* w, const float* dw, int T,
                                   int E, int K, int router, float* dz, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + kRouterWarps - 1) / kRouterWarps;
  LaunchScope ls(kKRouterBwd, s);
  if (router == 0)
    k_router_backward<0><<<blocks, 32 * kRouterWarps, 0, s>>>(ids, w, dw, T, E, K, dz);
  else
    k_router_backward<1><<<blocks, 32 * kRouterWarps, 0, s>>>(ids, w, dw, T, E, K, dz);
  return cudaGetLastError();
}

cudaError_t launch_router_weight_grad(const uint16_t* dy, const uint16_t* y_perm,
                                      const int32_t* inv, int T, int K, int D, float* dw,
                                      cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const long long slots = static_cast<long long>(T) * K;
  const int blocks = static_cast<int>((slots + kRouterWarps - 1) / kRouterWarps);
  LaunchScope ls(kKRouterWGrad, s);
  k_router_weight_grad<<<blocks, 32 * kRouterWarps, 0, s>>>(dy, y_perm, inv, T, K, D, dw);
  return cudaGetLastError();
}

}  // namespace moe
