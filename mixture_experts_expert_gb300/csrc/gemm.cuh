// Persistent, warp-specialised grouped GEMM for the MoE expert MLP on sm_103a.
//
// One CTA per SM, 192 threads:
//   warp 0      TMA producer (lane 0 issues cp.async.bulk.tensor into a ring of 48 KB stages)
//   warp 1      TMEM owner + MMA issuer (lane 0 issues tcgen05.mma, M = 128, fp32 accumulators
//               in two 256-column TMEM buffers, so one tile's epilogue overlaps the next
//               tile's MMAs)
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM lanes
//               32*(w%4)..+31), fused elementwise math, tile stores or reduce-adds through a
//               swizzled shared-memory ring and TMA.
//
// Tiles are scheduled statically (tile = blockIdx.x + i*gridDim.x) over a tile space
// whose size is read on the device from the expert offsets, so the launch is
// independent of the routing (no host sync; valid inside a captured CUDA graph).
//
// Kinds (row-major; "perm" rows are expert-sorted, padded to 128 rows per expert):
//   GateUp  act[s, i]  = silu(x_perm[s] W_g[e])_i * (x_perm[s] W_u[e])_i   N: 128 gate + 128 up
//   Down    y_perm[s]  = act[s] W_d[e]
//   DA      dA[s]      = w_perm[s] * dy_perm[s] W_d[e]^T        (fp32 out; dy_perm unscaled)
//   BwdGU   recompute G, U as GateUp; the epilogue reads dA and writes w*act (fp16),
//           dG = dA U silu'(G), dU = dA silu(G) (bf16 for Dx, fp16 for the dW GEMMs) and,
//           for experts split over several dW tiles, the fp16 residuals v - fp16(v)
//   Dx      dx_perm[s] = [dG dU][s] [W_g[e]; W_u[e]]^T                    (K = 2I)
//   DwGU    [dW_g dW_u][e] = x16_e^T [dG dU]16_e        (K = the expert's token rows)
//   DwD     dW_d[e]        = (w act)16_e^T dy16_e
// The weight-gradient GEMMs sum over up to thousands of token rows, so their operands
// are fp16 (10-bit mantissa; x and dY convert exactly) rather than bf16: the rounding of
// the intermediates (dG, dU, w*act) is what bounds dW's absolute error.  dW tiles cover
// at most kDwChunkRows token rows; an expert with more rows is split across tiles whose
// fp32 results are TMA reduce-added into a zeroed dW, and its rows run twice (values,
// then residuals) so that its error does not grow with the row count.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kStageBytes = 48 * 1024;      // A: 128x64 16-bit (16 KB) + B: up to 256x64 (32 KB)
constexpr int kStageBOffset = 16 * 1024;
constexpr int kMaxStages = 4;
constexpr int kEpiWarps = 4;
constexpr int kGemmThreads = 192;
constexpr int kTmemCols = 512;

struct __align__(8) GemmBarriers {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint32_t tmem_addr;
  int abort;
};

template <GemmKind KIND>
struct KindTraits {
  static constexpr bool kIsDw = (KIND == GemmKind::DwGU || KIND == GemmKind::DwD);
  static constexpr bool kTokenRows = !kIsDw;
  // Every kind is load-latency bound: four 48 KB stages in flight (three measured
  // slower even for the write-heavy weight-gradient GEMMs, given a deeper store ring).
  static constexpr int kStages = 4;
  static constexpr int kEpiBytes = 8 * 1024;                          // staging per epilogue warp
  static constexpr int kRing16 = kEpiBytes / 2048;                   // 2 KB 16-bit boxes
  static constexpr int kRing32 = kEpiBytes / 4096;                   // 4 KB fp32 boxes
  static constexpr int kSmemBytes =
      1024 /*barriers*/ + kStages * kStageBytes + kEpiWarps * kEpiBytes + 1024 /*align*/;
  // output columns per tile along N (DA: p.tile_n at run time)
  static constexpr int kTileN = (KIND == GemmKind::GateUp || KIND == GemmKind::BwdGU) ? 128 : 256;
};

struct TileInfo {
  int e;        // expert
  int m0;       // first row of the tile (token row, or feature row for dW)
  int n0;       // first output column
  int row0;     // dW: first token row of the K range
  int nkb;      // number of 64-deep K blocks
  int split;    // dW: the expert is split over several tiles (reduce-add)
  int kb_half;  // dW of a split expert: K blocks per operand pass (values, then residuals)
};

// Largest e in [0, E) with arr[e] <= v (arr non-decreasing, arr[0] <= v < arr[E]).
__device__ __forceinline__ int find_segment(const int* __restrict__ arr, int E, int v) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(arr + mid) <= v) lo = mid; else hi = mid;
  }
  return lo;
}

template <GemmKind KIND>
__device__ __forceinline__ int num_tiles(const GemmParams& p) {
  if constexpr (KindTraits<KIND>::kTokenRows) {
    return (__ldg(p.offsets + p.E) / kBM) * p.n_tiles;
  } else {
    return __ldg(p.dw_prefix + p.E) * p.m_tiles * p.n_tiles;
  }
}

template <GemmKind KIND>
__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, int t) {
  TileInfo ti;
  ti.split = 0;
  ti.row0 = 0;
  ti.kb_half = 0;
  if constexpr (KindTraits<KIND>::kTokenRows) {
    const int mt = t / p.n_tiles;
    const int nt = t - mt * p.n_tiles;
    ti.m0 = mt * kBM;
    ti.n0 = nt * (KIND == GemmKind::DA ? p.tile_n : KindTraits<KIND>::kTileN);
    ti.e = find_segment(p.offsets, p.E, ti.m0);
    if constexpr (KIND == GemmKind::GateUp || KIND == GemmKind::BwdGU || KIND == GemmKind::DA)
      ti.nkb = p.D / kBK;
    if constexpr (KIND == GemmKind::Down) ti.nkb = p.I / kBK;
    if constexpr (KIND == GemmKind::Dx) ti.nkb = 2 * (p.I / kBK);
  } else {
    const int tpc = p.m_tiles * p.n_tiles;
    const int g = t / tpc;
    const int l = t - g * tpc;
    ti.e = find_segment(p.dw_prefix, p.E, g);
    const int first = __ldg(p.dw_prefix + ti.e);
    const int nch = __ldg(p.dw_prefix + ti.e + 1) - first;
    const int j = g - first;
    const int beg = __ldg(p.offsets + ti.e);
    const int end = __ldg(p.offsets + ti.e + 1);
    ti.row0 = beg + j * kDwChunkRows;
    int rows = end - ti.row0;
    rows = rows < kDwChunkRows ? rows : kDwChunkRows;
    ti.nkb = rows > 0 ? rows / kBK : 0;
    ti.split = nch > 1;
    ti.kb_half = ti.nkb;
    if (ti.split) ti.nkb *= 2;   // compensated operands: the value pass, then the residual pass
    const int mt = l / p.n_tiles;
    const int nt = l - mt * p.n_tiles;
    ti.m0 = mt * kBM;
    ti.n0 = nt * 256;
  }
  return ti;
}

// ------------------------------------------------------------------ producer
// Issues the TMA loads of K block kb of tile ti into (sA, sB).
template <GemmKind KIND>
__device__ __forceinline__ void issue_kblock(const GemmParams& p, const TileInfo& ti, int kb,
                                             uint64_t* fb, uint8_t* sA, uint8_t* sB) {
  if constexpr (KIND == GemmKind::GateUp || KIND == GemmKind::BwdGU) {
    const int k0 = kb * kBK;
    const int wy = ti.e * p.D + k0;
    tma_load_2d(&p.mapA0, fb, sA, k0, ti.m0);
    // MN-major weight operands load as 3-D boxes: (64 columns) x (64 K rows) x (atoms)
    tma_load_3d(&p.mapB0, fb, sB, 0, wy, ti.n0 / 64);           // 2 gate atoms
    tma_load_3d(&p.mapB1, fb, sB + 16384, 0, wy, ti.n0 / 64);   // 2 up atoms
  } else if constexpr (KIND == GemmKind::DA) {
    // B = W_d[e] rows (features) as N x K, K-major: one box of tile_n rows
    const int k0 = kb * kBK;
    tma_load_2d(&p.mapA0, fb, sA, k0, ti.m0);
    tma_load_2d(&p.mapB0, fb, sB, k0, ti.e * p.I + ti.n0);
  } else if constexpr (KIND == GemmKind::Down) {
    const int k0 = kb * kBK;
    const int wy = ti.e * p.I + k0;
    tma_load_2d(&p.mapA0, fb, sA, k0, ti.m0);
    tma_load_3d(&p.mapB0, fb, sB, 0, wy, ti.n0 / 64);           // 4 atoms
  } else if constexpr (KIND == GemmKind::Dx) {
    const int k0 = kb * kBK;
    tma_load_2d(&p.mapA0, fb, sA, k0, ti.m0);
    if (k0 < p.I) tma_load_2d(&p.mapB0, fb, sB, k0, ti.e * p.D + ti.n0);
    else tma_load_2d(&p.mapB1, fb, sB, k0 - p.I, ti.e * p.D + ti.n0);
  } else {  // DwGU, DwD: both operands MN-major, K runs over token rows
    // a split expert runs its rows twice: with the fp16 values, then with the fp16
    // residuals of the rounded operand, into one accumulator
    const bool lo = ti.split && kb >= ti.kb_half;
    const int s0 = ti.row0 + (lo ? kb - ti.kb_half : kb) * kBK;
    const CUtensorMap* ma = (KIND == GemmKind::DwD && lo) ? &p.mapA1 : &p.mapA0;
    const CUtensorMap* mb = (KIND == GemmKind::DwGU && lo) ? &p.mapB1 : &p.mapB0;
    tma_load_3d(ma, fb, sA, 0, s0, ti.m0 / 64);   // 2 atoms
    tma_load_3d(mb, fb, sB, 0, s0, ti.n0 / 64);   // 4 atoms
  }
}

// Bytes one K block of a tile delivers to shared memory.
template <GemmKind KIND>
__device__ __forceinline__ uint32_t kblock_bytes(const GemmParams& p) {
  if constexpr (KIND == GemmKind::DA) return 16 * 1024 + static_cast<uint32_t>(p.tile_n) * 128;
  return 48 * 1024;
}

template <GemmKind KIND>
__device__ __forceinline__ void produce(const GemmParams& p, GemmBarriers* bars, uint8_t* stages,
                                        volatile int* abort) {
  constexpr int S = KindTraits<KIND>::kStages;
  int stage = 0;
  uint32_t phase = 0;
  const int ntiles = num_tiles<KIND>(p);
  const uint32_t bytes = kblock_bytes<KIND>(p);
  if (p.drop_loads) return;   // test hook: nothing arrives, the consumers' waits expire
  for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const TileInfo ti = decode_tile<KIND>(p, t);
    for (int kb = 0; kb < ti.nkb; ++kb) {
      if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort, p.err, kDevTimeoutProducer)) return;
      uint8_t* sA = stages + stage * kStageBytes;
      uint64_t* fb = &bars->full[stage];
      mbar_arrive_expect_tx(fb, bytes);   // posted before the copies are issued
      issue_kblock<KIND>(p, ti, kb, fb, sA, sA + kStageBOffset);
      if (++stage == S) { stage = 0; phase ^= 1u; }
    }
  }
}

// ------------------------------------------------------------------ MMA issuer
template <GemmKind KIND>
__device__ __forceinline__ void mma_issue(const GemmParams& p, GemmBarriers* bars,
                                          uint8_t* stages, uint32_t tmem_base,
                                          volatile int* abort) {
  using Tr = KindTraits<KIND>;
  constexpr int S = Tr::kStages;
  // operand majors: A K-major except the weight gradients (token rows are their K);
  // B MN-major except where the weights are read transposed (Dx, DA)
  constexpr bool kAmn = Tr::kIsDw;
  constexpr bool kBmn = !(KIND == GemmKind::Dx || KIND == GemmKind::DA);
  // the weight-gradient GEMMs read fp16 operands (they touch no weights); the rest bf16
  const int n_mma = (KIND == GemmKind::DA) ? p.tile_n : 256;
  const uint32_t idesc = umma_idesc_f16kind(128, n_mma, kAmn, kBmn, Tr::kIsDw);
  const uint32_t a_lbo = kAmn ? 8192u : 16u;
  const uint32_t a_step = kAmn ? 2048u : 32u;
  const uint32_t b_lbo = kBmn ? 8192u : 16u;
  const uint32_t b_step = kBmn ? 2048u : 32u;

  int stage = 0;
  uint32_t phase = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  const int ntiles = num_tiles<KIND>(p);
  for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const TileInfo ti = decode_tile<KIND>(p, t);
    if (ti.nkb == 0) continue;
    if (!mbar_wait(&bars->tempty[acc], acc_phase ^ 1u, abort, p.err, kDevTimeoutMma)) return;
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * 256);
    for (int kb = 0; kb < ti.nkb; ++kb) {
      if (!mbar_wait(&bars->full[stage], phase, abort, p.err, kDevTimeoutMma)) return;
      tc_fence_after();
      const uint32_t sa = smem_u32(stages + stage * kStageBytes);
      const uint32_t sb = sa + kStageBOffset;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t ad = umma_desc_sw128(sa + a_step * k, a_lbo, 1024u);
        const uint64_t bd = umma_desc_sw128(sb + b_step * k, b_lbo, 1024u);
        umma_bf16(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
      }
      umma_commit(&bars->empty[stage]);
      if (++stage == S) { stage = 0; phase ^= 1u; }
    }
    umma_commit(&bars->tfull[acc]);
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
  }
}

// ------------------------------------------------------------------ epilogue helpers
// Next buffer of the per-warp store ring; waits until the store that last read it is done.
template <int NBUF, int BYTES>
__device__ __forceinline__ uint8_t* ring_next(uint8_t* base, int& ring, int lane) {
  if (ring >= NBUF) {
    if (lane == 0) bulk_wait_read<NBUF - 1>();
    __syncwarp();
  }
  uint8_t* b = base + (ring % NBUF) * BYTES;
  ++ring;
  return b;
}

// 32 rows x 32 16-bit values (64-byte rows), 64-byte swizzle: 16-byte chunk c of row r
// sits at c ^ ((r>>1)&3).
__device__ __forceinline__ void stage_16_row(uint8_t* buf, int lane, const uint32_t (&pk)[16]) {
  uint8_t* rowp = buf + lane * 64;
  const int x = (lane >> 1) & 3;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(rowp + ((c ^ x) << 4)) =
        make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
}

// 32 rows x 32 fp32 (128-byte rows), 128-byte swizzle: chunk c of row r sits at c ^ (r&7).
__device__ __forceinline__ void stage_f32_row(uint8_t* buf, int lane, const float (&v)[32]) {
  uint8_t* rowp = buf + lane * 128;
  const int x = lane & 7;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<float4*>(rowp + ((c ^ x) << 4)) =
        make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
}

// Hand a staged box to TMA: every lane fences its writes, then lane 0 issues the copy.
__device__ __forceinline__ void store_box(const CUtensorMap* map, const uint8_t* buf, int x, int y,
                                          int lane, bool reduce_add) {
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (reduce_add) tma_reduce_add_2d(map, buf, x, y);
    else tma_store_2d(map, buf, x, y);
    bulk_commit();
  }
  __syncwarp();
}

// fp16 residuals (v0 - fp16(v0), v1 - fp16(v1)) given the packed fp16 pair.
__device__ __forceinline__ uint32_t f16x2_residual(uint32_t packed, float v0, float v1) {
  const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&packed));
  return pack_f16x2(v0 - hf.x, v1 - hf.y);
}

// ------------------------------------------------------------------ epilogue
template <GemmKind KIND>
__device__ __forceinline__ void epilogue(const GemmParams& p, GemmBarriers* bars, uint8_t* stg,
                                         uint32_t tmem_base, int warp, int lane,
                                         volatile int* abort) {
  using Tr = KindTraits<KIND>;
  constexpr int R16 = Tr::kRing16;
  constexpr int R32 = Tr::kRing32;
  const int q = warp & 3;  // TMEM lane quarter this warp may access
  int ring = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  const int ntiles = num_tiles<KIND>(p);
  for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const TileInfo ti = decode_tile<KIND>(p, t);
    const int row = ti.m0 + 32 * q;   // first of this warp's 32 rows; lane owns row + lane
    if constexpr (Tr::kIsDw) {
      if (ti.nkb == 0) {  // expert without tokens: its weight gradient is exactly zero
        float z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) z[i] = 0.f;
        for (int c = 0; c < 8; ++c) {
          uint8_t* buf = ring_next<R32, 4096>(stg, ring, lane);
          stage_f32_row(buf, lane, z);
          const int col = ti.n0 + 32 * c;
          if (KIND == GemmKind::DwGU) {
            if (col < p.I) store_box(&p.mapO0, buf, col, ti.e * p.D + row, lane, false);
            else store_box(&p.mapO1, buf, col - p.I, ti.e * p.D + row, lane, false);
          } else {
            store_box(&p.mapO0, buf, col, ti.e * p.I + row, lane, false);
          }
        }
        continue;
      }
    }
    int ok = 1;
    if (lane == 0) ok = mbar_wait(&bars->tfull[acc], acc_phase, abort, p.err, kDevTimeoutEpilogue);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    if (!ok) return;
    tc_fence_after();
    const uint32_t tb = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                        static_cast<uint32_t>(acc * 256);

    if constexpr (KIND == GemmKind::GateUp) {
      for (int c = 0; c < 4; ++c) {
        uint32_t g[32], u[32];
        tmem_ld32(tb + 32 * c, g);
        tmem_ld32(tb + 128 + 32 * c, u);
        tmem_ld_wait(g);
        tmem_ld_after_wait(u);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float a[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float gv = __uint_as_float(g[2 * i + h]);
            a[h] = gv * sigmoidf_fast(gv) * __uint_as_float(u[2 * i + h]);
          }
          pk[i] = pack_bf16x2(a[0], a[1]);
        }
        uint8_t* buf = ring_next<R16, 2048>(stg, ring, lane);
        stage_16_row(buf, lane, pk);
        store_box(&p.mapO0, buf, ti.n0 + 32 * c, row, lane, false);
      }
    } else if constexpr (KIND == GemmKind::Down || KIND == GemmKind::Dx) {
      for (int c = 0; c < 8; ++c) {
        uint32_t r[32];
        tmem_ld32(tb + 32 * c, r);
        tmem_ld_wait(r);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
        uint8_t* buf = ring_next<R16, 2048>(stg, ring, lane);
        stage_16_row(buf, lane, pk);
        store_box(&p.mapO0, buf, ti.n0 + 32 * c, row, lane, false);
      }
    } else if constexpr (KIND == GemmKind::DA) {
      const float wr = __ldg(p.w_perm + row + lane);   // router weight of this thread's row
      const int nch = p.tile_n / 32;
      for (int c = 0; c < nch; ++c) {
        uint32_t r[32];
        tmem_ld32(tb + 32 * c, r);
        tmem_ld_wait(r);
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = wr * __uint_as_float(r[i]);
        uint8_t* buf = ring_next<R32, 4096>(stg, ring, lane);
        stage_f32_row(buf, lane, v);
        store_box(&p.mapO0, buf, ti.n0 + 32 * c, row, lane, false);
      }
    } else if constexpr (KIND == GemmKind::BwdGU) {
      const int my_row = row + lane;
      const float wr = __ldg(p.w_perm + my_row);
      // rows of an expert whose dW is split over several tiles also get the fp16 residuals
      const bool want_lo =
          (__ldg(p.offsets + ti.e + 1) - __ldg(p.offsets + ti.e)) > kDwChunkRows;
      const float4* da_row =
          reinterpret_cast<const float4*>(p.dA + static_cast<size_t>(my_row) * p.I + ti.n0);
      for (int c = 0; c < 4; ++c) {
        float4 d4[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) d4[i] = __ldg(da_row + 8 * c + i);   // w-scaled dA, fp32
        uint32_t g[32], u[32];
        tmem_ld32(tb + 32 * c, g);
        tmem_ld32(tb + 128 + 32 * c, u);
        tmem_ld_wait(g);
        tmem_ld_after_wait(u);
        const float* da = reinterpret_cast<const float*>(d4);
        uint32_t pa[16], pg[16], pu[16], pg16[16], pu16[16], la[16], lg[16], lu[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float r[2][3];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float gv = __uint_as_float(g[2 * i + h]);
            const float uv = __uint_as_float(u[2 * i + h]);
            const float dv = da[2 * i + h];
            const float sg = sigmoidf_fast(gv);
            const float si = gv * sg;
            r[h][0] = wr * si * uv;                              // w * act (dW_down operand)
            r[h][1] = dv * uv * sg * (1.0f + gv * (1.0f - sg));  // dG
            r[h][2] = dv * si;                                   // dU
          }
          pa[i] = pack_f16x2(r[0][0], r[1][0]);
          pg[i] = pack_bf16x2(r[0][1], r[1][1]);
          pu[i] = pack_bf16x2(r[0][2], r[1][2]);
          pg16[i] = pack_f16x2(r[0][1], r[1][1]);
          pu16[i] = pack_f16x2(r[0][2], r[1][2]);
          la[i] = f16x2_residual(pa[i], r[0][0], r[1][0]);
          lg[i] = f16x2_residual(pg16[i], r[0][1], r[1][1]);
          lu[i] = f16x2_residual(pu16[i], r[0][2], r[1][2]);
        }
        const int col = ti.n0 + 32 * c;
        uint8_t* b0 = ring_next<R16, 2048>(stg, ring, lane);
        stage_16_row(b0, lane, pa);
        store_box(&p.mapO0, b0, col, row, lane, false);        // w*act, fp16
        uint8_t* b1 = ring_next<R16, 2048>(stg, ring, lane);
        stage_16_row(b1, lane, pg);
        store_box(&p.mapO1, b1, col, row, lane, false);        // dG, bf16
        uint8_t* b2 = ring_next<R16, 2048>(stg, ring, lane);
        stage_16_row(b2, lane, pu);
        store_box(&p.mapO1, b2, p.I + col, row, lane, false);  // dU, bf16
        uint8_t* b3 = ring_next<R16, 2048>(stg, ring, lane);
        stage_16_row(b3, lane, pg16);
        store_box(&p.mapO2, b3, col, row, lane, false);        // dG, fp16
        uint8_t* b4 = ring_next<R16, 2048>(stg, ring, lane);
        stage_16_row(b4, lane, pu16);
        store_box(&p.mapO2, b4, p.I + col, row, lane, false);  // dU, fp16
        if (want_lo) {
          uint8_t* c0 = ring_next<R16, 2048>(stg, ring, lane);
          stage_16_row(c0, lane, la);
          store_box(&p.mapO3, c0, col, row, lane, false);        // w*act residual
          uint8_t* c1 = ring_next<R16, 2048>(stg, ring, lane);
          stage_16_row(c1, lane, lg);
          store_box(&p.mapO4, c1, col, row, lane, false);        // dG residual
          uint8_t* c2 = ring_next<R16, 2048>(stg, ring, lane);
          stage_16_row(c2, lane, lu);
          store_box(&p.mapO4, c2, p.I + col, row, lane, false);  // dU residual
        }
      }
    } else {  // DwGU, DwD: fp32 out, plain store or split-K reduce-add
      for (int c = 0; c < 8; ++c) {
        uint32_t r[32];
        tmem_ld32(tb + 32 * c, r);
        tmem_ld_wait(r);
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
        uint8_t* buf = ring_next<R32, 4096>(stg, ring, lane);
        stage_f32_row(buf, lane, v);
        const int col = ti.n0 + 32 * c;
        if (KIND == GemmKind::DwGU) {
          if (col < p.I) store_box(&p.mapO0, buf, col, ti.e * p.D + row, lane, ti.split);
          else store_box(&p.mapO1, buf, col - p.I, ti.e * p.D + row, lane, ti.split);
        } else {
          store_box(&p.mapO0, buf, col, ti.e * p.I + row, lane, ti.split);
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->tempty[acc]);
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
  }
}

// ------------------------------------------------------------------ kernel
template <GemmKind KIND>
__global__ void __launch_bounds__(kGemmThreads, 1) k_grouped_gemm(const __grid_constant__ GemmParams p) {
  using Tr = KindTraits<KIND>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  GemmBarriers* bars = reinterpret_cast<GemmBarriers*>(smem);
  uint8_t* stages = smem + 1024;
  uint8_t* staging = stages + Tr::kStages * kStageBytes;
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < Tr::kStages; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->tfull[i], 1);
      mbar_init(&bars->tempty[i], kEpiWarps);
    }
    bars->abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.mapA0);
    tma_prefetch_desc(&p.mapB0);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_addr, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_addr;

  if (warp == 0) {
    if (lane == 0) produce<KIND>(p, bars, stages, abort);
  } else if (warp == 1) {
    if (lane == 0) mma_issue<KIND>(p, bars, stages, tmem_base, abort);
  } else {
    epilogue<KIND>(p, bars, staging + (warp - 2) * Tr::kEpiBytes, tmem_base, warp, lane, abort);
    if (lane == 0) bulk_wait_all();
  }

  if (*abort) {
    // A wait gave up: let copies and MMAs already in flight drain (bounded) before
    // the shared memory and TMEM are released.
    const unsigned long long t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2000000ull) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <GemmKind KIND>
cudaError_t launch_gemm_kind(const GemmParams& p, int max_tiles, int num_sms, cudaStream_t s) {
  constexpr int kSmem = KindTraits<KIND>::kSmemBytes;
  static_assert(kSmem <= 232448, "shared memory budget");
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_grouped_gemm<KIND>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  int grid = max_tiles < num_sms ? max_tiles : num_sms;
  if (grid < 1) grid = 1;
  k_grouped_gemm<KIND><<<grid, kGemmThreads, kSmem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
