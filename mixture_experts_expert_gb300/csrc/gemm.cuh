// Persistent, warp-specialised grouped GEMM for the MoE expert MLP on sm_103a.
//
// One CTA per SM, 192 threads:
//   warp 0      TMA producer (lane 0 issues cp.async.bulk.tensor into a ring of stages)
//   warp 1      TMEM owner + MMA issuer (lane 0 issues tcgen05.mma, fp32 accumulators in
//               two 256-column TMEM buffers, so one tile's epilogue overlaps the next
//               tile's MMAs)
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM lanes
//               32*(w%4)..+31), fused elementwise math, tile stores or reduce-adds through a
//               swizzled shared-memory ring and TMA.
//
// Token-row kinds run on CTA pairs (clusters of two): one M = 256 tcgen05.mma issued by the
// even CTA covers two 128-row tiles of one expert, each CTA loading its own 128 rows of A
// and half of the N columns of B.  A 64-deep K block then costs 32 KB of shared memory per
// SM instead of 48 KB, so six stages fit where four did: the main loop is bound by load
// latency, and the deeper ring hides more of it.  The pair's tile space enumerates, per
// expert, ceil(m_tiles / 2) row pairs; when an expert has an odd number of row tiles the
// odd CTA's half of its last pair is a ghost (loaded and multiplied, never stored).
// The weight-gradient kinds (K = token rows, M = feature rows) run one CTA per tile, M = 128.
//
// Tiles are scheduled statically (tile = cta (or pair) index + i * count) over a tile space
// whose size is read on the device from the expert offsets, so the launch is
// independent of the routing (no host sync; valid inside a captured CUDA graph).  Within
// an expert the pair kinds enumerate tiles row pair by row pair (consecutive tiles share
// the token rows) or, per the shape's tuning, N tile by N tile (consecutive tiles share a
// weight tile: better when an expert's weights are large and it has several row pairs).
// Odd last row tiles are computed transposed unless the tuning turns that off.
//
// Kinds (row-major; "perm" rows are expert-sorted, padded to 128 rows per expert):
//   GateUp  act[s, i]  = silu(x_perm[s] W_g[e])_i * (x_perm[s] W_u[e])_i   N: 128 gate + 128 up
//   Down    y_perm[s]  = act[s] W_d[e]
//   DA      dA[s]      = w_perm[s] * dy_perm[s] W_d[e]^T   (scaled in fp32, stored fp16; dy_perm
//           unscaled); for experts with compensated dW operands also the fp16 residual
//   BwdGU   recompute G, U as GateUp; the epilogue reads dA and writes w*act (fp16),
//           dG = dA U silu'(G), dU = dA silu(G) (bf16 for Dx, fp16 for the dW GEMMs) and,
//           for experts with compensated dW operands, the fp16 residuals v - fp16(v)
//   Dx      dx_perm[s] = [dG dU][s] [W_g[e]; W_u[e]]^T                    (K = 2I)
//   DwGU    [dW_g dW_u][e] = x16_e^T [dG dU]16_e        (K = the expert's token rows)
//   DwD     dW_d[e]        = (w act)16_e^T dy16_e
// The weight-gradient GEMMs sum over up to thousands of token rows, so their operands
// are fp16 (10-bit mantissa; x and dY convert exactly) rather than bf16: the rounding of
// the intermediates (dG, dU, w*act) is what bounds dW's absolute error.  dW tiles cover
// at most dw_chunk_rows token rows; an expert with more rows is split into equal chunks on
// tiles whose fp32 results are TMA reduce-added into a zeroed dW.  An expert with more
// than kDwCompRows real rows runs its rows twice (values, then residuals), so that its
// error stops growing with the row count.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kStageBOffset = 16 * 1024;    // B follows A (128 x 64 16-bit = 16 KB) in a stage
constexpr int kMaxStages = 6;
constexpr int kEpiWarps = 4;
constexpr int kGemmThreads = 192;
constexpr int kTmemCols = 512;

struct __align__(8) GemmBarriers {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t xfull[2];    // swapped gate/up tails: up warp -> gate warp exchange, per warp pair
  uint64_t xempty[2];
  uint32_t tmem_addr;
  int abort;
};

template <GemmKind KIND>
struct KindTraits {
  static constexpr bool kIsDw = (KIND == GemmKind::DwGU || KIND == GemmKind::DwD);
  static constexpr bool kTokenRows = !kIsDw;
  static constexpr bool kPair = kTokenRows;   // M = 256 over a CTA pair
  // weights stored N-contiguous (MN-major as the B operand / as the swapped A operand)
  static constexpr bool kWeightsMN =
      (KIND == GemmKind::GateUp || KIND == GemmKind::BwdGU || KIND == GemmKind::Down);
  // Stage = A (128 x 64) + this CTA's B: half of N on a pair (<= 128 x 64), else up to 256 x 64.
  static constexpr int kStageBytes = kPair ? 32 * 1024 : 48 * 1024;
  // Every kind is load-latency bound, so stages take what the epilogue staging leaves
  // (for the single-CTA kinds three stages measured slower than four even for the
  // write-heavy weight-gradient GEMMs, given a deeper store ring).
  static constexpr int kStages = kPair ? 6 : 4;
  static constexpr int kEpiBytes = kPair ? 6 * 1024 : 8 * 1024;      // staging per epilogue warp
  static constexpr int kRing16 = kEpiBytes / 2048;                   // 2 KB 16-bit boxes
  static constexpr int kRing32 = kEpiBytes / 4096;                   // 4 KB fp32 boxes
  // pair kinds: per-expert prefix of row pairs, [0, E]
  static constexpr int kPrefixBytes = kPair ? ((kMaxExperts + 1) * 4 + 127) / 128 * 128 : 0;
  static constexpr int kSmemBytes = 1024 /*barriers*/ + kStages * kStageBytes +
                                    kEpiWarps * kEpiBytes + kPrefixBytes + 1024 /*align*/;
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
  int comp;     // dW: compensated operands (a value pass, then a residual pass)
  int kb_half;  // dW of a compensated expert: K blocks per operand pass
  int ghost;    // pair kinds: this CTA's 128 rows lie past the expert's last row tile
  int swap;     // pair kinds: the expert's odd last row tile, computed transposed
  int tail_n;   // swap: token rows computed (a multiple of 32); the rest are padding
};

// Whether expert e's weight gradient takes compensated operands (see kDwCompRows): its real
// rows when the counts are given, else its padded rows.
__device__ __forceinline__ bool dw_compensated(const GemmParams& p, int e) {
  const int rows =
      p.counts ? __ldg(p.counts + e) : __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
  return rows > kDwCompRows;
}

// Largest e in [0, E) with arr[e] <= v (arr non-decreasing, arr[0] <= v < arr[E]).
__device__ __forceinline__ int find_segment(const int* __restrict__ arr, int E, int v) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(arr + mid) <= v) lo = mid; else hi = mid;
  }
  return lo;
}

// The same search over a prefix held in shared memory.
__device__ __forceinline__ int find_segment_smem(const int* arr, int E, int v) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (arr[mid] <= v) lo = mid; else hi = mid;
  }
  return lo;
}

// Pair kinds: pfx[e] = number of 256-row pairs of experts before e (pfx[E] = all pairs),
// an expert of m row tiles owning ceil(m / 2).  Computed by every CTA into shared memory
// (all threads take part; the caller synchronises before use).
__device__ __forceinline__ void build_pair_prefix(const GemmParams& p, int* pfx) {
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
    const int mt = (__ldg(p.offsets + e + 1) - __ldg(p.offsets + e)) / kBM;
    pfx[e + 1] = (mt + 1) >> 1;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (p.E + 31) / 32;          // each lane scans a contiguous run of experts
    const int b = lane * per;
    const int end = b + per < p.E ? b + per : p.E;
    int sum = 0;
    for (int e = b; e < end; ++e) sum += pfx[e + 1];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int e = b; e < end; ++e) {
      run += pfx[e + 1];
      pfx[e + 1] = run;
    }
    if (lane == 0) pfx[0] = 0;
  }
}

template <GemmKind KIND>
__device__ __forceinline__ int num_tiles(const GemmParams& p, const int* pfx) {
  if constexpr (KindTraits<KIND>::kPair) {
    return pfx[p.E] * p.n_tiles;
  } else if constexpr (KindTraits<KIND>::kTokenRows) {
    return (__ldg(p.offsets + p.E) / kBM) * p.n_tiles;
  } else {
    return __ldg(p.dw_prefix + p.E) * p.m_tiles * p.n_tiles;
  }
}

// First tile and stride of this CTA's static schedule (pairs step together).
template <GemmKind KIND>
__device__ __forceinline__ int first_tile() {
  if constexpr (KindTraits<KIND>::kPair) return static_cast<int>(cluster_id_x());
  return blockIdx.x;
}
template <GemmKind KIND>
__device__ __forceinline__ int tile_stride() {
  if constexpr (KindTraits<KIND>::kPair) return static_cast<int>(num_clusters_x());
  return gridDim.x;
}

template <GemmKind KIND>
__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, int t, const int* pfx,
                                                int rank) {
  TileInfo ti;
  ti.split = 0;
  ti.comp = 0;
  ti.row0 = 0;
  ti.kb_half = 0;
  ti.ghost = 0;
  ti.swap = 0;
  ti.tail_n = 0;
  if constexpr (KindTraits<KIND>::kTokenRows) {
    const int nt_all = t / p.n_tiles;
    const int nt = t - nt_all * p.n_tiles;
    ti.n0 = nt * (KIND == GemmKind::DA ? p.tile_n : KindTraits<KIND>::kTileN);
    if constexpr (KindTraits<KIND>::kPair) {
      // nt_all is the pair index: expert e, pair j of it, this CTA's half l = 2j + rank
      ti.e = find_segment_smem(pfx, p.E, nt_all);
      const int beg = __ldg(p.offsets + ti.e);
      const int mt = (__ldg(p.offsets + ti.e + 1) - beg) / kBM;
      int j = nt_all - pfx[ti.e];
      if (p.order == 1) {
        // the expert's tiles N tile by N tile: its row pairs share each weight tile back to back
        const int np = pfx[ti.e + 1] - pfx[ti.e];
        const int l = t - pfx[ti.e] * p.n_tiles;
        const int n_idx = l / np;
        j = l - n_idx * np;
        ti.n0 = n_idx * (KIND == GemmKind::DA ? p.tile_n : KindTraits<KIND>::kTileN);
      }
      // An odd last row tile has no partner tile: the pair computes it transposed
      // (weights as the M = 256 operand, its token rows as N), so only its real rows,
      // rounded up to 32, cost MMA time.  DA with 128-column tiles has no M = 256 form of
      // the swap and runs the tile with an idle (ghost) odd half instead.
      if (p.swap_tails && (mt & 1) && 2 * j + 1 == mt &&
          (KIND != GemmKind::DA || p.tile_n == 256)) {
        ti.swap = 1;
        ti.m0 = beg + (mt - 1) * kBM;
        int rows = kBM;
        if (p.counts) {
          rows = __ldg(p.counts + ti.e) - (mt - 1) * kBM;
          rows = rows < 0 ? 0 : (rows > kBM ? kBM : rows);
        }
        ti.tail_n = rows <= 32 ? 32 : (rows + 31) & ~31;
      } else {
        const int l = 2 * j + rank;
        ti.ghost = l >= mt;
        ti.m0 = beg + l * kBM;   // a ghost reads rows past the expert (never stored)
      }
    } else {
      ti.m0 = nt_all * kBM;
      ti.e = find_segment(p.offsets, p.E, ti.m0);
    }
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
    // nch equal chunks (rounded up to 64 rows), so no chunk is a sliver
    const int per = ((end - beg + nch - 1) / nch + kBK - 1) / kBK * kBK;
    ti.row0 = beg + j * per;
    // K runs over the chunk's rows up to the expert's last real row (with counts) rounded
    // up to 64: the padding rows after it are zero in every operand
    int last = end;
    if (p.counts) {
      const int real = beg + __ldg(p.counts + ti.e);
      last = real < end ? real : end;
    }
    int rows = last - ti.row0;
    rows = rows < per ? rows : per;
    ti.nkb = rows > 0 ? (rows + kBK - 1) / kBK : 0;
    ti.split = nch > 1;
    ti.comp = dw_compensated(p, ti.e);
    ti.kb_half = ti.nkb;
    if (ti.comp) ti.nkb *= 2;   // the value pass, then the residual pass
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
    const bool lo = ti.comp && kb >= ti.kb_half;
    const int s0 = ti.row0 + (lo ? kb - ti.kb_half : kb) * kBK;
    const CUtensorMap* ma = (KIND == GemmKind::DwD && lo) ? &p.mapA1 : &p.mapA0;
    const CUtensorMap* mb = (KIND == GemmKind::DwGU && lo) ? &p.mapB1 : &p.mapB0;
    tma_load_3d(ma, fb, sA, 0, s0, ti.m0 / 64);   // 2 atoms
    tma_load_3d(mb, fb, sB, 0, s0, ti.n0 / 64);   // 4 atoms
  }
}

// Pair kinds: this CTA's share of K block kb (its 128 rows of A, its half of B's columns);
// completion is counted on the even CTA's full barrier `fb` (a shared::cluster address).
template <GemmKind KIND>
__device__ __forceinline__ void issue_kblock_pair(const GemmParams& p, const TileInfo& ti, int kb,
                                                  uint32_t fb, uint8_t* sA, uint8_t* sB,
                                                  int rank) {
  const int k0 = kb * kBK;
  tma_load_2d_pair(&p.mapA0, fb, sA, k0, ti.m0);
  if constexpr (KIND == GemmKind::GateUp || KIND == GemmKind::BwdGU) {
    // N = 128 gate columns (even CTA) | the same 128 up columns (odd CTA), two 64-wide atoms
    tma_load_3d_pair(rank ? &p.mapB1 : &p.mapB0, fb, sB, 0, ti.e * p.D + k0, ti.n0 / 64);
  } else if constexpr (KIND == GemmKind::DA) {
    // W_d[e] feature rows, K-major: tile_n / 2 rows per CTA
    tma_load_2d_pair(&p.mapB0, fb, sB, k0, ti.e * p.I + ti.n0 + rank * (p.tile_n / 2));
  } else if constexpr (KIND == GemmKind::Down) {
    tma_load_3d_pair(&p.mapB0, fb, sB, 0, ti.e * p.I + k0, ti.n0 / 64 + 2 * rank);
  } else if constexpr (KIND == GemmKind::Dx) {
    const int r = ti.e * p.D + ti.n0 + 128 * rank;
    if (k0 < p.I) tma_load_2d_pair(&p.mapB0, fb, sB, k0, r);
    else tma_load_2d_pair(&p.mapB1, fb, sB, k0 - p.I, r);
  }
}

// Pair kinds, swapped tail tile: this CTA's 128 weight rows (the M operand: output
// features, or for gate/up 64 gate + the same 64 up features) into sA, and its half of
// the tail's token rows (the N operand; a fixed 64-row box, of which the MMA reads
// tail_n / 2) into sB.
template <GemmKind KIND>
__device__ __forceinline__ void issue_kblock_swap(const GemmParams& p, const TileInfo& ti, int kb,
                                                  uint32_t fb, uint8_t* sA, uint8_t* sB,
                                                  int rank) {
  const int k0 = kb * kBK;
  tma_load_2d_pair(&p.mapA1, fb, sB, k0, ti.m0 + rank * (ti.tail_n / 2));
  if constexpr (KIND == GemmKind::GateUp || KIND == GemmKind::BwdGU) {
    const int atom = (ti.n0 + 64 * rank) / 64;
    tma_load_3d_pair(&p.mapB2, fb, sA, 0, ti.e * p.D + k0, atom);          // gate, 1 atom
    tma_load_3d_pair(&p.mapB3, fb, sA + 8192, 0, ti.e * p.D + k0, atom);   // up, 1 atom
  } else if constexpr (KIND == GemmKind::DA) {
    tma_load_2d_pair(&p.mapB0, fb, sA, k0, ti.e * p.I + ti.n0 + 128 * rank);
  } else if constexpr (KIND == GemmKind::Down) {
    tma_load_3d_pair(&p.mapB0, fb, sA, 0, ti.e * p.I + k0, ti.n0 / 64 + 2 * rank);
  } else if constexpr (KIND == GemmKind::Dx) {
    const int r = ti.e * p.D + ti.n0 + 128 * rank;
    if (k0 < p.I) tma_load_2d_pair(&p.mapB0, fb, sA, k0, r);
    else tma_load_2d_pair(&p.mapB1, fb, sA, k0 - p.I, r);
  }
}

// Bytes one K block of a swapped tail delivers to each CTA: 128 weight rows + 64 token rows.
constexpr uint32_t kSwapKBlockBytes = 16 * 1024 + 8 * 1024;

// Bytes one K block of a tile delivers to this CTA's shared memory.
template <GemmKind KIND>
__device__ __forceinline__ uint32_t kblock_bytes(const GemmParams& p) {
  if constexpr (KindTraits<KIND>::kPair) {
    if constexpr (KIND == GemmKind::DA) return 16 * 1024 + static_cast<uint32_t>(p.tile_n) * 64;
    return 32 * 1024;
  }
  if constexpr (KIND == GemmKind::DA) return 16 * 1024 + static_cast<uint32_t>(p.tile_n) * 128;
  return 48 * 1024;
}

template <GemmKind KIND>
__device__ __forceinline__ void produce(const GemmParams& p, GemmBarriers* bars, uint8_t* stages,
                                        const int* pfx, volatile int* abort) {
  using Tr = KindTraits<KIND>;
  constexpr int S = Tr::kStages;
  int stage = 0;
  uint32_t phase = 0;
  const int ntiles = num_tiles<KIND>(p, pfx);
  const uint32_t bytes = kblock_bytes<KIND>(p);
  const int rank = Tr::kPair ? static_cast<int>(cluster_ctarank()) : 0;
  const uint32_t full0 = Tr::kPair ? mapa_shared(smem_u32(&bars->full[0]), 0) : 0u;
  if (p.drop_loads) return;   // test hook: nothing arrives, the consumers' waits expire
  for (int t = first_tile<KIND>(); t < ntiles; t += tile_stride<KIND>()) {
    const TileInfo ti = decode_tile<KIND>(p, t, pfx, rank);
    for (int kb = 0; kb < ti.nkb; ++kb) {
      if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort, p.err, kDevTimeoutProducer)) return;
      uint8_t* sA = stages + stage * Tr::kStageBytes;
      if constexpr (Tr::kPair) {
        // the even CTA's barrier counts both CTAs' bytes; expect_tx is posted by the even
        // CTA alone (the odd CTA's bytes may land first: the phase cannot complete before
        // the even CTA has arrived)
        const uint32_t fb = full0 + 8u * static_cast<uint32_t>(stage);
        if (rank == 0)
          mbar_arrive_expect_tx(&bars->full[stage], 2 * (ti.swap ? kSwapKBlockBytes : bytes));
        if (ti.swap) issue_kblock_swap<KIND>(p, ti, kb, fb, sA, sA + kStageBOffset, rank);
        else issue_kblock_pair<KIND>(p, ti, kb, fb, sA, sA + kStageBOffset, rank);
      } else {
        uint64_t* fb = &bars->full[stage];
        mbar_arrive_expect_tx(fb, bytes);   // posted before the copies are issued
        issue_kblock<KIND>(p, ti, kb, fb, sA, sA + kStageBOffset);
      }
      if (++stage == S) { stage = 0; phase ^= 1u; }
    }
  }
  if constexpr (Tr::kPair) {
    // Wait until the MMA issuer has released every stage: its releases arrive on this
    // CTA's barriers from the even CTA and must all have landed before the CTA exits.
    for (int i = 0; i < S; ++i) {
      if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort, p.err, kDevTimeoutProducer)) return;
      if (++stage == S) { stage = 0; phase ^= 1u; }
    }
  }
}

// ------------------------------------------------------------------ MMA issuer
template <GemmKind KIND>
__device__ __forceinline__ void mma_issue(const GemmParams& p, GemmBarriers* bars,
                                          uint8_t* stages, uint32_t tmem_base, const int* pfx,
                                          volatile int* abort) {
  using Tr = KindTraits<KIND>;
  constexpr int S = Tr::kStages;
  // on a pair only the even CTA issues; the odd CTA's MMA warp just owns its TMEM
  if constexpr (Tr::kPair) {
    if (cluster_ctarank() != 0) return;
  }
  // operand majors: A K-major except the weight gradients (token rows are their K);
  // B MN-major except where the weights are read transposed (Dx, DA)
  constexpr bool kAmn = Tr::kIsDw;
  constexpr bool kBmn = !(KIND == GemmKind::Dx || KIND == GemmKind::DA);
  // the weight-gradient GEMMs read fp16 operands (they touch no weights); the rest bf16
  const int n_mma = (KIND == GemmKind::DA) ? p.tile_n : 256;
  const uint32_t idesc = umma_idesc_f16kind(Tr::kPair ? 256 : 128, n_mma, kAmn, kBmn, Tr::kIsDw);
  // swapped tails: weights (sA) as the M operand, token rows (sB, K-major) as N
  const uint32_t w_lbo = Tr::kWeightsMN ? 8192u : 16u;
  const uint32_t w_step = Tr::kWeightsMN ? 2048u : 32u;
  const uint32_t a_lbo = kAmn ? 8192u : 16u;
  const uint32_t a_step = kAmn ? 2048u : 32u;
  const uint32_t b_lbo = kBmn ? 8192u : 16u;
  const uint32_t b_step = kBmn ? 2048u : 32u;

  int stage = 0;
  uint32_t phase = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  const int ntiles = num_tiles<KIND>(p, pfx);
  for (int t = first_tile<KIND>(); t < ntiles; t += tile_stride<KIND>()) {
    const TileInfo ti = decode_tile<KIND>(p, t, pfx, 0);
    if (ti.nkb == 0) continue;
    if (!mbar_wait(&bars->tempty[acc], acc_phase ^ 1u, abort, p.err, kDevTimeoutMma)) return;
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * 256);
    const uint32_t idesc_swap =
        umma_idesc_f16kind(256, ti.swap ? ti.tail_n : 32, Tr::kWeightsMN, false, false);
    for (int kb = 0; kb < ti.nkb; ++kb) {
      if (!mbar_wait(&bars->full[stage], phase, abort, p.err, kDevTimeoutMma)) return;
      tc_fence_after();
      const uint32_t sa = smem_u32(stages + stage * Tr::kStageBytes);
      const uint32_t sb = sa + kStageBOffset;
      if (Tr::kPair && ti.swap) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t ad = umma_desc_sw128(sa + w_step * k, w_lbo, 1024u);
          const uint64_t bd = umma_desc_sw128(sb + 32u * k, 16u, 1024u);
          umma_bf16_pair(d_tmem, ad, bd, idesc_swap, (kb > 0 || k > 0) ? 1u : 0u);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t ad = umma_desc_sw128(sa + a_step * k, a_lbo, 1024u);
          const uint64_t bd = umma_desc_sw128(sb + b_step * k, b_lbo, 1024u);
          if constexpr (Tr::kPair) umma_bf16_pair(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          else umma_bf16(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
        }
      }
      if constexpr (Tr::kPair) umma_commit_pair(&bars->empty[stage], 0x3);
      else umma_commit(&bars->empty[stage]);
      if (++stage == S) { stage = 0; phase ^= 1u; }
    }
    if constexpr (Tr::kPair) umma_commit_pair(&bars->tfull[acc], 0x3);
    else umma_commit(&bars->tfull[acc]);
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
  }
  if constexpr (Tr::kPair) {
    // Wait for both CTAs' epilogues to release both accumulators: the odd CTA's releases
    // arrive on this CTA's barriers and must all have landed before the pair exits.
    for (int i = 0; i < 2; ++i) {
      if (!mbar_wait(&bars->tempty[acc], acc_phase ^ 1u, abort, p.err, kDevTimeoutMma)) return;
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
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

// Group staging: before staging N boxes into the next N slots of an NBUF-slot ring, at
// most NBUF - N earlier stores may still be reading theirs (those used other slots).
template <int NBUF, int N>
__device__ __forceinline__ void ring_reserve(int lane) {
  static_assert(N <= NBUF, "group larger than the ring");
  if (lane == 0) bulk_wait_read<NBUF - N>();
  __syncwarp();
}
template <int NBUF, int BYTES>
__device__ __forceinline__ uint8_t* ring_slot(uint8_t* base, int& ring) {
  uint8_t* b = base + (ring % NBUF) * BYTES;
  ++ring;
  return b;
}

// Hands a staged box to TMA without a fence of its own: the caller fences once (all
// lanes, then __syncwarp) for every box it staged before issuing them.
__device__ __forceinline__ void issue_box(const CUtensorMap* map, const uint8_t* buf, int x,
                                          int y, int lane) {
  if (lane == 0) {
    tma_store_2d(map, buf, x, y);
    bulk_commit();
  }
}

// One proxy fence for a group of staged boxes.
__device__ __forceinline__ void fence_boxes() {
  fence_proxy_async_smem();
  __syncwarp();
}

// fp16 residuals (v0 - fp16(v0), v1 - fp16(v1)) given the packed fp16 pair.
__device__ __forceinline__ uint32_t f16x2_residual(uint32_t packed, float v0, float v1) {
  const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&packed));
  return pack_f16x2(v0 - hf.x, v1 - hf.y);
}

// ------------------------------------------------------------------ swapped tails
// The accumulator of a swapped tile is transposed: TMEM lane = output column (feature),
// TMEM column = token row.  Each lane of a warp holds one column for 32 consecutive rows;
// these place element (row i, column lane) into a 32 x 32 box.
// 16-bit, 64-byte swizzle (chunk c of row r at c ^ ((r>>1)&3)).
__device__ __forceinline__ void stage_16_col(uint8_t* buf, int lane, const float (&v)[32],
                                             bool fp16) {
  const int c = lane >> 3;
  const int off = (lane & 7) * 2;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const uint16_t h = fp16 ? __half_as_ushort(__float2half_rn(v[i]))
                            : __bfloat16_as_ushort(__float2bfloat16_rn(v[i]));
    *reinterpret_cast<uint16_t*>(buf + i * 64 + ((c ^ ((i >> 1) & 3)) << 4) + off) = h;
  }
}

// fp32, 128-byte swizzle (chunk c of row r at c ^ (r&7)).
__device__ __forceinline__ void stage_f32_col(uint8_t* buf, int lane, const float (&v)[32]) {
  const int c = lane >> 2;
  const int off = (lane & 3) * 4;
#pragma unroll
  for (int i = 0; i < 32; ++i)
    *reinterpret_cast<float*>(buf + i * 128 + ((c ^ (i & 7)) << 4) + off) = v[i];
}

// v[i] <- v[i] - fp16(v[i]): what the fp16 copy of v left out.
__device__ __forceinline__ void to_f16_residual(float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] -= __half2float(__float2half_rn(v[i]));
}

// Whether any of the values rounds to an fp16 infinity (|v| >= 65520).
__device__ __forceinline__ bool f16_overflows(const float (&v)[32]) {
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(v[i]));
  return m >= 65520.f;
}

// Scaled fp16 intermediates that overflowed: one report per warp.
__device__ __forceinline__ void report_f16_overflow(const GemmParams& p, bool ovf) {
  if (__any_sync(0xffffffffu, ovf) && (threadIdx.x & 31) == 0) report_error(p.err, kDevFp16Range);
}

// A zeroed box in the next ring buffer.
template <int NBUF, int BYTES>
__device__ __forceinline__ uint8_t* stage_zero(uint8_t* stg, int& ring, int lane) {
  uint8_t* buf = ring_next<NBUF, BYTES>(stg, ring, lane);
  for (int b = lane; b < BYTES / 16; b += 32)
    *reinterpret_cast<uint4*>(buf + 16 * b) = make_uint4(0u, 0u, 0u, 0u);
  return buf;
}

// Zeros for the padding rows of a swapped tile that were not computed (tail_n .. 127),
// 32 columns at x.
__device__ __forceinline__ void store_zero_rows(const CUtensorMap* map, const uint8_t* zbuf, int x,
                                                const TileInfo& ti, int lane) {
  for (int y = ti.m0 + ti.tail_n; y < ti.m0 + kBM; y += 32) store_box(map, zbuf, x, y, lane, false);
}

// Epilogue of a swapped tail tile; returns false when a bounded wait gave up.
// Down, Dx, DA: TMEM lanes 32q.. hold output columns n0 + 128*rank + 32q + lane.
// GateUp, BwdGU: lanes 0-63 hold gate and lanes 64-127 up of the same 64 act columns
// n0 + 64*rank + (0..63); the up warp of each 32 columns hands its values to the gate
// warp through its staging buffer (two mbarriers per warp pair), and the gate warp
// computes and stores every output.
template <GemmKind KIND>
__device__ __forceinline__ bool epilogue_swap(const GemmParams& p, GemmBarriers* bars, uint8_t* stg,
                                              uint8_t* stg_base, uint32_t tb, const TileInfo& ti,
                                              int q, int lane, int rank, int& ring, uint32_t& xph,
                                              volatile int* abort) {
  using Tr = KindTraits<KIND>;
  constexpr int R16 = Tr::kRing16;
  const int nch = ti.tail_n / 32;
  if constexpr (KIND == GemmKind::Down || KIND == GemmKind::Dx) {
    const int x = ti.n0 + 128 * rank + 32 * q;
    for (int j = 0; j < nch; ++j) {
      uint32_t r[32];
      tmem_ld32(tb + 32 * j, r);
      tmem_ld_wait(r);
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
      uint8_t* buf = ring_next<R16, 2048>(stg, ring, lane);
      stage_16_col(buf, lane, v, false);
      store_box(&p.mapO0, buf, x, ti.m0 + 32 * j, lane, false);
    }
    if (ti.tail_n < kBM)
      store_zero_rows(&p.mapO0, stage_zero<R16, 2048>(stg, ring, lane), x, ti, lane);
    return true;
  } else if constexpr (KIND == GemmKind::DA) {
    const int x = ti.n0 + 128 * rank + 32 * q;
    const bool want_lo = dw_compensated(p, ti.e);
    const float fa = pow2f(kDAExp - load_bwd_exps(p.maxabs).ey);
    bool ovf = false;
    for (int j = 0; j < nch; ++j) {
      // router weight of row `lane`, times dA's power-of-two scale (exact)
      const float wl = __ldg(p.w_perm + ti.m0 + 32 * j + lane) * fa;
      uint32_t r[32];
      tmem_ld32(tb + 32 * j, r);
      tmem_ld_wait(r);
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __shfl_sync(0xffffffffu, wl, i) * __uint_as_float(r[i]);
      ovf |= f16_overflows(v);
      uint8_t* buf = ring_next<R16, 2048>(stg, ring, lane);
      stage_16_col(buf, lane, v, true);
      store_box(&p.mapO0, buf, x, ti.m0 + 32 * j, lane, false);
      if (want_lo) {
        to_f16_residual(v);
        uint8_t* lb = ring_next<R16, 2048>(stg, ring, lane);
        stage_16_col(lb, lane, v, true);
        store_box(&p.mapO1, lb, x, ti.m0 + 32 * j, lane, false);
      }
    }
    if (ti.tail_n < kBM) {
      const uint8_t* z = stage_zero<R16, 2048>(stg, ring, lane);
      store_zero_rows(&p.mapO0, z, x, ti, lane);
      if (want_lo) store_zero_rows(&p.mapO1, z, x, ti, lane);
    }
    report_f16_overflow(p, ovf);
    return true;
  } else {
    const int pi = q & 1;
    float* xbuf = reinterpret_cast<float*>(stg_base + pi * Tr::kEpiBytes);
    if (q >= 2) {   // up warp
      if (lane == 0) bulk_wait_read<0>();   // its staging is now the exchange buffer
      __syncwarp();
      for (int j = 0; j < nch; ++j) {
        int ok = 1;
        if (lane == 0)
          ok = mbar_wait(&bars->xempty[pi], xph ^ 1u, abort, p.err, kDevTimeoutEpilogue);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return false;
        uint32_t r[32];
        tmem_ld32(tb + 32 * j, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int i = 0; i < 32; ++i) xbuf[i * 32 + lane] = __uint_as_float(r[i]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->xfull[pi]);
        xph ^= 1u;
      }
      // the staging buffer goes back to this warp's store ring with the next tile: the gate
      // warp must have read the last chunk out of it first
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait(&bars->xempty[pi], xph ^ 1u, abort, p.err, kDevTimeoutEpilogue);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      return ok != 0;
    }
    // gate warp: act columns f0 .. f0+31
    const int f0 = ti.n0 + 64 * rank + 32 * pi;
    bool want_lo = false;
    bool ovf = false;
    float fw = 1.f, fh = 1.f, fb = 1.f;   // backward: scales of w*act, dH fp16, dH bf16
    if constexpr (KIND == GemmKind::BwdGU) {
      want_lo = dw_compensated(p, ti.e);
      const BwdExps sc = load_bwd_exps(p.maxabs);
      fw = pow2f(kActExp - 2 * sc.ex);
      fh = pow2f(kDHExp - kDAExp - sc.ex);   // dA arrives scaled by 2^(kDAExp - ey)
      fb = pow2f(sc.ey - kDAExp);
    }
    for (int j = 0; j < nch; ++j) {
      const int row0 = ti.m0 + 32 * j;
      uint32_t g[32];
      tmem_ld32(tb + 32 * j, g);
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&bars->xfull[pi], xph, abort, p.err, kDevTimeoutEpilogue);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      tmem_ld_wait(g);
      if (!ok) return false;
      float u[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) u[i] = xbuf[i * 32 + lane];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->xempty[pi]);
      xph ^= 1u;
      float v[32];
      if constexpr (KIND == GemmKind::GateUp) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float gv = __uint_as_float(g[i]);
          v[i] = gv * sigmoidf_fast(gv) * u[i];
        }
        uint8_t* buf = ring_next<R16, 2048>(stg, ring, lane);
        stage_16_col(buf, lane, v, false);
        store_box(&p.mapO0, buf, f0, row0, lane, false);
      } else {
        const float wl = __ldg(p.w_perm + row0 + lane) * fw;
        const unsigned short* da = reinterpret_cast<const unsigned short*>(p.dA) +
                                   static_cast<size_t>(row0) * p.I + f0 + lane;
        float d[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
          d[i] = __half2float(__ushort_as_half(__ldg(da + static_cast<size_t>(i) * p.I)));
        if (want_lo) {   // dA's fp16 residual, for experts with compensated dW operands
          const unsigned short* dl = reinterpret_cast<const unsigned short*>(p.dA_lo) +
                                     static_cast<size_t>(row0) * p.I + f0 + lane;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            d[i] += __half2float(__ushort_as_half(__ldg(dl + static_cast<size_t>(i) * p.I)));
        }
        // w * act (scaled fp16; dW_down operand)
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float gv = __uint_as_float(g[i]);
          v[i] = __shfl_sync(0xffffffffu, wl, i) * gv * sigmoidf_fast(gv) * u[i];
        }
        ovf |= f16_overflows(v);
        uint8_t* b0 = ring_next<R16, 2048>(stg, ring, lane);
        stage_16_col(b0, lane, v, true);
        store_box(&p.mapO0, b0, f0, row0, lane, false);
        if (want_lo) {
          to_f16_residual(v);
          uint8_t* c0 = ring_next<R16, 2048>(stg, ring, lane);
          stage_16_col(c0, lane, v, true);
          store_box(&p.mapO3, c0, f0, row0, lane, false);
        }
        // dG = dA U silu'(G): bf16 unscaled (dX operand), fp16 scaled (dW operand)
        float vs[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float gv = __uint_as_float(g[i]);
          const float sg = sigmoidf_fast(gv);
          const float dg = d[i] * u[i] * sg * (1.0f + gv * (1.0f - sg));
          v[i] = dg * fb;
          vs[i] = dg * fh;
        }
        uint8_t* b1 = ring_next<R16, 2048>(stg, ring, lane);
        stage_16_col(b1, lane, v, false);
        store_box(&p.mapO1, b1, f0, row0, lane, false);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = vs[i];
        ovf |= f16_overflows(v);
        uint8_t* b2 = ring_next<R16, 2048>(stg, ring, lane);
        stage_16_col(b2, lane, v, true);
        store_box(&p.mapO2, b2, f0, row0, lane, false);
        if (want_lo) {
          to_f16_residual(v);
          uint8_t* c1 = ring_next<R16, 2048>(stg, ring, lane);
          stage_16_col(c1, lane, v, true);
          store_box(&p.mapO4, c1, f0, row0, lane, false);
        }
        // dU = dA silu(G)
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float gv = __uint_as_float(g[i]);
          const float du = d[i] * gv * sigmoidf_fast(gv);
          v[i] = du * fb;
          vs[i] = du * fh;
        }
        uint8_t* b3 = ring_next<R16, 2048>(stg, ring, lane);
        stage_16_col(b3, lane, v, false);
        store_box(&p.mapO1, b3, p.I + f0, row0, lane, false);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = vs[i];
        ovf |= f16_overflows(v);
        uint8_t* b4 = ring_next<R16, 2048>(stg, ring, lane);
        stage_16_col(b4, lane, v, true);
        store_box(&p.mapO2, b4, p.I + f0, row0, lane, false);
        if (want_lo) {
          to_f16_residual(v);
          uint8_t* c2 = ring_next<R16, 2048>(stg, ring, lane);
          stage_16_col(c2, lane, v, true);
          store_box(&p.mapO4, c2, p.I + f0, row0, lane, false);
        }
      }
    }
    if (ti.tail_n < kBM) {
      const uint8_t* z = stage_zero<R16, 2048>(stg, ring, lane);
      store_zero_rows(&p.mapO0, z, f0, ti, lane);
      if constexpr (KIND == GemmKind::BwdGU) {
        store_zero_rows(&p.mapO1, z, f0, ti, lane);
        store_zero_rows(&p.mapO1, z, p.I + f0, ti, lane);
        store_zero_rows(&p.mapO2, z, f0, ti, lane);
        store_zero_rows(&p.mapO2, z, p.I + f0, ti, lane);
        if (want_lo) {
          store_zero_rows(&p.mapO3, z, f0, ti, lane);
          store_zero_rows(&p.mapO4, z, f0, ti, lane);
          store_zero_rows(&p.mapO4, z, p.I + f0, ti, lane);
        }
      }
    }
    if constexpr (KIND == GemmKind::BwdGU) report_f16_overflow(p, ovf);
    return true;
  }
}

// Backward gate/up epilogue, one 32-column chunk c of a regular tile: recomputed G, U from
// TMEM and dA from memory give w*act (scaled fp16), dG and dU (bf16 and scaled fp16) and,
// for experts with compensated dW operands (LO), the fp16 residuals of the three fp16
// outputs.  `ovf` collects fp16 overflow bits (see f16x2_overflow_bits).
template <int R16, bool LO>
__device__ __forceinline__ void bwd_gu_chunk(const GemmParams& p, uint32_t tb, int c,
                                             const uint4* da_row, const uint4* dl_row, float wr,
                                             float fh, float fb, uint8_t* stg, int& ring, int row,
                                             int lane, uint32_t& ovf, int n0) {
  uint4 d4[4], l4[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) d4[i] = __ldg(da_row + 4 * c + i);   // w-scaled dA, fp16
  if constexpr (LO) {
#pragma unroll
    for (int i = 0; i < 4; ++i) l4[i] = __ldg(dl_row + 4 * c + i);   // its residual
  }
  uint32_t g[32], u[32];
  tmem_ld32(tb + 32 * c, g);
  tmem_ld32(tb + 128 + 32 * c, u);
  tmem_ld_wait(g);
  tmem_ld_after_wait(u);
  const __half2* h2 = reinterpret_cast<const __half2*>(d4);
  const __half2* l2 = reinterpret_cast<const __half2*>(l4);
  uint32_t pa[16], pg[16], pu[16], pg16[16], pu16[16], la[16], lg[16], lu[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float2 da = __half22float2(h2[i]);   // dA of this pair of columns (plus its residual)
    if constexpr (LO) {
      const float2 dl = __half22float2(l2[i]);
      da.x += dl.x;
      da.y += dl.y;
    }
    float r[2][3];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float gv = __uint_as_float(g[2 * i + h]);
      const float uv = __uint_as_float(u[2 * i + h]);
      const float dv = h ? da.y : da.x;
      const float sg = sigmoidf_fast(gv);
      const float si = gv * sg;
      r[h][0] = wr * si * uv;                              // w * act (dW_down operand)
      r[h][1] = dv * uv * sg * (1.0f + gv * (1.0f - sg));  // dG (scaled as dA)
      r[h][2] = dv * si;                                   // dU (scaled as dA)
    }
    pa[i] = pack_f16x2(r[0][0], r[1][0]);
    pg[i] = pack_bf16x2(r[0][1] * fb, r[1][1] * fb);
    pu[i] = pack_bf16x2(r[0][2] * fb, r[1][2] * fb);
    const float g0 = r[0][1] * fh, g1 = r[1][1] * fh;
    const float u0 = r[0][2] * fh, u1 = r[1][2] * fh;
    pg16[i] = pack_f16x2(g0, g1);
    pu16[i] = pack_f16x2(u0, u1);
    ovf |= f16x2_overflow_bits(pa[i]) | f16x2_overflow_bits(pg16[i]) |
           f16x2_overflow_bits(pu16[i]);
    if constexpr (LO) {
      la[i] = f16x2_residual(pa[i], r[0][0], r[1][0]);
      lg[i] = f16x2_residual(pg16[i], g0, g1);
      lu[i] = f16x2_residual(pu16[i], u0, u1);
    }
  }
  const int col = n0 + 32 * c;
  // boxes are staged in groups of up to R16 (the ring) and fenced once per group
  ring_reserve<R16, 3>(lane);
  uint8_t* b0 = ring_slot<R16, 2048>(stg, ring);
  stage_16_row(b0, lane, pa);
  uint8_t* b1 = ring_slot<R16, 2048>(stg, ring);
  stage_16_row(b1, lane, pg);
  uint8_t* b2 = ring_slot<R16, 2048>(stg, ring);
  stage_16_row(b2, lane, pu);
  fence_boxes();
  issue_box(&p.mapO0, b0, col, row, lane);        // w*act, fp16
  issue_box(&p.mapO1, b1, col, row, lane);        // dG, bf16
  issue_box(&p.mapO1, b2, p.I + col, row, lane);  // dU, bf16
  __syncwarp();
  ring_reserve<R16, 2>(lane);
  uint8_t* b3 = ring_slot<R16, 2048>(stg, ring);
  stage_16_row(b3, lane, pg16);
  uint8_t* b4 = ring_slot<R16, 2048>(stg, ring);
  stage_16_row(b4, lane, pu16);
  fence_boxes();
  issue_box(&p.mapO2, b3, col, row, lane);        // dG, fp16
  issue_box(&p.mapO2, b4, p.I + col, row, lane);  // dU, fp16
  __syncwarp();
  if constexpr (LO) {
    ring_reserve<R16, 3>(lane);
    uint8_t* c0 = ring_slot<R16, 2048>(stg, ring);
    stage_16_row(c0, lane, la);
    uint8_t* c1 = ring_slot<R16, 2048>(stg, ring);
    stage_16_row(c1, lane, lg);
    uint8_t* c2 = ring_slot<R16, 2048>(stg, ring);
    stage_16_row(c2, lane, lu);
    fence_boxes();
    issue_box(&p.mapO3, c0, col, row, lane);        // w*act residual
    issue_box(&p.mapO4, c1, col, row, lane);        // dG residual
    issue_box(&p.mapO4, c2, p.I + col, row, lane);  // dU residual
    __syncwarp();
  }
}

// ------------------------------------------------------------------ epilogue
template <GemmKind KIND>
__device__ __forceinline__ void epilogue(const GemmParams& p, GemmBarriers* bars, uint8_t* stg,
                                         uint32_t tmem_base, const int* pfx, int warp, int lane,
                                         volatile int* abort) {
  using Tr = KindTraits<KIND>;
  constexpr int R16 = Tr::kRing16;
  constexpr int R32 = Tr::kRing32;
  const int q = warp & 3;  // TMEM lane quarter this warp may access
  int ring = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  const int rank = Tr::kPair ? static_cast<int>(cluster_ctarank()) : 0;
  // accumulator releases go to the even CTA, whose MMA issuer waits on them
  const uint32_t tempty0 = Tr::kPair ? mapa_shared(smem_u32(&bars->tempty[0]), 0) : 0u;
  uint8_t* stg_base = stg - (warp - 2) * Tr::kEpiBytes;
  uint32_t xph = 0;   // swapped gate/up tails: exchange phase of this warp's pair
  const int ntiles = num_tiles<KIND>(p, pfx);
  for (int t = first_tile<KIND>(); t < ntiles; t += tile_stride<KIND>()) {
    const TileInfo ti = decode_tile<KIND>(p, t, pfx, rank);
    const int row = ti.m0 + 32 * q;   // first of this warp's 32 rows; lane owns row + lane
    if constexpr (Tr::kIsDw) {
      if (ti.nkb == 0 && ti.split) continue;   // a chunk without real rows adds nothing
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

    bool swapped = false;
    if constexpr (Tr::kPair) {
      if (ti.swap) {
        if (!epilogue_swap<KIND>(p, bars, stg, stg_base, tb, ti, q, lane, rank, ring, xph, abort))
          return;
        swapped = true;
      }
    }
    if (!swapped && !ti.ghost) {   // a ghost half only drains its accumulator
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
        // router weight of this thread's row times dA's power-of-two scale (exact)
        const float wr = __ldg(p.w_perm + row + lane) * pow2f(kDAExp - load_bwd_exps(p.maxabs).ey);
        const bool want_lo =
            dw_compensated(p, ti.e);
        const int nch = p.tile_n / 32;
        uint32_t ovf = 0;
        for (int c = 0; c < nch; ++c) {
          uint32_t r[32];
          tmem_ld32(tb + 32 * c, r);
          tmem_ld_wait(r);
          uint32_t pk[16], lo[16];
  #pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float v0 = wr * __uint_as_float(r[2 * i]);
            const float v1 = wr * __uint_as_float(r[2 * i + 1]);
            pk[i] = pack_f16x2(v0, v1);
            ovf |= f16x2_overflow_bits(pk[i]);
            if (want_lo) lo[i] = f16x2_residual(pk[i], v0, v1);
          }
          uint8_t* buf = ring_next<R16, 2048>(stg, ring, lane);
          stage_16_row(buf, lane, pk);
          store_box(&p.mapO0, buf, ti.n0 + 32 * c, row, lane, false);
          if (want_lo) {   // the fp16 residual, for experts with compensated dW operands
            uint8_t* lb = ring_next<R16, 2048>(stg, ring, lane);
            stage_16_row(lb, lane, lo);
            store_box(&p.mapO1, lb, ti.n0 + 32 * c, row, lane, false);
          }
        }
        report_f16_overflow(p, (ovf & 0x80008000u) != 0u);
      } else if constexpr (KIND == GemmKind::BwdGU) {
        const int my_row = row + lane;
        const BwdExps sc = load_bwd_exps(p.maxabs);
        // w * act scaled by 2^(kActExp - 2 ex); dA arrives scaled by 2^(kDAExp - ey), so dG
        // and dU take 2^(kDHExp - kDAExp - ex) for their fp16 copies and 2^(ey - kDAExp) back
        // to their true values for the bf16 ones
        const float wr = __ldg(p.w_perm + my_row) * pow2f(kActExp - 2 * sc.ex);
        const float fh = pow2f(kDHExp - kDAExp - sc.ex);
        const float fb = pow2f(sc.ey - kDAExp);
        uint32_t ovf = 0;
        // rows of an expert with compensated dW operands also get the fp16 residuals
        const bool want_lo =
            dw_compensated(p, ti.e);
        const uint4* da_row =
            reinterpret_cast<const uint4*>(p.dA + static_cast<size_t>(my_row) * p.I + ti.n0);
        const uint4* dl_row =
            reinterpret_cast<const uint4*>(p.dA_lo + static_cast<size_t>(my_row) * p.I + ti.n0);
        for (int c = 0; c < 4; ++c) {
          if (want_lo) bwd_gu_chunk<R16, true>(p, tb, c, da_row, dl_row, wr, fh, fb, stg, ring, row,
                                             lane, ovf, ti.n0);
          else bwd_gu_chunk<R16, false>(p, tb, c, da_row, dl_row, wr, fh, fb, stg, ring, row, lane,
                                        ovf, ti.n0);
        }
        report_f16_overflow(p, (ovf & 0x80008000u) != 0u);
      } else {  // DwGU, DwD: fp32 out, plain store or split-K reduce-add
        // undo the operands' power-of-two scales (exact): dW_gate|up = x16^T dH16 carries
        // 2^(kX16Exp - ex) 2^(kDHExp - ey - ex); dW_down = wact16^T dy16 carries
        // 2^(kActExp - 2 ex) 2^(kDy16Exp - ey).  Two factors, each a normal fp32 power of
        // two for |ex|, |ey| <= 59 (their product alone could leave fp32's range).
        const BwdExps sc = load_bwd_exps(p.maxabs);
        float f1, f2;
        if constexpr (KIND == GemmKind::DwGU) {
          f1 = pow2f(sc.ex - kX16Exp);
          f2 = pow2f(sc.ex + sc.ey - kDHExp);
        } else {
          f1 = pow2f(2 * sc.ex - kActExp);
          f2 = pow2f(sc.ey - kDy16Exp);
        }
        for (int c = 0; c < 8; ++c) {
          uint32_t r[32];
          tmem_ld32(tb + 32 * c, r);
          tmem_ld_wait(r);
          float v[32];
  #pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * f1 * f2;
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
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if constexpr (Tr::kPair) mbar_arrive_cluster(tempty0 + 8u * static_cast<uint32_t>(acc));
      else mbar_arrive(&bars->tempty[acc]);
    }
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
  }
}

// ------------------------------------------------------------------ kernel
template <GemmKind KIND>
__global__ void __launch_bounds__(kGemmThreads, 1) k_grouped_gemm(const __grid_constant__ GemmParams p) {
  using Tr = KindTraits<KIND>;
  extern __shared__ uint8_t smem_raw[];
  // identical offsets in both CTAs of a pair: the even CTA's descriptors address both
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  GemmBarriers* bars = reinterpret_cast<GemmBarriers*>(smem);
  uint8_t* stages = smem + 1024;
  uint8_t* staging = stages + Tr::kStages * Tr::kStageBytes;
  int* pfx = reinterpret_cast<int*>(staging + kEpiWarps * Tr::kEpiBytes);
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
      // a pair's accumulators are released by the epilogue warps of both CTAs
      mbar_init(&bars->tempty[i], Tr::kPair ? 2 * kEpiWarps : kEpiWarps);
      mbar_init(&bars->xfull[i], 1);
      mbar_init(&bars->xempty[i], 1);
    }
    bars->abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.mapA0);
    tma_prefetch_desc(&p.mapB0);
  }
  if constexpr (Tr::kPair) build_pair_prefix(p, pfx);   // contains a __syncthreads
  if (warp == 1) {
    if constexpr (Tr::kPair) {
      tmem_alloc_pair(&bars->tmem_addr, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&bars->tmem_addr, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  // the peer's barriers must be initialised before any copy or arrival targets them
  if constexpr (Tr::kPair) cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_addr;

  if (warp == 0) {
    if (lane == 0) produce<KIND>(p, bars, stages, pfx, abort);
  } else if (warp == 1) {
    if (lane == 0) mma_issue<KIND>(p, bars, stages, tmem_base, pfx, abort);
  } else {
    epilogue<KIND>(p, bars, staging + (warp - 2) * Tr::kEpiBytes, tmem_base, pfx, warp, lane,
                   abort);
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
  // neither CTA of a pair frees TMEM or exits while the other may still reach its memory
  if constexpr (Tr::kPair) cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (Tr::kPair) tmem_dealloc_pair(tmem_base, kTmemCols);
    else tmem_dealloc(tmem_base, kTmemCols);
  }
}

// `max_tiles` bounds the device-side tile count (pair kinds: pair tiles).
template <GemmKind KIND>
cudaError_t launch_gemm_kind(const GemmParams& p, int max_tiles, int num_sms, cudaStream_t s) {
  using Tr = KindTraits<KIND>;
  constexpr int kSmem = Tr::kSmemBytes;
  static_assert(kSmem <= 232448, "shared memory budget");
  static bool configured[64] = {};
  static int max_pairs[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_grouped_gemm<KIND>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  if constexpr (Tr::kPair) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (max_pairs[dev] == 0) {
      // pairs that fit on the GPU at once (clusters are placed within a GPC)
      cfg.gridDim = dim3(2 * (num_sms / 2));
      int n = 0;
      cudaError_t e = cudaOccupancyMaxActiveClusters(&n, k_grouped_gemm<KIND>, &cfg);
      if (e != cudaSuccess) return e;
      if (n < 1) return cudaErrorInvalidConfiguration;
      max_pairs[dev] = n;
    }
    int pairs = max_tiles < max_pairs[dev] ? max_tiles : max_pairs[dev];
    if (pairs < 1) pairs = 1;
    cfg.gridDim = dim3(2 * pairs);
    return cudaLaunchKernelEx(&cfg, k_grouped_gemm<KIND>, p);
  } else {
    int grid = max_tiles < num_sms ? max_tiles : num_sms;
    if (grid < 1) grid = 1;
    k_grouped_gemm<KIND><<<grid, kGemmThreads, kSmem, s>>>(p);
    return cudaGetLastError();
  }
}

}  // namespace moe
