// C ABI of libmoe_gb300: argument validation, workspace layout, TMA descriptor
// encoding and the launch sequence of every entry point.  No allocation, no host
// synchronisation on the compute path.
#include <atomic>
#include <mutex>
#include <vector>

#include "internal.h"
#include "moe_gb300.h"

#define MOE_EXPORT extern "C" __attribute__((visibility("default")))

namespace moe {

// ------------------------------------------------------------------ launch bookkeeping
static const char* const kKernelNames[kNumKernelIds] = {
    "route_count", "route_scan", "route_scatter", "gather_x",   "gemm_gateup_swiglu",
    "gemm_down",   "combine",    "bwd_prep_rows", "gemm_dA",    "gemm_bwd_gateup",
    "gemm_dx",     "dw_prep",    "gemm_dw_gateup", "gemm_dw_down", "router_topk",
    "router_weight_grad", "router_backward", "route_permute", "bwd_prep_pad", "combine_dx"};

const char* kernel_name(int id) {
  return (id >= 0 && id < kNumKernelIds) ? kKernelNames[id] : nullptr;
}

namespace {
std::atomic<long long> g_launch_total{0};
std::atomic<long long> g_launch_by_id[kNumKernelIds];
std::mutex g_timing_mu;
std::atomic<unsigned long long> g_timing_mask{0};   // bit id: bracket kernel id with events
struct TimingRec {
  int id;
  cudaEvent_t a, b;
};
std::vector<TimingRec> g_recs;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t pool_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
}  // namespace

LaunchScope::LaunchScope(int id_, cudaStream_t s) : id(id_), stream(s), slot(-1) {
  g_launch_total.fetch_add(1, std::memory_order_relaxed);
  if (id >= 0 && id < kNumKernelIds) g_launch_by_id[id].fetch_add(1, std::memory_order_relaxed);
  if (id >= 0 && id < kNumKernelIds && ((g_timing_mask.load() >> id) & 1ull)) {
    std::lock_guard<std::mutex> lk(g_timing_mu);
    TimingRec r{id, pool_event(), pool_event()};
    cudaEventRecord(r.a, s);
    g_recs.push_back(r);
    slot = static_cast<int>(g_recs.size()) - 1;
  }
}

LaunchScope::~LaunchScope() {
  if (slot >= 0) {
    std::lock_guard<std::mutex> lk(g_timing_mu);
    cudaEventRecord(g_recs[slot].b, stream);
  }
}

// ------------------------------------------------------------------ device facts
struct DevFacts {
  bool init = false;
  int num_sms = 0;
  int major = 0, minor = 0;
};
static DevFacts g_dev[64];
static std::mutex g_dev_mu;

static const DevFacts* dev_facts() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevFacts& f = g_dev[dev];
  if (!f.init) {
    if (cudaDeviceGetAttribute(&f.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return nullptr;
    cudaDeviceGetAttribute(&f.major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&f.minor, cudaDevAttrComputeCapabilityMinor, dev);
    f.init = true;
  }
  return &f;
}

// ------------------------------------------------------------------ side stream
// The backward reduces dx_perm to tokens (when the caller asks it to) on a second stream of
// the library's own, beside its weight-gradient GEMMs: the reduction's blocks fit on an SM
// next to a GEMM CTA (no shared memory, few registers) and use HBM bandwidth the
// latency-bound GEMMs leave idle.  The stream has the lowest priority, so that the GEMMs'
// CTAs are placed first.  (Running the fp16 operand copies beside the token-row GEMMs the
// same way measured slower: those GEMMs lost more time than the copies took.)  One side
// stream and three events per device, created by the first backward on it; the enqueue
// sequence of a backward holds the mutex, so concurrent callers cannot interleave their
// event records.
struct SideStream {
  bool init = false;
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr, spare = nullptr;
};
static SideStream g_side[64];
static std::mutex g_side_mu;

static SideStream* side_stream(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  SideStream& ss = g_side[dev];
  if (!ss.init) {
    int least = 0, greatest = 0;
    if ((*err = cudaDeviceGetStreamPriorityRange(&least, &greatest)) != cudaSuccess ||
        (*err = cudaStreamCreateWithPriority(&ss.s, cudaStreamNonBlocking, least)) != cudaSuccess)
      return nullptr;
    cudaEvent_t* evs[3] = {&ss.fork, &ss.join, &ss.spare};
    for (cudaEvent_t* e : evs)
      if ((*err = cudaEventCreateWithFlags(e, cudaEventDisableTiming)) != cudaSuccess) return nullptr;
    ss.init = true;
  }
  return &ss;
}

// Makes `to` wait for the work enqueued on `from` so far.
static cudaError_t stream_after(cudaStream_t to, cudaStream_t from, cudaEvent_t ev) {
  cudaError_t e = cudaEventRecord(ev, from);
  return e == cudaSuccess ? cudaStreamWaitEvent(to, ev, 0) : e;
}

// ------------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

enum class Elem { BF16, F16, F32 };

// 2-D map over a row-major [outer, inner] tensor with a box of [box_outer, box_inner].
static bool make_map(CUtensorMap* m, Elem el, const void* base, uint64_t inner, uint64_t outer,
                     uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const bool f32 = el == Elem::F32;
  const uint64_t esize = f32 ? 4 : 2;
  const CUtensorMapDataType dt = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                     : (el == Elem::F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * esize};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Operand load maps (128-byte swizzle, 64-element inner box) and store maps.
static bool map_kmajor(CUtensorMap* m, const void* b, uint64_t inner, uint64_t outer, uint32_t rows) {
  return make_map(m, Elem::BF16, b, inner, outer, 64, rows, CU_TENSOR_MAP_SWIZZLE_128B);
}
// MN-major operand map over a row-major [outer, inner] tensor viewed in 3-D as
// (64 columns, rows, inner / 64 column atoms), with a box of `atoms` 64x64 atoms: one TMA
// load fills the atoms at 8 KB strides, the layout the MN-major descriptors expect.
static bool map_mnmajor(CUtensorMap* m, const void* b, uint64_t inner, uint64_t outer,
                        uint32_t atoms, Elem el = Elem::BF16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || inner % 64 != 0) return false;
  const CUtensorMapDataType dt = el == Elem::F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[3] = {64, outer, inner / 64};
  cuuint64_t strides[2] = {inner * 2, 128};
  cuuint32_t box[3] = {64, 64, atoms};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(b), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
static bool map_store_16(CUtensorMap* m, const void* b, uint64_t inner, uint64_t outer,
                         Elem el = Elem::BF16) {
  return make_map(m, el, b, inner, outer, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}
static bool map_store_f32(CUtensorMap* m, const void* b, uint64_t inner, uint64_t outer) {
  return make_map(m, Elem::F32, b, inner, outer, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B);
}

// ------------------------------------------------------------------ sizes
bool basic_sizes_ok(int T, int K, int E, int align) {
  if (T < 0 || K < 1 || K > 32 || E < 1 || E > kMaxExperts || align < 1) return false;
  const long long R = static_cast<long long>(T) * K;
  const long long cap = R + static_cast<long long>(E) * (align - 1) + align;
  return R < (1ll << 31) && cap < (1ll << 31);
}

size_t capacity_of(int T, int K, int E, int align) {
  const size_t R = static_cast<size_t>(T) * K;
  const size_t c = R + static_cast<size_t>(E) * (align - 1);
  return (c + align - 1) / align * align;
}

static size_t up1k(size_t v) { return (v + 1023) & ~static_cast<size_t>(1023); }

struct WsLayout {
  size_t chunk_counts, dw_prefix, inv, act, dh, dyp, dh16, dyp16, xp16, act_lo, dh16_lo, da,
      da_lo, total;
};

// header | routing chunk counters | dW split prefix | slot -> sorted row [T*K] (backward
// row preparation) | act | dH | dy_perm | dH fp16 |
// dy_perm fp16 | x_perm fp16 | w*act fp16 residual | dH fp16 residual (the residuals
// are written only for experts whose weight gradient takes compensated operands) |
// router-weighted dA fp16 | its fp16 residual (those experts only)
static WsLayout ws_layout(int T, int K, int E, int D, int I, int align) {
  WsLayout L;
  const size_t cap = capacity_of(T, K, E, align);
  const size_t nch = static_cast<size_t>(route_num_chunks(T * K));
  size_t o = 1024;
  L.chunk_counts = o;
  o = up1k(o + static_cast<size_t>(E) * nch * 4);
  L.dw_prefix = o;
  o = up1k(o + static_cast<size_t>(E + 1) * 4);
  L.inv = o;
  o = up1k(o + static_cast<size_t>(T) * K * 4);
  L.act = o;
  o = up1k(o + cap * static_cast<size_t>(I) * 2);
  L.dh = o;
  o = up1k(o + cap * static_cast<size_t>(I) * 4);
  L.dyp = o;
  o = up1k(o + cap * static_cast<size_t>(D) * 2);
  L.dh16 = o;
  o = up1k(o + cap * static_cast<size_t>(I) * 4);
  L.dyp16 = o;
  o = up1k(o + cap * static_cast<size_t>(D) * 2);
  L.xp16 = o;
  o = up1k(o + cap * static_cast<size_t>(D) * 2);
  L.act_lo = o;
  o = up1k(o + cap * static_cast<size_t>(I) * 2);
  L.dh16_lo = o;
  o = up1k(o + cap * static_cast<size_t>(I) * 4);
  L.da = o;
  o = up1k(o + cap * static_cast<size_t>(I) * 2);
  L.da_lo = o;
  o = up1k(o + cap * static_cast<size_t>(I) * 2);
  L.total = o;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int check_device() {
  const DevFacts* f = dev_facts();
  if (!f) return MOE_ERR_CUDA;
  if (f->major != 10 || f->minor != 3) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

static bool gemm_shape_ok(int D, int I, int align) {
  return D >= 256 && I >= 128 && D % 256 == 0 && I % 128 == 0 && align % 128 == 0 &&
         static_cast<long long>(D) < (1ll << 24) && static_cast<long long>(I) < (1ll << 24);
}

static int to_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Test hook (moe_debug_drop_next_loads): the next grouped-GEMM launch of this host thread
// issues no loads, so its bounded waits run out and report a timeout.
static thread_local bool t_drop_next_loads = false;
static int take_drop_flag() {
  const bool d = t_drop_next_loads;
  t_drop_next_loads = false;
  return d ? 1 : 0;
}

// ------------------------------------------------------------------ per-shape tuning
struct TuneEntry {
  int T, K, E, D, I;
  int order[5];
  int swap_tails, da_tile_n, dw_chunk_rows;
};

static const TuneEntry kTuneTable[] = {
#include "tuning_table.inc"
};

static moe_tuning_t default_tuning() {
  moe_tuning_t t{};
  for (int i = 0; i < 5; ++i) t.order[i] = 0;
  t.swap_tails = 1;
  t.da_tile_n = 256;
  t.dw_chunk_rows = kDwChunkRows;
  return t;
}

static bool tuning_ok(const moe_tuning_t& t) {
  for (int i = 0; i < 5; ++i)
    if (t.order[i] != 0 && t.order[i] != 1) return false;
  return (t.swap_tails == 0 || t.swap_tails == 1) && (t.da_tile_n == 128 || t.da_tile_n == 256) &&
         t.dw_chunk_rows >= 256 && t.dw_chunk_rows <= 65536 && t.dw_chunk_rows % kBK == 0;
}

static std::mutex g_tune_mu;
static bool g_tune_override_on = false;
static moe_tuning_t g_tune_override;

// The override if set; else the table entry of the same K, E, D, I with the nearest T
// (by ratio; ties: the smaller T); else the defaults.
static moe_tuning_t select_tuning(int T, int K, int E, int D, int I, int* source) {
  {
    std::lock_guard<std::mutex> g(g_tune_mu);
    if (g_tune_override_on) {
      if (source) *source = 2;
      return g_tune_override;
    }
  }
  const TuneEntry* best = nullptr;
  double best_d = 0.0;
  const double tq = T > 0 ? static_cast<double>(T) : 1.0;
  for (const TuneEntry& en : kTuneTable) {
    if (en.T <= 0 || en.K != K || en.E != E || en.D != D || en.I != I) continue;
    const double r = tq > en.T ? tq / en.T : en.T / tq;
    if (!best || r < best_d || (r == best_d && en.T < best->T)) {
      best = &en;
      best_d = r;
    }
  }
  moe_tuning_t t = default_tuning();
  if (best) {
    for (int i = 0; i < 5; ++i) t.order[i] = best->order[i];
    t.swap_tails = best->swap_tails;
    t.da_tile_n = best->da_tile_n;
    t.dw_chunk_rows = best->dw_chunk_rows;
    if (!tuning_ok(t)) t = default_tuning();
  }
  if (source) *source = best ? 1 : 0;
  return t;
}

}  // namespace moe

using namespace moe;

// ------------------------------------------------------------------ exported API
MOE_EXPORT int moe_abi_version(void) { return MOE_ABI_VERSION; }

MOE_EXPORT const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported device or shape";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case MOE_ERR_BAD_INDEX: return "expert id out of range";
    case MOE_ERR_FP16_RANGE: return "value outside the range of the backward's scaled fp16 operands";
    default: return "unknown status";
  }
}

// Workspace header: [0] device error word; at kMaxAbsOffset the backward's {max|x|, max|dY|}
// (fp32 bits); at kRouteSyncOffset the fused routing kernel's grid-barrier counters
// {arrivals, exits} (zero between launches).
constexpr size_t kRouteSyncOffset = 512;

MOE_EXPORT size_t moe_capacity(int T, int K, int E, int align) {
  if (!basic_sizes_ok(T, K, E, align)) return 0;
  return capacity_of(T, K, E, align);
}

MOE_EXPORT size_t moe_workspace_bytes(int T, int K, int E, int D, int I, int align) {
  if (!basic_sizes_ok(T, K, E, align) || D < 0 || I < 0) return 0;
  return ws_layout(T, K, E, D, I, align).total;
}

MOE_EXPORT int moe_workspace_init(void* workspace, void* stream) {
  if (!workspace) return MOE_ERR_INVALID_ARG;
  return to_status(cudaMemsetAsync(workspace, 0, 1024, static_cast<cudaStream_t>(stream)));
}

MOE_EXPORT int moe_route_permute(const int32_t* topk_ids, const float* topk_w,
                                 const moe_bf16_t* x, int T, int K, int E, int D, int align,
                                 int32_t* counts, int32_t* offsets, int32_t* perm_src,
                                 int32_t* inv_perm, float* w_perm, moe_bf16_t* x_perm,
                                 void* workspace, void* stream) {
  if (!basic_sizes_ok(T, K, E, align)) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets || !perm_src || !w_perm || !workspace) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_ids || !topk_w || !inv_perm)) return MOE_ERR_INVALID_ARG;
  if (x && (!x_perm || D <= 0 || D % 8 != 0 || !aligned16(x) || !aligned16(x_perm)))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return MOE_ERR_INVALID_ARG;
  int st = check_device();
  if (st != MOE_OK) return st;
  const WsLayout L = ws_layout(T, K, E, D > 0 ? D : 0, 0, align);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int cap = static_cast<int>(capacity_of(T, K, E, align));
  return to_status(launch_route(topk_ids, topk_w, x, T, K, E, D, align, cap, counts, offsets,
                                perm_src, inv_perm, w_perm, x_perm,
                                reinterpret_cast<int32_t*>(ws + L.chunk_counts),
                                reinterpret_cast<int*>(ws),
                                reinterpret_cast<unsigned*>(ws + kRouteSyncOffset),
                                static_cast<cudaStream_t>(stream)));
}

MOE_EXPORT int moe_combine(const moe_bf16_t* src_perm, const int32_t* inv_perm,
                           const float* topk_w, int T, int K, int D, moe_bf16_t* out,
                           void* stream) {
  if (T < 0 || K < 1 || K > 32 || D <= 0 || D % 8 != 0) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!src_perm || !inv_perm || !out)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!aligned16(src_perm) || !aligned16(out))) return MOE_ERR_INVALID_ARG;
  if (static_cast<long long>(T) * K >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
  int st = check_device();
  if (st != MOE_OK) return st;
  return to_status(launch_combine(src_perm, inv_perm, topk_w, T, K, D, out,
                                  static_cast<cudaStream_t>(stream)));
}

MOE_EXPORT int moe_expert_mlp_fwd(const moe_bf16_t* x_perm, const moe_bf16_t* w_gate,
                                  const moe_bf16_t* w_up, const moe_bf16_t* w_down,
                                  const int32_t* offsets, const int32_t* counts, int T, int K,
                                  int E, int D, int I, int align, moe_bf16_t* y_perm,
                                  void* workspace, void* stream) {
  if (!basic_sizes_ok(T, K, E, align)) return MOE_ERR_INVALID_ARG;
  if (!gemm_shape_ok(D, I, align)) return MOE_ERR_UNSUPPORTED;
  if (!x_perm || !w_gate || !w_up || !w_down || !offsets || !y_perm || !workspace)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_perm) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
      !aligned16(y_perm) || !aligned16(workspace))
    return MOE_ERR_INVALID_ARG;
  int st = check_device();
  if (st != MOE_OK) return st;
  const DevFacts* f = dev_facts();
  const WsLayout L = ws_layout(T, K, E, D, I, align);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const uint64_t cap = capacity_of(T, K, E, align);
  void* act = ws + L.act;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // token-row GEMMs run on CTA pairs: at most (row tiles + E) / 2 pairs of 256 rows
  const int pairs_max = static_cast<int>((cap / kBM + E + 1) / 2);
  const moe_tuning_t tun = select_tuning(T, K, E, D, I, nullptr);

  GemmParams p{};
  p.offsets = offsets;
  p.counts = counts;
  p.err = reinterpret_cast<int*>(ws);
  p.E = E; p.D = D; p.I = I;
  p.order = tun.order[MOE_GEMM_GATE_UP];
  p.swap_tails = tun.swap_tails;
  p.dw_chunk_rows = tun.dw_chunk_rows;
  // gate/up + SwiGLU (A1, B2, B3: the token rows and one-atom weight boxes of the
  // swapped tail tiles)
  bool ok = map_kmajor(&p.mapA0, x_perm, D, cap, 128) &&
            map_kmajor(&p.mapA1, x_perm, D, cap, 64) &&
            map_mnmajor(&p.mapB0, w_gate, I, static_cast<uint64_t>(E) * D, 2) &&
            map_mnmajor(&p.mapB1, w_up, I, static_cast<uint64_t>(E) * D, 2) &&
            map_mnmajor(&p.mapB2, w_gate, I, static_cast<uint64_t>(E) * D, 1) &&
            map_mnmajor(&p.mapB3, w_up, I, static_cast<uint64_t>(E) * D, 1) &&
            map_store_16(&p.mapO0, act, I, cap);
  if (!ok) return MOE_ERR_CUDA;
  p.n_tiles = I / 128;
  p.drop_loads = take_drop_flag();
  cudaError_t e;
  {
    LaunchScope ls(kKGemmGateUp, s);
    e = launch_gemm_kind<GemmKind::GateUp>(p, pairs_max * p.n_tiles, f->num_sms, s);
  }
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  // down projection
  GemmParams q{};
  q.offsets = offsets;
  q.counts = counts;
  q.err = p.err;
  q.E = E; q.D = D; q.I = I;
  q.order = tun.order[MOE_GEMM_DOWN];
  q.swap_tails = tun.swap_tails;
  q.dw_chunk_rows = tun.dw_chunk_rows;
  ok = map_kmajor(&q.mapA0, act, I, cap, 128) && map_kmajor(&q.mapA1, act, I, cap, 64) &&
       map_mnmajor(&q.mapB0, w_down, D, static_cast<uint64_t>(E) * I, 2) &&
       map_store_16(&q.mapO0, y_perm, D, cap);
  if (!ok) return MOE_ERR_CUDA;
  q.n_tiles = D / 256;
  {
    LaunchScope ls(kKGemmDown, s);
    e = launch_gemm_kind<GemmKind::Down>(q, pairs_max * q.n_tiles, f->num_sms, s);
  }
  return to_status(e);
}

// The dx reduction the backward runs on its side stream (none when ss is null).
struct SideWork {
  SideStream* ss;
  const moe_bf16_t* dx_perm;
  const int32_t* inv_perm;
  moe_bf16_t* dx;
  int T, K, D;
};

static int bwd_weight_grads(const int32_t* offsets, const int32_t* counts, int* dw_prefix,
                            int* err, const uint32_t* maxabs, int E, int D, int I, uint64_t cap,
                            int chunk, void* act, void* act_lo, void* dh16, void* dh16_lo,
                            moe_bf16_t* xp16, moe_bf16_t* dyp16, float* dw_gate, float* dw_up,
                            float* dw_down, int num_sms, const SideWork& side, cudaStream_t s);

MOE_EXPORT int moe_expert_mlp_bwd(const moe_bf16_t* dy, const moe_bf16_t* x,
                                  const moe_bf16_t* x_perm,
                                  const int32_t* perm_src, const float* w_perm,
                                  const int32_t* offsets, const int32_t* counts,
                                  const moe_bf16_t* w_gate,
                                  const moe_bf16_t* w_up, const moe_bf16_t* w_down, int T, int K,
                                  int E, int D, int I, int align, moe_bf16_t* dx_perm,
                                  float* dw_gate, float* dw_up, float* dw_down,
                                  const int32_t* inv_perm, moe_bf16_t* dx, void* workspace,
                                  void* stream) {
  if (!basic_sizes_ok(T, K, E, align)) return MOE_ERR_INVALID_ARG;
  if (!gemm_shape_ok(D, I, align)) return MOE_ERR_UNSUPPORTED;
  if (!x_perm || !perm_src || !w_perm || !offsets || !w_gate || !w_up || !w_down || !dx_perm ||
      !dw_gate || !dw_up || !dw_down || !workspace || (T > 0 && !dy))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_perm) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
      !aligned16(dx_perm) || !aligned16(dw_gate) || !aligned16(dw_up) || !aligned16(dw_down) ||
      !aligned16(workspace) || (dy && !aligned16(dy)) || (x && !aligned16(x)))
    return MOE_ERR_INVALID_ARG;
  // optional: the reduction of dx_perm to tokens, done inside this call
  if ((dx == nullptr) != (inv_perm == nullptr) || (dx && !aligned16(dx)))
    return MOE_ERR_INVALID_ARG;
  int st = check_device();
  if (st != MOE_OK) return st;
  const DevFacts* f = dev_facts();
  std::unique_lock<std::mutex> side_lock(g_side_mu, std::defer_lock);
  SideStream* ss = nullptr;
  if (dx && T > 0) {
    side_lock.lock();
    cudaError_t se = cudaSuccess;
    ss = side_stream(&se);
    if (!ss) return MOE_ERR_CUDA;
  }
  const WsLayout L = ws_layout(T, K, E, D, I, align);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const uint64_t cap = capacity_of(T, K, E, align);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = reinterpret_cast<int*>(ws);
  void* act = ws + L.act;
  void* dh = ws + L.dh;
  moe_bf16_t* dyp = reinterpret_cast<moe_bf16_t*>(ws + L.dyp);
  int* dw_prefix = reinterpret_cast<int*>(ws + L.dw_prefix);
  const int pairs_max = static_cast<int>((cap / kBM + E + 1) / 2);
  const uint64_t ED = static_cast<uint64_t>(E) * D, EI = static_cast<uint64_t>(E) * I;
  const moe_tuning_t tun = select_tuning(T, K, E, D, I, nullptr);
  const int chunk = tun.dw_chunk_rows;
  cudaError_t e;

  void* dh16 = ws + L.dh16;
  moe_bf16_t* dyp16 = reinterpret_cast<moe_bf16_t*>(ws + L.dyp16);
  moe_bf16_t* xp16 = reinterpret_cast<moe_bf16_t*>(ws + L.xp16);
  void* act_lo = ws + L.act_lo;
  void* dh16_lo = ws + L.dh16_lo;
  uint32_t* maxabs = reinterpret_cast<uint32_t*>(ws + kMaxAbsOffset);

  // 1. max|x| and max|dY| (the power-of-two scales of the fp16 operands), the routed
  //    expert-output gradient rows (unscaled; the router weight is applied to dA in fp32)
  //    and the scaled fp16 operand copies of the weight-gradient GEMMs
  e = launch_bwd_prep_rows(dy, x, x_perm, perm_src, offsets, T, E, K, D, static_cast<int>(cap),
                           reinterpret_cast<int32_t*>(ws + L.inv), dyp, dyp16, xp16, maxabs,
                           err, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  // 2. dA = w * dy_perm W_d^T (scaled in fp32, kept in fp16), then the gate/up recompute
  //    with the SwiGLU' epilogue
  uint16_t* dA = reinterpret_cast<uint16_t*>(ws + L.da);
  uint16_t* dA_lo = reinterpret_cast<uint16_t*>(ws + L.da_lo);
  GemmParams da{};
  da.offsets = offsets; da.counts = counts; da.w_perm = w_perm; da.err = err;
  da.maxabs = maxabs;
  da.E = E; da.D = D; da.I = I;
  da.order = tun.order[MOE_GEMM_DA];
  da.swap_tails = tun.swap_tails;
  da.dw_chunk_rows = chunk;
  da.tile_n = (tun.da_tile_n == 256 && I % 256 == 0) ? 256 : 128;
  bool ok = map_kmajor(&da.mapA0, dyp, D, cap, 128) && map_kmajor(&da.mapA1, dyp, D, cap, 64) &&
            map_kmajor(&da.mapB0, w_down, D, EI, static_cast<uint32_t>(da.tile_n / 2)) &&
            map_store_16(&da.mapO0, dA, I, cap, Elem::F16) &&
            map_store_16(&da.mapO1, dA_lo, I, cap, Elem::F16);
  if (!ok) return MOE_ERR_CUDA;
  da.n_tiles = I / da.tile_n;
  {
    LaunchScope ls(kKGemmDA, s);
    e = launch_gemm_kind<GemmKind::DA>(da, pairs_max * da.n_tiles, f->num_sms, s);
  }
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  GemmParams a{};
  a.offsets = offsets; a.counts = counts; a.w_perm = w_perm; a.dA = dA; a.dA_lo = dA_lo;
  a.err = err; a.maxabs = maxabs;
  a.E = E; a.D = D; a.I = I;
  a.order = tun.order[MOE_GEMM_BWD_GATE_UP];
  a.swap_tails = tun.swap_tails;
  a.dw_chunk_rows = chunk;
  ok = map_kmajor(&a.mapA0, x_perm, D, cap, 128) && map_kmajor(&a.mapA1, x_perm, D, cap, 64) &&
       map_mnmajor(&a.mapB0, w_gate, I, ED, 2) && map_mnmajor(&a.mapB1, w_up, I, ED, 2) &&
       map_mnmajor(&a.mapB2, w_gate, I, ED, 1) && map_mnmajor(&a.mapB3, w_up, I, ED, 1) &&
       map_store_16(&a.mapO0, act, I, cap, Elem::F16) &&
       map_store_16(&a.mapO1, dh, 2ull * I, cap) &&
       map_store_16(&a.mapO2, dh16, 2ull * I, cap, Elem::F16) &&
       map_store_16(&a.mapO3, act_lo, I, cap, Elem::F16) &&
       map_store_16(&a.mapO4, dh16_lo, 2ull * I, cap, Elem::F16);
  if (!ok) return MOE_ERR_CUDA;
  a.n_tiles = I / 128;
  {
    LaunchScope ls(kKGemmBwdGU, s);
    e = launch_gemm_kind<GemmKind::BwdGU>(a, pairs_max * a.n_tiles, f->num_sms, s);
  }
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  // 3. input gradient
  GemmParams xg{};
  xg.offsets = offsets; xg.counts = counts; xg.err = err; xg.E = E; xg.D = D; xg.I = I;
  xg.order = tun.order[MOE_GEMM_DX];
  xg.swap_tails = tun.swap_tails;
  xg.dw_chunk_rows = chunk;
  ok = map_kmajor(&xg.mapA0, dh, 2ull * I, cap, 128) && map_kmajor(&xg.mapA1, dh, 2ull * I, cap, 64) &&
       map_kmajor(&xg.mapB0, w_gate, I, ED, 128) &&
       map_kmajor(&xg.mapB1, w_up, I, ED, 128) && map_store_16(&xg.mapO0, dx_perm, D, cap);
  if (!ok) return MOE_ERR_CUDA;
  xg.n_tiles = D / 256;
  {
    LaunchScope ls(kKGemmDx, s);
    e = launch_gemm_kind<GemmKind::Dx>(xg, pairs_max * xg.n_tiles, f->num_sms, s);
  }
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  // the dx reduction to tokens (when asked for) on the side stream, beside the
  // weight-gradient GEMMs; joined back before the call returns
  const SideWork side{ss, dx_perm, inv_perm, dx, T, K, D};
  return bwd_weight_grads(offsets, counts, dw_prefix, err, maxabs, E, D, I, cap, chunk, act,
                          act_lo, dh16, dh16_lo, xp16, dyp16, dw_gate, dw_up, dw_down, f->num_sms,
                          side, s);
}

// Step 4 of the backward: the weight gradients (fp16 operands, fp32 accumulate and output).
static int bwd_weight_grads(const int32_t* offsets, const int32_t* counts, int* dw_prefix,
                            int* err, const uint32_t* maxabs, int E, int D, int I, uint64_t cap,
                            int chunk, void* act, void* act_lo, void* dh16, void* dh16_lo,
                            moe_bf16_t* xp16, moe_bf16_t* dyp16, float* dw_gate, float* dw_up,
                            float* dw_down, int num_sms, const SideWork& side, cudaStream_t s) {
  const uint64_t ED = static_cast<uint64_t>(E) * D, EI = static_cast<uint64_t>(E) * I;
  cudaError_t e;
  bool ok;

  e = launch_dw_prep(offsets, E, chunk, dw_prefix, dw_gate, dw_up, dw_down, D, I, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  const int max_chunks = E + static_cast<int>(cap / chunk) + 1;
  GemmParams g{};
  g.offsets = offsets; g.counts = counts; g.dw_prefix = dw_prefix; g.err = err;
  g.maxabs = maxabs;
  g.E = E; g.D = D; g.I = I;
  g.dw_chunk_rows = chunk;
  ok = map_mnmajor(&g.mapA0, xp16, D, cap, 2, Elem::F16) &&
       map_mnmajor(&g.mapB0, dh16, 2ull * I, cap, 4, Elem::F16) &&
       map_mnmajor(&g.mapB1, dh16_lo, 2ull * I, cap, 4, Elem::F16) &&
       map_store_f32(&g.mapO0, dw_gate, I, ED) && map_store_f32(&g.mapO1, dw_up, I, ED);
  if (!ok) return MOE_ERR_CUDA;
  g.m_tiles = D / 128;
  g.n_tiles = (2 * I) / 256;
  {
    LaunchScope ls(kKGemmDwGU, s);
    e = launch_gemm_kind<GemmKind::DwGU>(g, max_chunks * g.m_tiles * g.n_tiles, num_sms, s);
  }
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  GemmParams d{};
  d.offsets = offsets; d.counts = counts; d.dw_prefix = dw_prefix; d.err = err;
  d.maxabs = maxabs;
  d.E = E; d.D = D; d.I = I;
  d.dw_chunk_rows = chunk;
  ok = map_mnmajor(&d.mapA0, act, I, cap, 2, Elem::F16) &&
       map_mnmajor(&d.mapA1, act_lo, I, cap, 2, Elem::F16) &&
       map_mnmajor(&d.mapB0, dyp16, D, cap, 4, Elem::F16) &&
       map_store_f32(&d.mapO0, dw_down, D, EI);
  if (!ok) return MOE_ERR_CUDA;
  d.m_tiles = I / 128;
  d.n_tiles = D / 256;
  if (!side.ss) {
    LaunchScope ls(kKGemmDwD, s);
    return to_status(
        launch_gemm_kind<GemmKind::DwD>(d, max_chunks * d.m_tiles * d.n_tiles, num_sms, s));
  }
  // the dx reduction on the side stream, beside the dW_down GEMM (it only needs the dX
  // GEMM, which is done by now); every exit from here joins the side stream back
  SideStream* ss = side.ss;
  if (stream_after(ss->s, s, ss->fork) != cudaSuccess) return MOE_ERR_CUDA;
  e = launch_combine(side.dx_perm, side.inv_perm, nullptr, side.T, side.K, side.D, side.dx,
                     ss->s, kKCombineDx);
  if (e == cudaSuccess) {
    LaunchScope ls(kKGemmDwD, s);
    e = launch_gemm_kind<GemmKind::DwD>(d, max_chunks * d.m_tiles * d.n_tiles, num_sms, s);
  }
  const cudaError_t je = stream_after(s, ss->s, ss->join);
  return e != cudaSuccess ? MOE_ERR_CUDA : to_status(je);
}

MOE_EXPORT int moe_tuning_get(int T, int K, int E, int D, int I, moe_tuning_t* out,
                              int* source) {
  if (!out || !basic_sizes_ok(T, K, E, 128) || D < 1 || I < 1) return MOE_ERR_INVALID_ARG;
  *out = select_tuning(T, K, E, D, I, source);
  return MOE_OK;
}

MOE_EXPORT int moe_tuning_override(const moe_tuning_t* t) {
  std::lock_guard<std::mutex> g(g_tune_mu);
  if (!t) {
    g_tune_override_on = false;
    return MOE_OK;
  }
  if (!tuning_ok(*t)) return MOE_ERR_INVALID_ARG;
  g_tune_override = *t;
  g_tune_override_on = true;
  return MOE_OK;
}

static bool router_args_ok(int T, int E, int K, int router) {
  if (T < 0 || K < 1 || K > 32 || E < K || E > kMaxExperts) return false;
  if (router != MOE_ROUTER_SOFTMAX_TOPK && router != MOE_ROUTER_SIGMOID_TOP1) return false;
  if (router == MOE_ROUTER_SIGMOID_TOP1 && K != 1) return false;
  return static_cast<long long>(T) * (E > K ? E : K) < (1ll << 31);
}

MOE_EXPORT int moe_router_topk(const float* logits, int T, int E, int K, int router,
                               int32_t* topk_ids, float* topk_w, void* stream) {
  if (!router_args_ok(T, E, K, router)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!logits || !topk_ids || !topk_w)) return MOE_ERR_INVALID_ARG;
  int st = check_device();
  if (st != MOE_OK) return st;
  return to_status(launch_router_topk(logits, T, E, K, router, topk_ids, topk_w,
                                      static_cast<cudaStream_t>(stream)));
}

MOE_EXPORT int moe_router_weight_grad(const moe_bf16_t* dy, const moe_bf16_t* y_perm,
                                      const int32_t* inv_perm, int T, int K, int D,
                                      float* d_topk_w, void* stream) {
  if (T < 0 || K < 1 || K > 32 || D <= 0 || D % 8 != 0) return MOE_ERR_INVALID_ARG;
  if (static_cast<long long>(T) * K >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!dy || !y_perm || !inv_perm || !d_topk_w)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!aligned16(dy) || !aligned16(y_perm))) return MOE_ERR_INVALID_ARG;
  int st = check_device();
  if (st != MOE_OK) return st;
  return to_status(launch_router_weight_grad(dy, y_perm, inv_perm, T, K, D, d_topk_w,
                                             static_cast<cudaStream_t>(stream)));
}

MOE_EXPORT int moe_router_backward(const int32_t* topk_ids, const float* topk_w,
                                   const float* d_topk_w, int T, int E, int K, int router,
                                   float* d_logits, void* stream) {
  if (!router_args_ok(T, E, K, router)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_ids || !topk_w || !d_topk_w || !d_logits)) return MOE_ERR_INVALID_ARG;
  int st = check_device();
  if (st != MOE_OK) return st;
  return to_status(launch_router_backward(topk_ids, topk_w, d_topk_w, T, E, K, router, d_logits,
                                          static_cast<cudaStream_t>(stream)));
}

MOE_EXPORT int moe_get_device_error(void* workspace, int* code, int* detail, void* stream) {
  if (!workspace || !code) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int raw = 0;
  if (cudaMemcpyAsync(&raw, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (detail) *detail = raw;
  if (raw == kDevOk) *code = MOE_OK;
  else if (raw == kDevBadExpertId) *code = MOE_ERR_BAD_INDEX;
  else if (raw == kDevFp16Range) *code = MOE_ERR_FP16_RANGE;
  else *code = MOE_ERR_DEVICE_TIMEOUT;
  if (raw != 0) {
    // clears the word and the header's barrier counters a kernel that gave up may leave set
    if (cudaMemsetAsync(workspace, 0, 1024, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

MOE_EXPORT int moe_debug_drop_next_loads(void) {
  t_drop_next_loads = true;
  return MOE_OK;
}

MOE_EXPORT int moe_num_kernels(void) { return kNumKernelIds; }

MOE_EXPORT const char* moe_kernel_name(int id) { return kernel_name(id); }

MOE_EXPORT long long moe_launch_count(long long* counts) {
  if (counts)
    for (int i = 0; i < kNumKernelIds; ++i) counts[i] = g_launch_by_id[i].load();
  return g_launch_total.load();
}

MOE_EXPORT int moe_timing_enable(int on) {
  g_timing_mask.store(on ? ~0ull : 0ull);
  return MOE_OK;
}

MOE_EXPORT int moe_timing_enable_mask(unsigned long long kernel_mask) {
  g_timing_mask.store(kernel_mask);
  return MOE_OK;
}

MOE_EXPORT int moe_timing_collect(double* ms, long long* launches) {
  std::lock_guard<std::mutex> lk(g_timing_mu);
  int status = MOE_OK;
  for (auto& r : g_recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) {
      status = MOE_ERR_CUDA;
    } else if (r.id >= 0 && r.id < kNumKernelIds) {
      if (ms) ms[r.id] += t;
      if (launches) launches[r.id] += 1;
    }
    g_event_pool.push_back(r.a);
    g_event_pool.push_back(r.b);
  }
  g_recs.clear();
  return status;
}
