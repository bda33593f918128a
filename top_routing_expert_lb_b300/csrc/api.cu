// Host side of the C ABI declared in include/moe.h: argument checks,
// workspace layout, TMA descriptors and the launch sequence of the layer.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include "../../include/moe.h"
#include "bounds.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

std::atomic<uint64_t> g_timeout_ns{2000000000ull};

// ---------------------------------------------------------------- accounting
uint64_t g_launches = 0;
uint32_t g_prof_mask = 0;  // bit (1 << kernel id) set: that kernel is bracketed
struct ProfRec {
  int32_t kernel;
  cudaEvent_t start, stop;
};
std::vector<ProfRec> g_prof;        // recorded pairs, launch order
std::vector<cudaEvent_t> g_ev_pool;  // reusable events
size_t g_ev_used = 0;

cudaEvent_t pool_event() {
  if (g_ev_used == g_ev_pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    g_ev_pool.push_back(e);
  }
  return g_ev_pool[g_ev_used++];
}

// Records `e` on `st`; inside a stream capture as an external event node, so
// that every replay of the graph records it again.
void record_event(cudaEvent_t e, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
  else
    cudaEventRecord(e, st);
}

// Runs one launcher; counts it and, when profiling, brackets it with events.
template <typename F>
int tracked(int32_t kernel, cudaStream_t st, F&& launch) {
  cudaEvent_t a = nullptr, b = nullptr;
  const bool prof = (g_prof_mask >> kernel) & 1u;
  if (prof) {
    a = pool_event();
    b = pool_event();
    if (a) record_event(a, st);
  }
  const int rc = launch();
  if (rc == 0) ++g_launches;
  if (prof && a && b) {
    record_event(b, st);
    g_prof.push_back({kernel, a, b});
  }
  return rc;
}

constexpr size_t kAlign = 256;
// router accumulator block: counts [256] int32 at 0, P sums [256] u64 at 1024,
// importance sums [256] u64 at 3072, entropy sum u64 at 5120, finished tiles
// int32 at 5128
constexpr size_t kRaccBytes = 5376;
constexpr int64_t kPartUnits = 256;  // K-split units whose partial logits the workspace holds
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Workspace regions (byte offsets from the workspace base).
struct Layout {
  size_t status, tile_hist, tile_psum, tile_lse2, tile_base, exp_count, exp_psum, offsets;
  size_t tile_imp, tile_ent, exp_imp;
  size_t racc, tile_arrive, chunk_acc, part;  // router accumulators and K-split partials
  int32_t max_split, chunk_tiles, n_chunks;
  size_t slot_row, row_token;
  size_t pair_score, stage_q, stage_key, all_offsets;  // priority capacity
  size_t scores_t, sel_t, row_gate;                    // expert choice
  size_t x_perm, h, y_perm, h_s, y_s, total;
  int64_t ntiles, rmax, C, r;
};

int check_shape(const moe_shape_t* s) {
  if (s == nullptr) return MOE_ERR_INVALID_ARG;
  if (s->T < 0 || s->d <= 0 || s->M <= 0 || s->E <= 0 || s->k < 0 || s->n_shared < 0)
    return MOE_ERR_INVALID_ARG;
  if (s->k > s->E) return MOE_ERR_INVALID_ARG;
  if (!std::isfinite(s->capacity_factor) || !std::isfinite(s->balance_coef))
    return MOE_ERR_INVALID_ARG;
  if ((s->flags & ~(MOE_FLAG_SIGMOID | MOE_FLAG_NO_RENORM | MOE_FLAG_PRIORITY_CAPACITY |
                    MOE_FLAG_EXPERT_CHOICE)) != 0)
    return MOE_ERR_UNSUPPORTED;
  if ((s->flags & MOE_FLAG_PRIORITY_CAPACITY) && (s->flags & MOE_FLAG_EXPERT_CHOICE))
    return MOE_ERR_UNSUPPORTED;
  if (s->E > MOE_MAX_EXPERTS || s->k > MOE_MAX_TOPK) return MOE_ERR_UNSUPPORTED;
  if (s->T > (1 << 24)) return MOE_ERR_UNSUPPORTED;
  if (s->d % 64 != 0 || s->d < 64 || s->d > 16384) return MOE_ERR_UNSUPPORTED;
  if (s->M % 128 != 0 || s->M < 128 || s->M > 32768) return MOE_ERR_UNSUPPORTED;
  if (s->n_shared > 8) return MOE_ERR_UNSUPPORTED;
  if (s->reserved != 0) return MOE_ERR_INVALID_ARG;
  const moe_tuning_t& t = s->tuning;
  auto tile_ok = [](int32_t v) { return v == 0 || v == 128 || v == 256; };
  if (!tile_ok(t.gemm1_tile) || !tile_ok(t.gemm2_tile)) return MOE_ERR_INVALID_ARG;
  if (t.tile_order < 0 || t.tile_order > 2) return MOE_ERR_INVALID_ARG;
  if (t.tail_max_n > 0 && (t.tail_max_n < 16 || t.tail_max_n > 128)) return MOE_ERR_INVALID_ARG;
  if (t.n_block < 0 || t.n_block > 64 || t.block_min_rows < 0) return MOE_ERR_INVALID_ARG;
  if ((t.options & ~(MOE_TUNE_NO_HALF_TILES | MOE_TUNE_GEMM1_SPLIT | MOE_TUNE_FUSED_GATHER |
                     MOE_TUNE_GATE_IN_EPILOGUE | MOE_TUNE_SWAP_ALL_TAILS |
                     MOE_TUNE_TWO_CTAS_PER_SM | MOE_TUNE_NO_PDL)) != 0 ||
      t.reserved != 0)
    return MOE_ERR_INVALID_ARG;
  if ((t.options & MOE_TUNE_FUSED_GATHER) && t.gemm1_tile == 256) return MOE_ERR_INVALID_ARG;
  if (t.gemm2_tile == 256 && s->d % 256 != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// Limit of this call's bounded device waits.
uint64_t timeout_of(const moe_shape_t* s) {
  return s->tuning.wait_timeout_ns != 0 ? s->tuning.wait_timeout_ns
                                          : g_timeout_ns.load(std::memory_order_relaxed);
}

// Whether this call's router, scatter, GEMM and combine launches use
// programmatic dependent launch (each may start while the kernel before it
// finishes; each waits for it before reading what it wrote).
bool use_pdl(const moe_shape_t* s) { return (s->tuning.options & MOE_TUNE_NO_PDL) == 0; }

int64_t capacity_of(const moe_shape_t* s) {
  if (!(s->capacity_factor > 0.0f)) return -1;
  const double c = static_cast<double>(s->capacity_factor);
  return static_cast<int64_t>(
      std::ceil(c * static_cast<double>(s->k) * static_cast<double>(s->T) /
                static_cast<double>(s->E)));
}

inline bool is_ec(const moe_shape_t* s) { return (s->flags & MOE_FLAG_EXPERT_CHOICE) != 0; }
inline bool is_priority(const moe_shape_t* s) {
  return (s->flags & MOE_FLAG_PRIORITY_CAPACITY) != 0 && capacity_of(s) >= 0;
}

// Expert choice: tokens per expert, min(T, ceil(c k T / E)), c <= 0 read as 1.
int64_t ec_capacity_of(const moe_shape_t* s) {
  const double c = s->capacity_factor > 0.0f ? static_cast<double>(s->capacity_factor) : 1.0;
  const int64_t r = static_cast<int64_t>(std::ceil(
      c * static_cast<double>(s->k) * static_cast<double>(s->T) / static_cast<double>(s->E)));
  return r < s->T ? r : s->T;
}

Layout layout_of(const moe_shape_t* s) {
  Layout L{};
  const int64_t T = s->T, d = s->d, M = s->M, E = s->E, k = s->k;
  const int64_t Ms = static_cast<int64_t>(s->n_shared) * M;
  L.ntiles = (T + kTileTokens - 1) / kTileTokens;
  L.C = capacity_of(s);
  L.rmax = T * k;
  if (L.C >= 0 && E * L.C < L.rmax) L.rmax = E * L.C;
  L.r = -1;
  if (is_ec(s)) {
    L.C = -1;
    L.r = ec_capacity_of(s);
    L.rmax = E * L.r;
  }
  const bool prio = is_priority(s) && !is_ec(s);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align_up(bytes);
    return at;
  };
  L.status = take(kAlign);
  L.tile_hist = take(L.ntiles * E * 4);
  L.tile_psum = take(L.ntiles * E * 4);
  L.tile_lse2 = take(L.ntiles * 4);
  L.tile_base = take(L.ntiles * E * 4);
  L.exp_count = take(E * 4);
  L.exp_psum = take(E * 8);
  L.tile_imp = take(L.ntiles * E * 4);
  L.tile_ent = take(L.ntiles * 4);
  L.exp_imp = take(E * 8);
  L.offsets = take((E + 1) * 4);
  // router: [E] counts (int32), [E] P and [E] importance sums (fixed point,
  // 64-bit), the entropy sum and the finished-tile counter; per-tile arrival
  // counters of K-split slices; per-chunk expert counts; partial logits of
  // K-split units (at most kPartUnits units of E x 128 fp32)
  L.racc = take(kRaccBytes);
  L.tile_arrive = take(L.ntiles * 4);
  L.chunk_tiles = L.ntiles <= 1024 ? 32 : 1;
  while (static_cast<int64_t>(L.chunk_tiles) * 32 < L.ntiles) L.chunk_tiles *= 2;
  L.n_chunks = static_cast<int32_t>((L.ntiles + L.chunk_tiles - 1) / L.chunk_tiles);
  L.chunk_acc = take(static_cast<size_t>(L.n_chunks) * E * 4);
  L.max_split = 1;
  while (L.max_split < kMaxSplitUnits && L.ntiles * 2 * L.max_split <= kPartUnits)
    L.max_split *= 2;
  L.part = take(L.max_split > 1 ? static_cast<size_t>(L.ntiles) * L.max_split * E * 128 * 4 : 0);
  L.slot_row = take(T * k * 4);
  L.row_token = take(L.rmax * 4);
  L.pair_score = take(prio ? T * k * 4 : 0);
  L.stage_q = take(prio ? T * k * 4 : 0);
  L.stage_key = take(prio ? T * k * 4 : 0);
  L.all_offsets = take(prio ? (E + 1) * 4 : 0);
  L.scores_t = take(is_ec(s) ? E * T * 4 : 0);
  L.sel_t = take(is_ec(s) ? E * T * 4 : 0);
  L.row_gate = take(L.rmax * 4);
  L.x_perm = take(L.rmax * d * 2);
  L.h = take(L.rmax * M * 2);
  L.y_perm = take(L.rmax * d * 2);
  L.h_s = take(T * Ms * 2);
  L.y_s = take(T * d * 2);
  L.total = o;
  return L;
}

template <typename Tp>
Tp* at(void* ws, size_t off) {
  return reinterpret_cast<Tp*>(static_cast<uint8_t*>(ws) + off);
}

int check_ws(const moe_shape_t* s, void* ws, size_t ws_bytes, Layout* L) {
  *L = layout_of(s);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0)
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < L->total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

int sm_count_cached() {
  static std::atomic<int> cache[64];  // 0 until looked up; racing writers store the same value
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

inline int cuda_rc(int rc) {
  if (rc == 0) return MOE_OK;
  if (rc == -2) return MOE_ERR_UNSUPPORTED;
  return MOE_ERR_CUDA;
}

// ---------------------------------------------------------------- stages
// Extra router / finalize outputs of the priority-capacity and expert-choice
// paths.
struct RouteExtras {
  float* pair_score = nullptr;      // [T][k] scores of the selected pairs
  int32_t* all_offsets = nullptr;   // [E+1] scan of the counts before capacity
  float* scores_t = nullptr;        // [E][T] expert choice: every score
  int32_t fixed_count = -1;         // expert choice: r
  double n_pairs = -1.0;            // expert choice: E r
};

// Points the router's scratch fields at the accumulator block `racc` and the
// given per-tile / partial regions.
void set_router_scratch(RouterArgs* ra, uint8_t* racc, float* tile_lse2, int* tile_arrive,
                        float* part, int max_split) {
  ra->acc_count = reinterpret_cast<int*>(racc);
  ra->acc_psum = reinterpret_cast<unsigned long long*>(racc + 1024);
  ra->acc_ent = reinterpret_cast<unsigned long long*>(racc + 5120);
  ra->tiles_done = reinterpret_cast<int*>(racc + 5128);
  ra->tile_lse2 = tile_lse2;
  ra->tile_arrive = tile_arrive;
  ra->part_logits = part;
  ra->max_split = max_split;
}

int do_route(const moe_shape_t* s, const uint16_t* x, const uint16_t* wr, const float* off,
             const float* bias, int32_t* ids, float* gates, int32_t* counts, float* f, float* P,
             float* bal, float* z, void* ws, const Layout& L, bool for_layer,
             int32_t* offsets, cudaStream_t st, float* importance = nullptr,
             float* importance_cv2 = nullptr, float* entropy_mean = nullptr,
             const RouteExtras& ex = RouteExtras()) {
  const bool want_imp = (importance != nullptr || importance_cv2 != nullptr) && s->k > 0;
  RouterArgs ra{};
  ra.T = s->T;
  ra.d = s->d;
  ra.E = s->E;
  ra.k = ex.scores_t ? 0 : s->k;  // expert choice: no per-token Top-k
  ra.logit_offset = off;
  ra.sel_bias = bias;
  ra.ids = ids;
  ra.gates = gates;
  ra.status = at<int>(ws, L.status);
  ra.timeout_ns = timeout_of(s);
  ra.flags = s->flags & (kRouteSigmoid | kRouteNoRenorm);
  ra.pair_score = ex.pair_score;
  ra.scores_t = ex.scores_t;
  uint8_t* racc = at<uint8_t>(ws, L.racc);
  set_router_scratch(&ra, racc, at<float>(ws, L.tile_lse2), at<int>(ws, L.tile_arrive),
                     L.max_split > 1 ? at<float>(ws, L.part) : nullptr, L.max_split);
  if (want_imp) ra.acc_imp = reinterpret_cast<unsigned long long*>(racc + 3072);
  if (entropy_mean == nullptr) ra.acc_ent = nullptr;
  if (for_layer) {
    // the permutation's inputs: per-tile counts and per-chunk bases
    ra.tile_hist = at<int32_t>(ws, L.tile_hist);
    ra.chunk_acc = at<int32_t>(ws, L.chunk_acc);
    ra.chunk_base = at<int32_t>(ws, L.tile_base);
    ra.chunk_tiles = L.chunk_tiles;
    ra.n_chunks = L.n_chunks;
  }
  ra.C = L.C;
  ra.balance_coef = s->balance_coef;
  ra.counts = counts;
  ra.f = f;
  ra.P = P;
  ra.bal_loss = bal;
  ra.z_loss = z;
  ra.offsets = offsets;
  ra.all_offsets = ex.all_offsets;
  ra.importance = want_imp ? importance : nullptr;
  ra.importance_cv2 = want_imp ? importance_cv2 : nullptr;
  ra.entropy_mean = entropy_mean;
  ra.fixed_count = ex.fixed_count;
  ra.n_pairs = ex.n_pairs;
  ra.pdl = use_pdl(s) ? 1 : 0;
  CUtensorMap mx, mw;
  std::memset(&mx, 0, sizeof(mx));
  std::memset(&mw, 0, sizeof(mw));
  if (s->T > 0) {
    const uint32_t nr = static_cast<uint32_t>((s->E + 15) / 16 * 16);
    if (!make_tmap_bf16(&mx, x, s->T, s->d, 128)) return MOE_ERR_CUDA;
    if (!make_tmap_bf16(&mw, wr, s->E, s->d, nr)) return MOE_ERR_CUDA;
  }
  if (s->k == 0 || ex.scores_t) {
    // no Top-k: zero importance (its definition has no selected experts)
    if (importance) cudaMemsetAsync(importance, 0, sizeof(float) * s->E, st);
    if (importance_cv2) cudaMemsetAsync(importance_cv2, 0, sizeof(float), st);
  }
  return cuda_rc(tracked(MOE_KERNEL_ROUTER, st, [&] {
    return launch_router(mx, mw, ra, sm_count_cached(), st);
  }));
}

// chunk_tiles: tiles per base in the workspace's tile_base region (the
// router's chunks in the layer, 1 after finalize_kernel in moe_permute)
int do_scatter(const moe_shape_t* s, const uint16_t* x, const int32_t* ids, const Layout& L,
               void* ws, const int32_t* offsets, int32_t* slot_row, int32_t* row_token,
               uint8_t* drop_mask, uint16_t* x_perm, cudaStream_t st, int32_t chunk_tiles,
               const float* gates = nullptr, float* row_gate = nullptr) {
  ScatterArgs sa{};
  sa.T = s->T;
  sa.d = s->d;
  sa.E = s->E;
  sa.k = s->k;
  sa.C = L.C;
  sa.ids = ids;
  sa.tile_base = at<int32_t>(ws, L.tile_base);
  sa.tile_hist = at<int32_t>(ws, L.tile_hist);
  sa.chunk_tiles = chunk_tiles;
  sa.offsets = offsets;
  sa.x = x;
  sa.slot_row = slot_row;
  sa.row_token = row_token;
  sa.drop_mask = drop_mask;
  sa.x_perm = x_perm;
  sa.num_sms = sm_count_cached();
  sa.gates = gates;
  sa.row_gate = row_gate;
  sa.rmax = L.rmax;
  sa.status = at<int>(ws, L.status);
  sa.pdl = use_pdl(s) ? 1 : 0;
  return cuda_rc(tracked(MOE_KERNEL_SCATTER, st, [&] { return launch_scatter(sa, st); }));
}

// Priority capacity: stage every pair by expert, cut each expert at its C
// highest scores, then gather the kept rows.
int do_priority_dispatch(const moe_shape_t* s, const uint16_t* x, const int32_t* ids,
                         const Layout& L, void* ws, const int32_t* offsets, int32_t* slot_row,
                         int32_t* row_token, uint8_t* drop_mask, uint16_t* x_perm,
                         cudaStream_t st, const float* gates = nullptr,
                         float* row_gate = nullptr) {
  ScatterArgs sa{};
  sa.T = s->T;
  sa.d = s->d;
  sa.E = s->E;
  sa.k = s->k;
  sa.C = L.C;
  sa.ids = ids;
  sa.tile_base = at<int32_t>(ws, L.tile_base);
  sa.tile_hist = at<int32_t>(ws, L.tile_hist);
  sa.chunk_tiles = L.chunk_tiles;
  sa.offsets = offsets;
  sa.x = x;
  sa.num_sms = sm_count_cached();
  sa.stage_q = at<int32_t>(ws, L.stage_q);
  sa.stage_key = at<float>(ws, L.stage_key);
  sa.pair_score = at<float>(ws, L.pair_score);
  sa.all_offsets = at<int32_t>(ws, L.all_offsets);
  sa.rmax = static_cast<int64_t>(s->T) * s->k;  // staging rows: every pair
  sa.status = at<int>(ws, L.status);
  int rc = cuda_rc(tracked(MOE_KERNEL_SCATTER, st, [&] { return launch_scatter(sa, st); }));
  if (rc != MOE_OK) return rc;
  PrioritySelectArgs pa{};
  pa.E = s->E;
  pa.k = s->k;
  pa.C = L.C;
  pa.all_offsets = sa.all_offsets;
  pa.offsets = offsets;
  pa.stage_q = sa.stage_q;
  pa.stage_key = sa.stage_key;
  pa.slot_row = slot_row;
  pa.drop_mask = drop_mask;
  pa.row_token = row_token;
  pa.gates = gates;
  pa.row_gate = row_gate;
  pa.rmax = L.rmax;
  pa.n_pairs = static_cast<int64_t>(s->T) * s->k;
  pa.status = at<int>(ws, L.status);
  rc = cuda_rc(tracked(MOE_KERNEL_SELECT, st, [&] { return launch_priority_select(pa, st); }));
  if (rc != MOE_OK || x_perm == nullptr) return rc;  // no x_perm: GEMM-1 gathers the rows
  return cuda_rc(tracked(MOE_KERNEL_GATHER, st, [&] {
    return launch_gather_rows(x, row_token, offsets, s->E, s->d, L.rmax, x_perm,
                              sm_count_cached(), s->T, at<int>(ws, L.status), st);
  }));
}

// Expert choice: router (every score, expert-major) + finalize with fixed
// counts, then each expert's top-r cut.
int do_ec_route(const moe_shape_t* s, const uint16_t* x, const uint16_t* wr, const float* off,
                int32_t* row_token, float* row_gate, int32_t* counts, float* f, float* P,
                float* bal, float* z, void* ws, const Layout& L, cudaStream_t st) {
  RouteExtras ex;
  ex.scores_t = at<float>(ws, L.scores_t);
  ex.fixed_count = static_cast<int32_t>(L.r);
  ex.n_pairs = static_cast<double>(s->E) * static_cast<double>(L.r);
  int rc = do_route(s, x, wr, off, nullptr, nullptr, nullptr, counts, f, P, bal, z, ws, L,
                    false, at<int32_t>(ws, L.offsets), st, nullptr, nullptr, nullptr, ex);
  if (rc != MOE_OK || s->T == 0) return rc;
  EcSelectArgs ea{};
  ea.T = s->T;
  ea.E = s->E;
  ea.r = static_cast<int32_t>(L.r);
  ea.scores_t = ex.scores_t;
  ea.sel_t = at<int32_t>(ws, L.sel_t);
  ea.row_token = row_token;
  ea.row_gate = row_gate;
  return cuda_rc(tracked(MOE_KERNEL_SELECT, st, [&] { return launch_ec_select(ea, st); }));
}

// The gate/up projection feeds from the token rows itself (TMA 4-row gathers by
// row_token, no x_perm) only with MOE_TUNE_FUSED_GATHER: the gather issues 32
// TMA instructions per k-block instead of one and measured about 3.5x slower
// in GEMM-1, so the default materialises x_perm in the scatter.
// MOE_TUNE_GATE_IN_EPILOGUE: the down projection's epilogue multiplies each
// routed row by its gate (fp32, before rounding) and the combine only adds the
// rows in slot order (or expert order).  Same bytes, one multiply moved; off
// by default (measured within noise).
bool gate_in_epilogue(const moe_shape_t* s) {
  return (s->tuning.options & MOE_TUNE_GATE_IN_EPILOGUE) != 0;
}

bool fused_gather(const moe_shape_t* s) {
  return (s->tuning.options & MOE_TUNE_FUSED_GATHER) != 0;
}

// x_perm: routed rows, or null with gather_rows (token row of every routed
// row, read from x by the GEMM's producer).
int do_ffn(const moe_shape_t* s, const uint16_t* x_perm, const int32_t* offsets,
           const uint16_t* w13, const uint16_t* w2, uint16_t* y_perm, const uint16_t* x,
           const uint16_t* w13s, const uint16_t* w2s, uint16_t* y_s, void* ws, const Layout& L,
           cudaStream_t st, const int32_t* gather_rows = nullptr,
           const float* row_scale = nullptr) {
  const int64_t T = s->T, d = s->d, M = s->M, E = s->E;
  const int64_t Ms = static_cast<int64_t>(s->n_shared) * M;
  const bool routed = L.rmax > 0;
  const bool shared = Ms > 0 && T > 0;
  if (!routed && !shared) return MOE_OK;
  uint16_t* h = at<uint16_t>(ws, L.h);
  uint16_t* h_s = at<uint16_t>(ws, L.h_s);
  const int bn2 = (d % 256 == 0) ? 256 : (d % 128 == 0 ? 128 : 64);
  const int nsm = sm_count_cached();
  const int64_t rows_per_expert =
      L.r >= 0 ? L.r : (E > 0 ? (static_cast<int64_t>(T) * s->k) / E : 0);
  // The gate/up projection runs on single-CTA 128 x 256 tiles (transposed
  // tails) unless gemm1_tile asks for 256 x 256 CTA-pair tiles.  Timed against
  // each other call by call in one process (200 alternating layer calls, L2
  // flushed before each), single-CTA tiles made the Mixtral layer 4.3 %
  // faster (2.51 against 2.63 ms median), early and late in the power-capped
  // run alike, and the pair tiles cost DeepSeekMoE-16B 11 % (the 256-row
  // padding of its many small experts).  Gathered rows need the single-CTA
  // kernel.
  const moe_tuning_t& tune = s->tuning;
  if (tune.gemm1_tile == 256 && gather_rows != nullptr) return MOE_ERR_INVALID_ARG;  // needs x_perm
  const bool paired = gather_rows == nullptr && tune.gemm1_tile == 256;
  const uint32_t bbox = paired ? 128u : 256u;
  // MOE_TUNE_GEMM1_SPLIT: the first projection runs each group's whole 256-row
  // blocks on CTA-pair tiles and only the remaining rows (< 256 per group) on
  // single-CTA tiles (two launches, both counted as the gate/up kernel).
  // Measured 9 % slower than single-CTA tiles throughout on Mixtral, so off
  // by default.
  const bool split1 = (tune.options & MOE_TUNE_GEMM1_SPLIT) != 0 && !paired &&
                      gather_rows == nullptr && nsm >= 2;

  // projection 1: [x_perm | x] -> h = SiLU(gate) * up
  CUtensorMap a0, a1, b0, b1;
  if (routed) {
    if (gather_rows != nullptr) {
      if (!make_tmap_bf16(&a0, x, T, d, 1)) return MOE_ERR_CUDA;  // one-row box: gather
    } else if (!make_tmap_bf16(&a0, x_perm, L.rmax, d, 128)) {
      return MOE_ERR_CUDA;
    }
    if (!make_tmap_bf16(&b0, w13, E * 2 * M, d, bbox)) return MOE_ERR_CUDA;
  }
  if (shared) {
    if (!make_tmap_bf16(&a1, x, T, d, 128)) return MOE_ERR_CUDA;
    if (!make_tmap_bf16(&b1, w13s, 2 * Ms, d, bbox)) return MOE_ERR_CUDA;
  }
  if (!routed) { a0 = a1; b0 = b1; }
  if (!shared) { a1 = a0; b1 = b0; }
  // pair launches of this projection: the B tensors again with 64-row boxes
  // (a group's last tile of at most 128 rows loads 64 gate + 64 up rows per CTA)
  CUtensorMap bh0 = b0, bh1 = b1;
  if (paired || split1) {
    if (routed && !make_tmap_bf16(&bh0, w13, E * 2 * M, d, 64)) return MOE_ERR_CUDA;
    if (shared && !make_tmap_bf16(&bh1, w13s, 2 * Ms, d, 64)) return MOE_ERR_CUDA;
    if (!routed) bh0 = bh1;
    if (!shared) bh1 = bh0;
  }
  // the outputs h / h_s as tensor maps (the epilogue's block stores)
  CUtensorMap o0, o1;
  if (routed && !make_tmap_out_bf16(&o0, h, L.rmax, M)) return MOE_ERR_CUDA;
  if (shared && !make_tmap_out_bf16(&o1, h_s, T, Ms)) return MOE_ERR_CUDA;
  if (!routed) o0 = o1;
  if (!shared) o1 = o0;
  CUtensorMap bp0 = b0, bp1 = b1;  // 128-row boxes for the pair launch
  if (split1) {
    if (routed && !make_tmap_bf16(&bp0, w13, E * 2 * M, d, 128)) return MOE_ERR_CUDA;
    if (shared && !make_tmap_bf16(&bp1, w13s, 2 * Ms, d, 128)) return MOE_ERR_CUDA;
    if (!routed) bp0 = bp1;
    if (!shared) bp1 = bp0;
  }
  GroupedGemmArgs g1{};
  g1.offsets = offsets;
  g1.n_routed = routed ? static_cast<int32_t>(E) : 0;
  g1.shared_rows = shared ? static_cast<int32_t>(T) : 0;
  g1.n_cols_routed = static_cast<int32_t>(2 * M);
  g1.n_cols_shared = static_cast<int32_t>(2 * Ms);
  g1.k_routed = static_cast<int32_t>(d);
  g1.k_shared = static_cast<int32_t>(d);
  g1.out_routed = h;
  g1.ld_routed = M;
  g1.out_shared = h_s;
  g1.ld_shared = Ms;
  g1.status = at<int>(ws, L.status);
  g1.timeout_ns = timeout_of(s);
  g1.gather_rows = routed ? gather_rows : nullptr;
  g1.out_rows_routed = L.rmax;
  g1.out_rows_shared = T;
  g1.gather_limit = T;
  if (tune.tail_max_n != 0) g1.tail_max_n = tune.tail_max_n < 0 ? 0 : tune.tail_max_n;
  // A wide single-CTA gate/up projection (at least 64 n-tiles, 2M >= 16384)
  // takes every group of more than 512 rows in blocks of 4 n-tiles: 5.4 %
  // faster on the Mixtral shape (1577 against 1667 us, 80 alternating layer
  // calls), while the narrow projections of DeepSeek-V2 keep blocks of 8 for
  // groups of more than 2048 rows (blocks of 4 there: +1 %).
  const bool wide1 = !paired && 2 * M / 256 >= 64;
  const int32_t n_block1 = tune.n_block != 0 ? tune.n_block : (wide1 ? 4 : g1.n_block);
  const int32_t min_rows1 =
      tune.block_min_rows != 0 ? tune.block_min_rows : (wide1 ? 512 : g1.block_min_rows);
  const int32_t n_block2 = tune.n_block != 0 ? tune.n_block : g1.n_block;
  const int32_t min_rows2 = tune.block_min_rows != 0 ? tune.block_min_rows : g1.block_min_rows;
  g1.n_block = n_block1;
  g1.block_min_rows = min_rows1;
  // CTA-pair launches with long tiles (K >= 4096) take their tiles from a
  // counter in the workspace: the dynamic order keeps the pairs that share a
  // weight tile in step (Mixtral: DRAM bytes of the gate/up projection down
  // from 2.7 GB to the algorithmic 1.95 GB).  With short tiles on skewed
  // shapes (DeepSeekMoE-16B, K = 1408) the static round-robin order measured
  // 3 % faster.  tile_order 1 / 2 forces either order.
  int* tile_counter = at<int>(ws, L.status + 128);
  auto dynamic_for = [&](int64_t K) {
    return (tune.tile_order == 2 || (tune.tile_order == 0 && K >= 4096)) ? tile_counter : nullptr;
  };
  g1.tile_counter = dynamic_for(d);
  g1.half_tiles = (tune.options & MOE_TUNE_NO_HALF_TILES) ? 0 : 1;
  // every tail transposed for short reductions (K <= 1024: Switch's gate/up
  // projection, 12 us per layer faster), else only a group's only m-tile
  const bool swap_all = (tune.options & MOE_TUNE_SWAP_ALL_TAILS) != 0;
  g1.swap_all_tails = (swap_all || d <= 1024) ? 1 : 0;
  g1.two_per_sm = (tune.options & MOE_TUNE_TWO_CTAS_PER_SM) ? 1 : 0;
  g1.pdl = use_pdl(s) ? 1 : 0;
  int rc = 0;
  if (split1) {
    GroupedGemmArgs g1p = g1;
    g1p.row_split = 1;
    rc = tracked(MOE_KERNEL_GEMM_SWIGLU, st, [&] {
      return launch_grouped_gemm(a0, a1, bp0, bp1, o0, o1, g1p, true, 256, true, nsm, st, &bh0,
                                 &bh1);
    });
    if (rc != 0) return cuda_rc(rc);
    g1.row_split = 2;
  }
  rc = tracked(MOE_KERNEL_GEMM_SWIGLU, st,
               [&] {
                 return launch_grouped_gemm(a0, a1, b0, b1, o0, o1, g1, true, 256, paired, nsm,
                                            st, &bh0, &bh1);
               });
  if (rc != 0) return cuda_rc(rc);
  g1.row_split = 0;

  // projection 2: [h | h_s] -> [y_perm | y_s]
  // The down projection (K = M, long tiles) runs on 256 x 256 CTA-pair tiles
  // for a few large experts (at most 16, averaging at least 512 rows): the
  // pair halves the operand bytes per FLOP and the 256-row padding stays
  // small (Mixtral: single-CTA tiles +119 us per layer in alternating calls).
  // With many experts of skewed sizes the padding costs more than the pair
  // saves (DeepSeekMoE-16B, 64 experts averaging 768 rows: pair tiles +10 us
  // in this projection).  gemm2_tile 128 / 256 overrides.
  bool paired2 = bn2 == 256 && (paired || (rows_per_expert >= 512 && E <= 16));
  if (tune.gemm2_tile == 128) paired2 = false;
  if (tune.gemm2_tile == 256) paired2 = bn2 == 256;
  // the pair form loads B in 128-row halves
  const uint32_t bbox2 = paired2 ? 128u : static_cast<uint32_t>(bn2);
  if (routed) {
    if (!make_tmap_bf16(&a0, h, L.rmax, M, 128)) return MOE_ERR_CUDA;
    if (!make_tmap_bf16(&b0, w2, E * d, M, bbox2)) return MOE_ERR_CUDA;
  }
  if (shared) {
    if (!make_tmap_bf16(&a1, h_s, T, Ms, 128)) return MOE_ERR_CUDA;
    if (!make_tmap_bf16(&b1, w2s, d, Ms, bbox2)) return MOE_ERR_CUDA;
  }
  if (!routed) { a0 = a1; b0 = b1; }
  if (!shared) { a1 = a0; b1 = b0; }
  if (routed && !make_tmap_out_bf16(&o0, y_perm, L.rmax, d)) return MOE_ERR_CUDA;
  if (shared && !make_tmap_out_bf16(&o1, y_s, T, d)) return MOE_ERR_CUDA;
  if (!routed) o0 = o1;
  if (!shared) o1 = o0;
  GroupedGemmArgs g2 = g1;
  g2.swap_all_tails = (swap_all || M <= 1024) ? 1 : 0;
  // A short down projection (K = M <= 2048) over many small experts (fewer
  // than 512 rows on average) runs two CTAs per SM: DeepSeek-V2's took 1190
  // against 1242 us in alternating calls; the gate/up projections and longer
  // reductions ran slower that way (DeepSeekMoE-16B, Switch, Mixtral).
  g2.two_per_sm = (g1.two_per_sm || (M <= 2048 && rows_per_expert < 512)) ? 1 : 0;
  g2.n_block = n_block2;
  g2.block_min_rows = min_rows2;
  g2.tile_counter = dynamic_for(M);
  g2.gather_rows = nullptr;
  g2.row_scale = routed ? row_scale : nullptr;
  g2.n_cols_routed = static_cast<int32_t>(d);
  g2.n_cols_shared = static_cast<int32_t>(d);
  g2.k_routed = static_cast<int32_t>(M);
  g2.k_shared = static_cast<int32_t>(Ms > 0 ? Ms : 64);
  g2.out_routed = y_perm;
  g2.ld_routed = d;
  g2.out_rows_routed = L.rmax;
  g2.out_rows_shared = T;
  g2.out_shared = y_s;
  g2.ld_shared = d;
  rc = tracked(MOE_KERNEL_GEMM_DOWN, st,
               [&] {
                 return launch_grouped_gemm(a0, a1, b0, b1, o0, o1, g2, false, bn2, paired2, nsm,
                                            st);
               });
  return cuda_rc(rc);
}

}  // namespace

uint64_t default_wait_timeout_ns() { return g_timeout_ns.load(std::memory_order_relaxed); }

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_error_string(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_CUDA: return "CUDA call failed";
    case MOE_ERR_TIMEOUT: return "bounded device wait timed out";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_BOUNDS: return "device index out of range (bounds-checked build)";
    default: return "unknown error";
  }
}

int moe_workspace_size(const moe_shape_t* shape, size_t* bytes) {
  const int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = layout_of(shape).total;
  return MOE_OK;
}

int moe_capacity(const moe_shape_t* shape, int64_t* C) {
  const int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (C == nullptr) return MOE_ERR_INVALID_ARG;
  *C = capacity_of(shape);
  return MOE_OK;
}

int moe_max_rows(const moe_shape_t* shape, int64_t* rows) {
  const int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (rows == nullptr) return MOE_ERR_INVALID_ARG;
  *rows = layout_of(shape).rmax;
  return MOE_OK;
}

int moe_pack_w13(int32_t G, int32_t Mw, int32_t d, const uint16_t* w1, const uint16_t* w3,
                 uint16_t* w13, void* stream) {
  if (G < 0 || Mw < 0 || d <= 0) return MOE_ERR_INVALID_ARG;
  if (Mw % 128 != 0 || d % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(G) * Mw == 0) return MOE_OK;
  if (!w1 || !w3 || !w13 || !aligned16(w1) || !aligned16(w3) || !aligned16(w13))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return cuda_rc(tracked(MOE_KERNEL_OTHER, st, [&] { return launch_pack_w13(G, Mw, d, w1, w3, w13, st); }));
}

int moe_route(const moe_shape_t* s, const uint16_t* x, const uint16_t* w_router,
              const float* logit_offset, const float* sel_bias, int32_t* ids, float* gates,
              int32_t* counts, float* f, float* P, float* bal_loss, float* z_loss, void* ws,
              size_t ws_bytes, void* stream) {
  int rc = check_shape(s);
  if (rc != MOE_OK) return rc;
  Layout L;
  if ((rc = check_ws(s, ws, ws_bytes, &L)) != MOE_OK) return rc;
  if (is_ec(s)) return MOE_ERR_INVALID_ARG;
  if (!counts || !f || !P || !bal_loss || !z_loss) return MOE_ERR_INVALID_ARG;
  if (s->T > 0) {
    if (!x || !w_router || !aligned16(x) || !aligned16(w_router)) return MOE_ERR_INVALID_ARG;
    if (s->k > 0 && (!ids || !gates)) return MOE_ERR_INVALID_ARG;
  }
  return do_route(s, x, w_router, logit_offset, sel_bias, ids, gates, counts, f, P, bal_loss,
                  z_loss, ws, L, false, nullptr, static_cast<cudaStream_t>(stream));
}

int moe_route_ex(const moe_shape_t* s, const uint16_t* x, const uint16_t* w_router,
                 const float* logit_offset, const float* sel_bias, const moe_route_out_t* o,
                 void* ws, size_t ws_bytes, void* stream) {
  int rc = check_shape(s);
  if (rc != MOE_OK) return rc;
  Layout L;
  if ((rc = check_ws(s, ws, ws_bytes, &L)) != MOE_OK) return rc;
  if (is_ec(s)) return MOE_ERR_INVALID_ARG;
  if (!o || !o->counts || !o->f || !o->P || !o->bal_loss || !o->z_loss) return MOE_ERR_INVALID_ARG;
  if (s->T > 0) {
    if (!x || !w_router || !aligned16(x) || !aligned16(w_router)) return MOE_ERR_INVALID_ARG;
    if (s->k > 0 && (!o->ids || !o->gates)) return MOE_ERR_INVALID_ARG;
  }
  return do_route(s, x, w_router, logit_offset, sel_bias, o->ids, o->gates, o->counts, o->f,
                  o->P, o->bal_loss, o->z_loss, ws, L, false, nullptr,
                  static_cast<cudaStream_t>(stream), o->importance, o->importance_cv2,
                  o->entropy_mean);
}

int moe_permute(const moe_shape_t* s, const uint16_t* x, const int32_t* ids, int32_t* offsets,
                int32_t* slot_row, int32_t* row_token, uint8_t* drop_mask, uint16_t* x_perm,
                void* ws, size_t ws_bytes, void* stream) {
  int rc = check_shape(s);
  if (rc != MOE_OK) return rc;
  Layout L;
  if ((rc = check_ws(s, ws, ws_bytes, &L)) != MOE_OK) return rc;
  if (is_ec(s)) return MOE_ERR_INVALID_ARG;
  if (is_priority(s)) return MOE_ERR_UNSUPPORTED;  // needs the router's pair scores
  if (!offsets) return MOE_ERR_INVALID_ARG;
  const bool work = s->T > 0 && s->k > 0;
  if (work && (!x || !ids || !slot_row || !row_token || !drop_mask || !x_perm ||
               !aligned16(x) || !aligned16(x_perm)))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* tile_hist = at<int32_t>(ws, L.tile_hist);
  if (work) {
    if ((rc = cuda_rc(tracked(MOE_KERNEL_TILE_HIST, st, [&] {
           return launch_tile_hist(ids, s->T, s->k, s->E, tile_hist, at<int>(ws, L.status), st);
         }))) != MOE_OK)
      return rc;
  }
  FinalizeArgs fa{};
  fa.T = work ? s->T : 0;
  fa.E = s->E;
  fa.k = s->k;
  fa.C = L.C;
  fa.tile_hist = tile_hist;
  fa.tile_base = at<int32_t>(ws, L.tile_base);
  fa.offsets = offsets;
  fa.exp_count = at<int32_t>(ws, L.exp_count);
  fa.exp_psum = at<double>(ws, L.exp_psum);
  fa.done_counter = at<int>(ws, L.status + 64);
  if ((rc = cuda_rc(tracked(MOE_KERNEL_FINALIZE, st, [&] { return launch_finalize(fa, st); }))) !=
      MOE_OK)
    return rc;
  if (!work) return MOE_OK;
  return do_scatter(s, x, ids, L, ws, offsets, slot_row, row_token, drop_mask, x_perm, st, 1);
}

int moe_grouped_ffn(const moe_shape_t* s, const uint16_t* x_perm, const int32_t* offsets,
                    const uint16_t* w13, const uint16_t* w2, uint16_t* y_perm, const uint16_t* x,
                    const uint16_t* w13_shared, const uint16_t* w2_shared, uint16_t* y_shared,
                    void* ws, size_t ws_bytes, void* stream) {
  int rc = check_shape(s);
  if (rc != MOE_OK) return rc;
  Layout L;
  if ((rc = check_ws(s, ws, ws_bytes, &L)) != MOE_OK) return rc;
  if (L.rmax > 0) {
    if (!x_perm || !offsets || !w13 || !w2 || !y_perm || !aligned16(x_perm) ||
        !aligned16(w13) || !aligned16(w2) || !aligned16(y_perm))
      return MOE_ERR_INVALID_ARG;
  }
  if (s->n_shared > 0 && s->T > 0) {
    if (!x || !w13_shared || !w2_shared || !y_shared || !aligned16(x) ||
        !aligned16(w13_shared) || !aligned16(w2_shared) || !aligned16(y_shared))
      return MOE_ERR_INVALID_ARG;
  }
  return do_ffn(s, x_perm, offsets, w13, w2, y_perm, x, w13_shared, w2_shared, y_shared, ws, L,
                static_cast<cudaStream_t>(stream));
}

int moe_combine(const moe_shape_t* s, const uint16_t* y_perm, const int32_t* slot_row,
                const float* gates, const uint16_t* y_shared, uint16_t* y, void* stream) {
  const int rc = check_shape(s);
  if (rc != MOE_OK) return rc;
  if (is_ec(s)) return MOE_ERR_INVALID_ARG;
  if (s->T == 0) return MOE_OK;
  if (!y || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  if (s->k > 0 && (!y_perm || !slot_row || !gates || !aligned16(y_perm)))
    return MOE_ERR_INVALID_ARG;
  if (y_shared && !aligned16(y_shared)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return cuda_rc(tracked(MOE_KERNEL_COMBINE, st, [&] {
    // no workspace: a failed index check (bounds-checked builds) skips the row
    // without recording it
    return launch_combine(s->T, s->d, s->k, y_perm, slot_row, gates, y_shared, y,
                          layout_of(s).rmax, nullptr, st, use_pdl(s));
  }));
}

int moe_layer_forward(const moe_shape_t* s, const uint16_t* x, const uint16_t* w_router,
                      const float* logit_offset, const float* sel_bias, const uint16_t* w13,
                      const uint16_t* w2, const uint16_t* w13_shared, const uint16_t* w2_shared,
                      uint16_t* y, int32_t* ids, float* gates, int32_t* counts,
                      uint8_t* drop_mask, float* f, float* P, float* bal_loss, float* z_loss,
                      void* ws, size_t ws_bytes, void* stream) {
  int rc = check_shape(s);
  if (rc != MOE_OK) return rc;
  Layout L;
  if ((rc = check_ws(s, ws, ws_bytes, &L)) != MOE_OK) return rc;
  if (is_ec(s)) return MOE_ERR_INVALID_ARG;
  if (!counts || !f || !P || !bal_loss || !z_loss) return MOE_ERR_INVALID_ARG;
  if (s->T > 0) {
    if (!x || !w_router || !y || !aligned16(x) || !aligned16(w_router) || !aligned16(y))
      return MOE_ERR_INVALID_ARG;
    if (s->k > 0 && (!ids || !gates || !drop_mask || !w13 || !w2 || !aligned16(w13) ||
                     !aligned16(w2)))
      return MOE_ERR_INVALID_ARG;
    if (s->n_shared > 0 && (!w13_shared || !w2_shared || !aligned16(w13_shared) ||
                            !aligned16(w2_shared)))
      return MOE_ERR_INVALID_ARG;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  const bool prio = is_priority(s);
  RouteExtras ex;
  if (prio) {
    ex.pair_score = at<float>(ws, L.pair_score);
    ex.all_offsets = at<int32_t>(ws, L.all_offsets);
  }
  rc = do_route(s, x, w_router, logit_offset, sel_bias, ids, gates, counts, f, P, bal_loss,
                z_loss, ws, L, true, offsets, st, nullptr, nullptr, nullptr, ex);
  if (rc != MOE_OK || s->T == 0) return rc;
  int32_t* slot_row = at<int32_t>(ws, L.slot_row);
  uint16_t* x_perm = at<uint16_t>(ws, L.x_perm);
  uint16_t* y_perm = at<uint16_t>(ws, L.y_perm);
  uint16_t* y_s = s->n_shared > 0 ? at<uint16_t>(ws, L.y_s) : nullptr;
  const bool fused = fused_gather(s);
  const bool gate_epi = gate_in_epilogue(s) && s->k > 0;
  int32_t* row_token = at<int32_t>(ws, L.row_token);
  float* row_gate = gate_epi ? at<float>(ws, L.row_gate) : nullptr;
  if (s->k > 0) {
    uint16_t* xp = fused ? nullptr : x_perm;
    if (prio)
      rc = do_priority_dispatch(s, x, ids, L, ws, offsets, slot_row, row_token, drop_mask, xp,
                                st, gates, row_gate);
    else
      rc = do_scatter(s, x, ids, L, ws, offsets, slot_row, row_token, drop_mask, xp, st,
                      L.chunk_tiles, gates, row_gate);
    if (rc != MOE_OK) return rc;
  }
  rc = do_ffn(s, fused ? nullptr : x_perm, offsets, w13, w2, y_perm, x, w13_shared, w2_shared,
              y_s, ws, L, st, fused ? row_token : nullptr, row_gate);
  if (rc != MOE_OK) return rc;
  const float* combine_gates = gate_epi ? nullptr : gates;
  return cuda_rc(tracked(MOE_KERNEL_COMBINE, st, [&] {
    return launch_combine(s->T, s->d, s->k, y_perm, slot_row, combine_gates, y_s, y, L.rmax,
                          at<int>(ws, L.status), st, use_pdl(s));
  }));
}

int moe_layer_forward_host(const moe_shape_t* s, const uint16_t* x_host, uint16_t* x_dev,
                           const uint16_t* w_router, const float* logit_offset,
                           const float* sel_bias, const uint16_t* w13, const uint16_t* w2,
                           const uint16_t* w13_shared, const uint16_t* w2_shared,
                           uint16_t* y_dev, uint16_t* y_host, float* losses_host, int32_t* ids,
                           float* gates, int32_t* counts, uint8_t* drop_mask, float* f,
                           float* P, float* bal_loss, float* z_loss, void* ws, size_t ws_bytes,
                           void* stream) {
  int rc = check_shape(s);
  if (rc != MOE_OK) return rc;
  if (s->T > 0 && (!x_host || !x_dev || !y_dev || !y_host)) return MOE_ERR_INVALID_ARG;
  if (!losses_host) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = static_cast<size_t>(s->T) * s->d * 2;
  if (bytes && cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  rc = moe_layer_forward(s, x_dev, w_router, logit_offset, sel_bias, w13, w2, w13_shared,
                         w2_shared, y_dev, ids, gates, counts, drop_mask, f, P, bal_loss, z_loss,
                         ws, ws_bytes, stream);
  if (rc != MOE_OK) return rc;
  if (bytes && cudaMemcpyAsync(y_host, y_dev, bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaMemcpyAsync(losses_host, bal_loss, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemcpyAsync(losses_host + 1, z_loss, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_layer_forward_host_batches(
    const moe_shape_t* s, int32_t n_batches, const uint16_t* x_host, uint16_t* y_host,
    float* losses_host, uint16_t* x_dev, uint16_t* y_dev, float* loss_dev,
    const uint16_t* w_router, const float* logit_offset, const float* sel_bias,
    const uint16_t* w13, const uint16_t* w2, const uint16_t* w13_shared, const uint16_t* w2_shared,
    int32_t* ids, float* gates, int32_t* counts, uint8_t* drop_mask, float* f, float* P,
    void* ws, size_t ws_bytes, void* stream, void* h2d_stream, void* d2h_stream) {
  int rc = check_shape(s);
  if (rc != MOE_OK) return rc;
  if (n_batches < 0 || !losses_host || !loss_dev) return MOE_ERR_INVALID_ARG;
  if (s->T > 0 && (!x_host || !x_dev || !y_dev || !y_host)) return MOE_ERR_INVALID_ARG;
  if (is_ec(s)) return MOE_ERR_INVALID_ARG;
  Layout L;  // the workspace is checked before anything is enqueued
  if ((rc = check_ws(s, ws, ws_bytes, &L)) != MOE_OK) return rc;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaStream_t hs = static_cast<cudaStream_t>(h2d_stream);
  cudaStream_t ds = static_cast<cudaStream_t>(d2h_stream);
  if (n_batches == 0) return MOE_OK;
  const size_t elems = static_cast<size_t>(s->T) * s->d;
  const size_t bytes = elems * 2;
  // per slot: x copied in, layer done, y and losses copied out
  cudaEvent_t in_done[2] = {}, fwd_done[2] = {}, out_done[2] = {};
  bool ev_ok = true;
  for (int a = 0; a < 2; ++a)
    ev_ok = ev_ok &&
            cudaEventCreateWithFlags(&in_done[a], cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&fwd_done[a], cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&out_done[a], cudaEventDisableTiming) == cudaSuccess;
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  rc = ev_ok ? MOE_OK : MOE_ERR_CUDA;
  for (int32_t i = 0; i < n_batches && rc == MOE_OK; ++i) {
    const int a = i & 1;
    uint16_t* xd = x_dev + a * elems;
    uint16_t* yd = y_dev + a * elems;
    float* ld = loss_dev + 2 * a;
    // copy in batch i once the layer of batch i-2 has read this x slot
    if (i >= 2 && !ok(cudaStreamWaitEvent(hs, fwd_done[a], 0))) { rc = MOE_ERR_CUDA; break; }
    if (bytes && !ok(cudaMemcpyAsync(xd, x_host + i * elems, bytes, cudaMemcpyHostToDevice, hs))) {
      rc = MOE_ERR_CUDA;
      break;
    }
    if (!ok(cudaEventRecord(in_done[a], hs)) || !ok(cudaStreamWaitEvent(cs, in_done[a], 0))) {
      rc = MOE_ERR_CUDA;
      break;
    }
    // the layer may overwrite this y slot once batch i-2 has been copied out
    if (i >= 2 && !ok(cudaStreamWaitEvent(cs, out_done[a], 0))) { rc = MOE_ERR_CUDA; break; }
    rc = moe_layer_forward(s, xd, w_router, logit_offset, sel_bias, w13, w2, w13_shared,
                           w2_shared, yd, ids, gates, counts, drop_mask, f, P, ld, ld + 1, ws,
                           ws_bytes, stream);
    if (rc != MOE_OK) break;
    if (!ok(cudaEventRecord(fwd_done[a], cs)) || !ok(cudaStreamWaitEvent(ds, fwd_done[a], 0))) {
      rc = MOE_ERR_CUDA;
      break;
    }
    if ((bytes && !ok(cudaMemcpyAsync(y_host + i * elems, yd, bytes, cudaMemcpyDeviceToHost, ds))) ||
        !ok(cudaMemcpyAsync(losses_host + 2 * static_cast<size_t>(i), ld, 8,
                            cudaMemcpyDeviceToHost, ds)) ||
        !ok(cudaEventRecord(out_done[a], ds))) {
      rc = MOE_ERR_CUDA;
      break;
    }
  }
  // wait for everything enqueued so far, whether or not a step failed
  const bool synced = ok(cudaStreamSynchronize(hs)) & ok(cudaStreamSynchronize(cs)) &
                      ok(cudaStreamSynchronize(ds));
  for (int a = 0; a < 2; ++a) {
    if (in_done[a]) cudaEventDestroy(in_done[a]);
    if (fwd_done[a]) cudaEventDestroy(fwd_done[a]);
    if (out_done[a]) cudaEventDestroy(out_done[a]);
  }
  if (rc == MOE_OK && !synced) rc = MOE_ERR_CUDA;
  return rc;
}

int moe_alf_bias_update(const moe_shape_t* s, const int32_t* counts, float gamma, float* bias,
                        void* stream) {
  const int rc = check_shape(s);
  if (rc != MOE_OK) return rc;
  if (!counts || !bias || !std::isfinite(gamma) || gamma < 0.0f) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return cuda_rc(tracked(MOE_KERNEL_OTHER, st, [&] {
    return launch_alf_bias_update(s->E, s->T, s->k, counts, gamma, bias, st);
  }));
}

int moe_ec_capacity(const moe_shape_t* s, int64_t* r) {
  const int rc = check_shape(s);
  if (rc != MOE_OK) return rc;
  if (!is_ec(s) || r == nullptr) return MOE_ERR_INVALID_ARG;
  *r = ec_capacity_of(s);
  return MOE_OK;
}

int moe_ec_route(const moe_shape_t* s, const uint16_t* x, const uint16_t* w_router,
                 const float* logit_offset, int32_t* row_token, float* row_gate, int32_t* counts,
                 float* f, float* P, float* bal_loss, float* z_loss, void* ws, size_t ws_bytes,
                 void* stream) {
  int rc = check_shape(s);
  if (rc != MOE_OK) return rc;
  if (!is_ec(s)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if ((rc = check_ws(s, ws, ws_bytes, &L)) != MOE_OK) return rc;
  if (!counts || !f || !P || !bal_loss || !z_loss) return MOE_ERR_INVALID_ARG;
  if (s->T > 0) {
    if (!x || !w_router || !aligned16(x) || !aligned16(w_router)) return MOE_ERR_INVALID_ARG;
    if (L.rmax > 0 && (!row_token || !row_gate)) return MOE_ERR_INVALID_ARG;
  }
  return do_ec_route(s, x, w_router, logit_offset, row_token, row_gate, counts, f, P, bal_loss,
                     z_loss, ws, L, static_cast<cudaStream_t>(stream));
}

int moe_ec_layer_forward(const moe_shape_t* s, const uint16_t* x, const uint16_t* w_router,
                         const float* logit_offset, const uint16_t* w13, const uint16_t* w2,
                         const uint16_t* w13_shared, const uint16_t* w2_shared, uint16_t* y,
                         int32_t* row_token, float* row_gate, int32_t* counts, float* f,
                         float* P, float* bal_loss, float* z_loss, void* ws, size_t ws_bytes,
                         void* stream) {
  int rc = check_shape(s);
  if (rc != MOE_OK) return rc;
  if (!is_ec(s)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if ((rc = check_ws(s, ws, ws_bytes, &L)) != MOE_OK) return rc;
  if (!counts || !f || !P || !bal_loss || !z_loss) return MOE_ERR_INVALID_ARG;
  if (s->T > 0) {
    if (!x || !w_router || !y || !aligned16(x) || !aligned16(w_router) || !aligned16(y))
      return MOE_ERR_INVALID_ARG;
    if (L.rmax > 0 && (!row_token || !row_gate || !w13 || !w2 || !aligned16(w13) ||
                       !aligned16(w2)))
      return MOE_ERR_INVALID_ARG;
    if (s->n_shared > 0 && (!w13_shared || !w2_shared || !aligned16(w13_shared) ||
                            !aligned16(w2_shared)))
      return MOE_ERR_INVALID_ARG;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  rc = do_ec_route(s, x, w_router, logit_offset, row_token, row_gate, counts, f, P, bal_loss,
                   z_loss, ws, L, st);
  if (rc != MOE_OK || s->T == 0) return rc;
  const int32_t* offsets = at<int32_t>(ws, L.offsets);
  uint16_t* x_perm = at<uint16_t>(ws, L.x_perm);
  uint16_t* y_perm = at<uint16_t>(ws, L.y_perm);
  uint16_t* y_s = s->n_shared > 0 ? at<uint16_t>(ws, L.y_s) : nullptr;
  const bool fused = fused_gather(s);
  if (L.rmax > 0 && !fused) {
    rc = cuda_rc(tracked(MOE_KERNEL_GATHER, st, [&] {
      return launch_gather_rows(x, row_token, offsets, s->E, s->d, L.rmax, x_perm,
                                sm_count_cached(), s->T, at<int>(ws, L.status), st);
    }));
    if (rc != MOE_OK) return rc;
  }
  const bool gate_epi = gate_in_epilogue(s) && L.rmax > 0;
  rc = do_ffn(s, fused ? nullptr : x_perm, offsets, w13, w2, y_perm, x, w13_shared, w2_shared,
              y_s, ws, L, st, fused ? row_token : nullptr, gate_epi ? row_gate : nullptr);
  if (rc != MOE_OK) return rc;
  const float* combine_gates = gate_epi ? nullptr : row_gate;
  return cuda_rc(tracked(MOE_KERNEL_COMBINE, st, [&] {
    return launch_ec_combine(s->T, s->d, s->E, at<int32_t>(ws, L.sel_t), combine_gates, y_perm,
                             y_s, y, L.rmax, at<int>(ws, L.status), st);
  }));
}

int moe_check_status(void* ws, int* status, void* stream) {
  if (!ws || !status) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  *status = (v == 0) ? MOE_OK : (v == kStatusBounds ? MOE_ERR_BOUNDS : MOE_ERR_TIMEOUT);
  return MOE_OK;
}

int moe_set_wait_timeout_ns(uint64_t ns) {
  if (ns == 0) return MOE_ERR_INVALID_ARG;
  g_timeout_ns.store(ns, std::memory_order_relaxed);
  return MOE_OK;
}

int moe_debug_timeout_probe(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < sizeof(int) || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0)
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return cuda_rc(tracked(MOE_KERNEL_OTHER, st, [&] {
    return launch_timeout_probe(static_cast<int*>(ws), default_wait_timeout_ns(), st);
  }));
}

int moe_profile_enable(int on) {
  g_prof_mask = (on == 0) ? 0u : (on == 1 ? 0xFFFFFFFFu : static_cast<uint32_t>(on));
  return MOE_OK;
}

int moe_profile_collect(int cap, int* n, int32_t* kernel_ids, float* ms) {
  if (!n || cap < 0 || (cap > 0 && (!kernel_ids || !ms))) return MOE_ERR_INVALID_ARG;
  int out = 0;
  int rc = MOE_OK;
  for (const ProfRec& r : g_prof) {
    if (out >= cap) break;
    float t = 0.0f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess ||
        cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess) {
      rc = MOE_ERR_CUDA;
      break;
    }
    kernel_ids[out] = r.kernel;
    ms[out] = t;
    ++out;
  }
  *n = out;
  g_prof.clear();
  g_ev_used = 0;
  return rc;
}

int moe_launch_count(uint64_t* n) {
  if (!n) return MOE_ERR_INVALID_ARG;
  *n = g_launches;
  return MOE_OK;
}

}  // extern "C"
