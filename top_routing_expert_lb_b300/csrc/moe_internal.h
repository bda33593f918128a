// Internal launcher interfaces shared by the .cu files of libmoe_b300.so.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace moe {

constexpr int kTileTokens = 128;  // tokens per router / permute tile (= MMA M)
constexpr int kMaxTopK = 8;
constexpr int kMaxSplitUnits = 8;  // largest K split of a router tile
// routing variants (the values of MOE_FLAG_SIGMOID / MOE_FLAG_NO_RENORM)
constexpr uint32_t kRouteSigmoid = 1u;
constexpr uint32_t kRouteNoRenorm = 2u;
constexpr uint32_t kRoutePriority = 4u;      // capacity keeps the highest scores
constexpr uint32_t kRouteExpertChoice = 8u;  // experts pick tokens

// Launches `kern` on `stream`.  With pdl, the launch allows programmatic
// dependent launch: the kernel's CTAs may start while the previous kernel in
// the stream is still running (after every CTA of that kernel has started),
// so launch latency and the prologue (barrier set-up, TMEM allocation,
// descriptor prefetch) overlap its tail; the kernel waits (pdl_wait) before
// it touches memory that earlier work wrote.  cluster_x > 1 launches clusters
// of that many CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, bool pdl, unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  unsigned n = 0;
  if (pdl) {
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = cluster_x;
    attrs[n].val.clusterDim.y = 1;
    attrs[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Ragged grouped GEMM  out[g] = A[g] * B[g]^T  over E routed groups (rows from
// device offsets) and an optional shared group (fixed row count).
struct GroupedGemmArgs {
  const int32_t* offsets;  // [E+1] device, routed group row ranges in A0 / out0
  int32_t n_routed;        // number of routed groups (0 if none)
  int32_t shared_rows;     // rows of the shared group (0 = no shared group)
  int32_t n_cols_routed;   // N of every routed group
  int32_t n_cols_shared;   // N of the shared group
  int32_t k_routed;        // K of the routed groups (multiple of 64)
  int32_t k_shared;        // K of the shared group (multiple of 64)
  void* out_routed;        // bf16 [rows][ld_routed]
  int64_t ld_routed;
  void* out_shared;        // bf16 [shared_rows][ld_shared]
  int64_t ld_shared;
  int* status;             // device status word
  uint64_t timeout_ns;
  // When set (single-CTA kernel only), routed A rows are gathered: row r of
  // the routed activations is row gather_rows[r] of the tensor behind A0,
  // whose map then has a 64 x 1 box.
  const int32_t* gather_rows = nullptr;
  // 0: every row of each group; 1: only its whole 256-row blocks; 2: only the
  // rows after them (fewer than 256).  One projection can thus run its long
  // blocks on CTA pairs and the remainders on single CTAs.
  int32_t row_split = 0;
  // A group's last m-tile with r valid rows runs transposed when r rounded up
  // to 16 is at most tail_max_n (0: never), and, unless swap_all_tails, only
  // when it is the group's only m-tile.
  int32_t tail_max_n = 112;
  int32_t swap_all_tails = 0;
  // Single-CTA kernel with BN = 256 (no row scaling): two CTAs per SM, each
  // with a 2-stage ring and one TMEM accumulator.
  int32_t two_per_sm = 0;
  // Plain projection only: routed output row r is scaled by row_scale[r]
  // (fp32, before rounding); the shared group is never scaled.
  const float* row_scale = nullptr;
  // Tile order inside a group with more than block_min_rows rows: blocks of
  // n_block n-tiles, m-tile major inside a block (n_block <= 1: n-tile major
  // throughout).
  int32_t n_block = 8;
  int32_t block_min_rows = 2048;
  // Pair kernel: when set, tiles are taken dynamically from this counter
  // ([0] next tile, [1] CTAs done; both zero before the launch, and left zero
  // by it); null: static round-robin schedule.
  int* tile_counter = nullptr;
  // Pair kernel: a group's last tile with at most 128 rows runs as one M = 128
  // pair MMA (half the padding) instead of a 256-row tile.
  int32_t half_tiles = 1;
  // Bounds-checked builds: rows of the two outputs and of the gathered tensor
  int64_t out_rows_routed = INT64_MAX;
  int64_t out_rows_shared = INT64_MAX;
  int64_t gather_limit = INT64_MAX;
  int32_t pdl = 0;  // launch with programmatic dependent launch (see launch_kernel)
};

// A0/A1: activations [rows][K] (routed / shared), B0/B1: weights [rows][K].
// swiglu: epilogue writes h = SiLU(acc[:, :128]) * acc[:, 128:] per 256-wide
// tile (packed gate/up weights); else writes acc as bf16.
// paired: 256 x 256 tiles on CTA pairs (tcgen05 cta_group::2; bn must be 256;
// the B tensor maps then use 128-row boxes); else 128 x bn tiles per CTA.
// b0h / b1h (paired SwiGLU only): the same B tensors with 64-row boxes, for
// the half-height tiles that end a group with at most 128 rows.
// o0 / o1: the routed / shared outputs (out_routed, out_shared) as tensor maps
// from make_tmap_out_bf16; the epilogue writes every 32-row block of a tile
// whose rows are all valid through them.
int launch_grouped_gemm(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0,
                        const CUtensorMap& b1, const CUtensorMap& o0, const CUtensorMap& o1,
                        const GroupedGemmArgs& args, bool swiglu, int bn, bool paired,
                        int num_sms, cudaStream_t stream, const CUtensorMap* b0h = nullptr,
                        const CUtensorMap* b1h = nullptr);

// Encodes a 2-D bf16 tensor map over a row-major [rows][cols] tensor with a
// 64-column x box_rows box and 128-byte swizzle.  Returns false on failure.
bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows);

// The GEMM outputs' tensor maps: bf16 [rows][cols] row-major, 32 x 32 boxes
// with 64-byte swizzle (the epilogue's staging layout).  cols must be a
// multiple of 8.  Returns false on failure.
bool make_tmap_out_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols);

// Router: logits tile GEMM + softmax / bias / Top-k epilogue on a persistent
// grid, and the reduction of the side outputs by the CTA that completes the
// last tile.  Accumulators (acc_*, tiles_done, tile_arrive, chunk_acc) must be
// zero before the launch; the kernel leaves them at zero.
struct RouterArgs {
  int32_t T, d, E, k;
  const float* logit_offset;  // [E] or null
  const float* sel_bias;      // [E] or null
  int32_t* ids;               // [T][k]
  float* gates;               // [T][k]
  int* status;
  uint64_t timeout_ns;
  uint32_t flags;             // kRouteSigmoid | kRouteNoRenorm
  int32_t max_split = kMaxSplitUnits;  // largest K split the caller's scratch allows
  int32_t split = 1;          // set by the launcher
  int32_t stages = 1;         // set by the launcher
  float* pair_score = nullptr;  // [T][k] unbiased score of each selected pair, or null
  float* scores_t = nullptr;    // [E][T] every score, expert-major, or null
  // scratch
  float* part_logits = nullptr;         // [S][ntiles][E][128] partial logits (K split)
  int* tile_arrive = nullptr;           // [ntiles] slices stored per tile (K split)
  float* tile_lse2 = nullptr;           // [ntiles] sum of lse^2 over each tile's rows
  int* tiles_done = nullptr;            // [1]
  int* acc_count = nullptr;             // [E] pairs per expert
  unsigned long long* acc_psum = nullptr;  // [E] sum of scores, fixed point 2^-32
  unsigned long long* acc_imp = nullptr;   // [E] importance, fixed point, or null
  unsigned long long* acc_ent = nullptr;   // [1] entropy sum, fixed point, or null
  int32_t* tile_hist = nullptr;         // [ntiles][E] per-tile counts, or null
  int32_t* chunk_acc = nullptr;         // [n_chunks][E] counts per chunk of tiles, or null
  int32_t* chunk_base = nullptr;        // [n_chunks][E] exclusive scan of chunk_acc over chunks
  int32_t chunk_tiles = 1;              // tiles per chunk
  int32_t n_chunks = 0;
  // outputs of the reduction
  int64_t C = -1;                       // capacity or -1
  float balance_coef = 0.0f;
  int32_t* counts = nullptr;            // [E]
  float* f = nullptr;                   // [E]
  float* P = nullptr;                   // [E]
  float* bal_loss = nullptr;            // [1]
  float* z_loss = nullptr;              // [1]
  int32_t* offsets = nullptr;           // [E+1] kept-row offsets, or null
  int32_t* all_offsets = nullptr;       // [E+1] offsets before capacity, or null
  float* importance = nullptr;          // [E] or null
  float* importance_cv2 = nullptr;      // [1] or null
  float* entropy_mean = nullptr;        // [1] or null
  int32_t fixed_count = -1;             // >= 0: every expert's count (expert choice)
  double n_pairs = -1.0;                // denominator of f; < 0: k T
  int32_t pdl = 0;                      // programmatic dependent launch (see launch_kernel)
};
int launch_router(const CUtensorMap& x_map, const CUtensorMap& wr_map, RouterArgs args,
                  int num_sms, cudaStream_t stream);
// K split the router takes for this shape (1 = none).
int router_split(int T, int d, int num_sms, int max_split);

// Per-tile expert histogram of ids (when the router did not produce it).
int launch_tile_hist(const int32_t* ids, int32_t T, int32_t k, int32_t E, int32_t* tile_hist,
                     int* status, cudaStream_t stream);

// Reduces the per-tile partials: counts, f, P, losses (optional) and the
// permutation scan (offsets of kept rows, per-tile bases).
struct FinalizeArgs {
  int32_t T, E, k;
  int64_t C;                  // capacity or -1
  float balance_coef;
  const int32_t* tile_hist;   // [ntiles][E]
  const float* tile_psum;     // [ntiles][E] or null (no losses)
  const float* tile_lse2;     // [ntiles] or null
  int32_t* counts;            // [E] or null
  float* f;                   // [E] or null
  float* P;                   // [E] or null
  float* bal_loss;            // [1] or null
  float* z_loss;              // [1] or null
  int32_t* tile_base;         // [ntiles][E] or null (no scan)
  int32_t* offsets;           // [E+1] or null
  int32_t* exp_count;         // [E] scratch: per-expert totals
  double* exp_psum;           // [E] scratch
  int* done_counter;          // zero between calls; the last CTA resets it
  const float* tile_imp;      // [ntiles][E] or null
  const float* tile_ent;      // [ntiles] or null
  double* exp_imp;            // [E] scratch (when tile_imp)
  float* importance;          // [E] or null
  float* importance_cv2;      // [1] or null
  float* entropy_mean;        // [1] or null
  int32_t fixed_count = -1;   // >= 0: every expert's count (expert choice); -1: from tile_hist
  double n_pairs = -1.0;      // denominator of f; < 0: k T (E r for expert choice)
  int32_t* all_offsets = nullptr;  // [E+1] scan of the counts before capacity, or null
};
int launch_finalize(const FinalizeArgs& args, cudaStream_t stream);

// Capacity cut + permutation + row gather, one CTA per 128-token tile.
struct ScatterArgs {
  int32_t T, d, E, k;
  int64_t C;
  const int32_t* ids;        // [T][k]
  // base of tile t for expert e: tile_base[(t / chunk_tiles) E + e] plus the
  // counts of the chunk's earlier tiles, tile_hist[t' E + e]
  const int32_t* tile_base;  // [ceil(ntiles / chunk_tiles)][E]
  const int32_t* tile_hist = nullptr;  // [ntiles][E] (chunk_tiles > 1)
  int32_t chunk_tiles = 1;
  const int32_t* offsets;    // [E+1]
  const uint16_t* x;         // [T][d]
  int32_t* slot_row;         // [T][k]
  int32_t* row_token;        // [R_max]
  uint8_t* drop_mask;        // [T][k] or null
  uint16_t* x_perm;          // [R_max][d]
  int32_t num_sms;           // sizes the gather split
  // when set, the gate of each kept pair is written to its row (row_gate[row])
  const float* gates = nullptr;  // [T][k]
  float* row_gate = nullptr;     // [R_max]
  // staging mode (priority capacity): when stage_q is set, the pair at rank r
  // of expert e goes to stage_q/stage_key[all_offsets[e] + r] instead (its
  // flat index and pair_score); nothing else is written
  int32_t* stage_q = nullptr;          // [T*k] or null
  float* stage_key = nullptr;          // [T*k]
  const float* pair_score = nullptr;   // [T][k]
  const int32_t* all_offsets = nullptr;  // [E+1]
  int64_t rmax = 0;                    // rows of x_perm / row_token / row_gate (staging: T k)
  int* status = nullptr;               // bounds-checked builds: where a failed check is recorded
  int32_t pdl = 0;                     // programmatic dependent launch (see launch_kernel)
};
int launch_scatter(const ScatterArgs& args, cudaStream_t stream);

// Priority capacity cut over the staged pairs: one CTA per expert.
struct PrioritySelectArgs {
  int32_t E, k;
  int64_t C;
  const int32_t* all_offsets;  // [E+1] staging segments
  const int32_t* offsets;      // [E+1] kept-row offsets
  const int32_t* stage_q;      // [T*k]
  const float* stage_key;      // [T*k]
  int32_t* slot_row;           // [T][k]
  uint8_t* drop_mask;          // [T][k] or null
  int32_t* row_token;          // [R]
  const float* gates = nullptr;  // [T][k]; with row_gate, each kept row gets its gate
  float* row_gate = nullptr;     // [R] or null
  int64_t rmax = 0;              // rows of row_token / row_gate
  int64_t n_pairs = 0;           // T k: pair numbers in stage_q lie below
  int* status = nullptr;         // bounds-checked builds
};
int launch_priority_select(const PrioritySelectArgs& args, cudaStream_t stream);

// Expert choice: expert e takes the r largest scores of scores_t[e][0..T).
struct EcSelectArgs {
  int32_t T, E, r;
  const float* scores_t;  // [E][T]
  int32_t* sel_t;         // [E][T] row of (e, t), or -1
  int32_t* row_token;     // [E*r]
  float* row_gate;        // [E*r]
};
int launch_ec_select(const EcSelectArgs& args, cudaStream_t stream);

// x_perm[row] = x[row_token[row]] for row < offsets[E] (read on the device).
// x_rows: rows of x (row_token values must lie below); status: bounds-checked
// builds record a failed index check there (null: not recorded).
int launch_gather_rows(const uint16_t* x, const int32_t* row_token, const int32_t* offsets,
                       int32_t E, int32_t d, int64_t max_rows, uint16_t* x_perm, int num_sms,
                       int64_t x_rows, int* status, cudaStream_t stream);

// rmax: rows of y_perm (every row index read must lie below).
int launch_ec_combine(int32_t T, int32_t d, int32_t E, const int32_t* sel_t,
                      const float* row_gate, const uint16_t* y_perm, const uint16_t* y_shared,
                      uint16_t* y, int64_t rmax, int* status, cudaStream_t stream);

int launch_combine(int32_t T, int32_t d, int32_t k, const uint16_t* y_perm,
                   const int32_t* slot_row, const float* gates, const uint16_t* y_shared,
                   uint16_t* y, int64_t rmax, int* status, cudaStream_t stream,
                   bool pdl = false);

int launch_pack_w13(int32_t G, int32_t Mw, int32_t d, const uint16_t* w1, const uint16_t* w3,
                    uint16_t* w13, cudaStream_t stream);

int launch_timeout_probe(int* status, uint64_t timeout_ns, cudaStream_t stream);

int launch_alf_bias_update(int32_t E, int32_t T, int32_t k, const int32_t* counts, float gamma,
                           float* bias, cudaStream_t stream);

// The process-wide limit of bounded device waits (moe_set_wait_timeout_ns).
uint64_t default_wait_timeout_ns();

}  // namespace moe
