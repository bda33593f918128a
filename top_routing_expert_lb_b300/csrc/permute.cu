// Dispatch: loads, capacity cut and the permutation into expert-contiguous
// rows, plus the reduction of the router's per-tile partials.
//
// The CSDN note's moe_infer (DeepseekV3MoE excerpt) builds tokens_per_expert
// from a one-hot scatter, argsorts the flattened ids and gathers the token
// rows; the toy MoE demo keeps the first C tokens of each expert in token
// order.  Here the same result comes from integer work only:
//   1. per 128-token tile, an expert histogram (from the router, or
//      tile_hist_kernel);
//   2. counts n_e, kept_e = min(n_e, C) (C = ceil(c k T / E),
//      "MoE：条件计算与路由" §3), offsets = exclusive scan of kept_e, and
//      exclusive bases per chunk of tiles (the router's last CTA, chunks of up
//      to 32 tiles) or per tile (finalize_kernel, for ids given by the caller);
//   3. scatter_kernel: the rank of pair (t, s) among its expert's pairs in
//      token-major order is the tile's base (its chunk's base plus the counts
//      of the chunk's earlier tiles) + rank inside the tile (warp match +
//      per-warp counts); the pair is kept iff rank < C and lands on row
//      offsets[e] + rank.  Each token row is read once and written to each of
//      its kept rows.  With probability-priority capacity the same ranks
//      instead place every pair (and its score) in a per-expert staging list,
//      which the priority cut (select.cu) turns into rows.
// Every step is deterministic and bit-reproducible.
//
// finalize_kernel also reduces the side outputs in a fixed order:
// f_e = n_e / (k T), P_e = (1/T) sum_t p_e(t), L_bal = lambda E sum f_e P_e
// ("MoE：条件计算与路由" balance loss; P as in "MOE大模型对比篇" §2.1) and
// L_z = (1/T) sum_t lse_t^2 ("MOE大模型对比篇" §2.2).
#include <cuda_runtime.h>

#include "bounds.cuh"
#include "moe_internal.h"
#include "sm100_primitives.cuh"

namespace moe {

namespace {

__global__ void tile_hist_kernel(const int32_t* __restrict__ ids, int32_t T, int32_t k,
                                 int32_t E, int32_t* __restrict__ tile_hist, int* status) {
  __shared__ int hist[256];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int tile = blockIdx.x;
  const int t0 = tile * kTileTokens;
  const int pairs = min(kTileTokens, T - t0) * k;
  const int32_t* tid = ids + static_cast<int64_t>(t0) * k;
  for (int q = threadIdx.x; q < pairs; q += blockDim.x) {
    const int e = tid[q];
    if (idx_ok(e, E, status)) atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    tile_hist[static_cast<int64_t>(tile) * E + e] = hist[e];
}

constexpr int kFinThreads = 256;

// Exclusive scan of one int per thread over the block (fixed order).
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (kFinThreads / 32) ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < (kFinThreads / 32)) warp_tot[lane] = w;  // inclusive warp prefix
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_tot[warp - 1] : 0) + x - v;
  if (total) *total = warp_tot[kFinThreads / 32 - 1];
  __syncthreads();
  return before;
}

// Sum of one double per thread over the block, fixed tree order; result in
// thread 0.
__device__ __forceinline__ double block_sum(double v, double* red) {
  red[threadIdx.x] = v;
  __syncthreads();
  for (int s = kFinThreads / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  const double r = red[0];
  __syncthreads();
  return r;
}

// One CTA per expert: column scan of the tile histogram (tile bases), n_e
// and sum_t p_e.  The last CTA to finish reduces across experts: offsets of
// the kept rows, f, P and both losses.  Every sum has a fixed order.
__global__ void __launch_bounds__(kFinThreads) finalize_kernel(const FinalizeArgs a) {
  __shared__ int warp_tot[kFinThreads / 32];
  __shared__ double red[kFinThreads];
  __shared__ int is_last;
  const int E = a.E;
  const int ntiles = (a.T + kTileTokens - 1) / kTileTokens;
  const int e = blockIdx.x;
  // ---- phase A: column e
  int carry = 0;
  double psum = 0.0, isum = 0.0;
  for (int c0 = 0; c0 < ntiles; c0 += kFinThreads) {
    const int tl = c0 + threadIdx.x;
    const int64_t idx = static_cast<int64_t>(tl) * E + e;
    const int h = (tl < ntiles && a.fixed_count < 0) ? __ldcg(a.tile_hist + idx) : 0;
    if (a.tile_psum && tl < ntiles) psum += static_cast<double>(__ldcg(a.tile_psum + idx));
    if (a.tile_imp && tl < ntiles) isum += static_cast<double>(__ldcg(a.tile_imp + idx));
    int tot = 0;
    const int ex = block_exclusive_scan(h, warp_tot, &tot);
    if (a.tile_base && tl < ntiles) a.tile_base[idx] = carry + ex;
    carry += tot;
  }
  const double ps = block_sum(psum, red);
  const double is = a.tile_imp ? block_sum(isum, red) : 0.0;
  if (a.fixed_count >= 0) carry = a.fixed_count;
  if (threadIdx.x == 0) {
    a.exp_count[e] = carry;
    a.exp_psum[e] = ps;
    if (a.tile_imp) a.exp_imp[e] = is;
    __threadfence();
    is_last = (atomicAdd(a.done_counter, 1) == static_cast<int>(gridDim.x) - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // ---- phase B: across experts (E <= 256 = one per thread)
  const int j = threadIdx.x;
  const int n = j < E ? __ldcg(a.exp_count + j) : 0;
  const double pj = j < E ? __ldcg(a.exp_psum + j) : 0.0;
  const double n_pairs =
      a.n_pairs >= 0.0 ? a.n_pairs : static_cast<double>(a.k) * static_cast<double>(a.T);
  const double fe = (j < E && a.T > 0 && n_pairs > 0.0) ? static_cast<double>(n) / n_pairs : 0.0;
  const double Pe = (j < E && a.T > 0) ? pj / a.T : 0.0;
  if (j < E) {
    if (a.counts) a.counts[j] = n;
    if (a.f) a.f[j] = static_cast<float>(fe);
    if (a.P) a.P[j] = static_cast<float>(Pe);
  }
  const int kept = (j < E) ? ((a.C >= 0 && n > a.C) ? static_cast<int>(a.C) : n) : 0;
  int R = 0;
  const int off = block_exclusive_scan(kept, warp_tot, &R);
  if (a.offsets) {
    if (j < E) a.offsets[j] = off;
    if (j == 0) a.offsets[E] = R;
  }
  if (a.all_offsets) {
    int n_all = 0;
    const int off_all = block_exclusive_scan(j < E ? n : 0, warp_tot, &n_all);
    if (j < E) a.all_offsets[j] = off_all;
    if (j == 0) a.all_offsets[E] = n_all;
  }
  const double sfp = block_sum(fe * Pe, red);
  double z = 0.0;
  if (a.tile_lse2)
    for (int tl = j; tl < ntiles; tl += kFinThreads) z += static_cast<double>(__ldcg(a.tile_lse2 + tl));
  const double zs = block_sum(z, red);
  if (a.tile_imp) {
    // importance per expert and its squared coefficient of variation
    // (population statistics over the E experts)
    const double imp = j < E ? __ldcg(a.exp_imp + j) : 0.0;
    if (j < E && a.importance) a.importance[j] = static_cast<float>(imp);
    const double mean = block_sum(imp, red) / E;
    const double dev = j < E ? (imp - mean) * (imp - mean) : 0.0;
    const double var = block_sum(dev, red) / E;
    if (j == 0 && a.importance_cv2)
      *a.importance_cv2 = static_cast<float>(mean != 0.0 ? var / (mean * mean) : 0.0);
  }
  if (a.tile_ent) {
    double h = 0.0;
    for (int tl = j; tl < ntiles; tl += kFinThreads) h += static_cast<double>(__ldcg(a.tile_ent + tl));
    const double hs = block_sum(h, red);
    if (j == 0 && a.entropy_mean) *a.entropy_mean = (a.T > 0) ? static_cast<float>(hs / a.T) : 0.0f;
  }
  if (j == 0) {
    if (a.bal_loss) *a.bal_loss = static_cast<float>(static_cast<double>(a.balance_coef) * E * sfp);
    if (a.z_loss) *a.z_loss = (a.T > 0) ? static_cast<float>(zs / a.T) : 0.0f;
    *a.done_counter = 0;  // ready for the next call on this workspace
  }
}

constexpr int kScatterThreads = 256;
constexpr int kScatterWarps = kScatterThreads / 32;
constexpr int kGatherUnroll = 4;

// grid = (tiles, G): the G CTAs of a tile all compute the tile's destination
// rows (cheap integer work on <= 1024 pairs); CTA 0 publishes the slot rows,
// drop mask and row->token map, and each CTA gathers 1/G of the tile's tokens.
__global__ void __launch_bounds__(kScatterThreads) scatter_kernel(const ScatterArgs a) {
  __shared__ int run[256];                      // pairs of e seen in earlier rounds
  __shared__ int wcnt[kScatterWarps][256];      // pairs of e per warp, this round
  __shared__ int base[256];                     // tile_base
  __shared__ int rows[kTileTokens * kMaxTopK];  // destination row per pair (-1 dropped)
  pdl_wait();  // ids, offsets and bases come from the router
  const int E = a.E, k = a.k;
  const int tile = blockIdx.x;
  const int t0 = tile * kTileTokens;
  const int ntok = min(kTileTokens, a.T - t0);
  const int pairs = ntok * k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this tile's base per expert: its chunk's base plus the counts of the
  // chunk's earlier tiles (chunk_tiles = 1: a per-tile base)
  const int chunk = tile / a.chunk_tiles;
  const int first = chunk * a.chunk_tiles;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    run[e] = 0;
    int b = a.tile_base[static_cast<int64_t>(chunk) * E + e];
    for (int tt = first; tt < tile; ++tt) b += __ldg(a.tile_hist + static_cast<int64_t>(tt) * E + e);
    base[e] = b;
#pragma unroll
    for (int w = 0; w < kScatterWarps; ++w) wcnt[w][e] = 0;
  }
  __syncthreads();
  const int32_t* tid = a.ids + static_cast<int64_t>(t0) * k;
  const unsigned lt_mask = (1u << lane) - 1u;
  const bool staging = a.stage_q != nullptr;
  for (int q0 = 0; q0 < pairs; q0 += kScatterThreads) {
    const int q = q0 + threadIdx.x;
    bool active = q < pairs;
    int e = active ? tid[q] : -1;
    if (kBoundsChecked && active && !idx_ok(e, E, a.status)) {
      active = false;  // an expert id outside [0, E): the pair is left unplaced
      e = -1;
      rows[q] = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank_w = __popc(peers & lt_mask);
    if (active && rank_w == 0) wcnt[warp][e] = __popc(peers);
    __syncthreads();
    if (active) {
      int r = run[e] + rank_w;
      for (int w = 0; w < warp; ++w) r += wcnt[w][e];
      const int64_t rank = static_cast<int64_t>(base[e]) + r;  // rank within expert
      if (staging) {
        rows[q] = static_cast<int>(a.all_offsets[e] + rank);
      } else {
        const bool kept = (a.C < 0) || (rank < a.C);
        rows[q] = kept ? static_cast<int>(a.offsets[e] + rank) : -1;
      }
    }
    __syncthreads();
    for (int ee = threadIdx.x; ee < E; ee += blockDim.x) {
      int s = 0;
#pragma unroll
      for (int w = 0; w < kScatterWarps; ++w) {
        s += wcnt[w][ee];
        wcnt[w][ee] = 0;
      }
      run[ee] += s;
    }
    __syncthreads();
  }
  if (staging) {
    for (int q = threadIdx.x; q < pairs; q += blockDim.x) {
      const int64_t gq = static_cast<int64_t>(t0) * k + q;
      if (!idx_ok(rows[q], a.rmax, a.status)) continue;
      a.stage_q[rows[q]] = static_cast<int32_t>(gq);
      a.stage_key[rows[q]] = __ldg(a.pair_score + gq);
    }
    return;
  }
  if (blockIdx.y == 0) {
    for (int q = threadIdx.x; q < pairs; q += blockDim.x) {
      const int row = rows[q];
      const int64_t gq = static_cast<int64_t>(t0) * k + q;
      a.slot_row[gq] = row;
      if (a.drop_mask) a.drop_mask[gq] = row < 0 ? 1 : 0;
      if (row >= 0 && idx_ok(row, a.rmax, a.status)) {
        a.row_token[row] = t0 + q / k;
        if (a.row_gate) a.row_gate[row] = a.gates[gq];
      }
    }
  }
  if (a.x_perm == nullptr) return;  // rows only: the GEMM gathers the token rows itself
  // gather this CTA's share of tokens: warp per token, the row is read once
  const int G = gridDim.y;
  const int per = (ntok + G - 1) / G;
  const int tb = blockIdx.y * per;
  const int te = min(ntok, tb + per);
  const int nvec = a.d / 8;  // 16-byte vectors per row
  for (int tl = tb + warp; tl < te; tl += kScatterWarps) {
    const int t = t0 + tl;
    int dst[kMaxTopK];
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s) {
      dst[s] = (s < k) ? rows[tl * k + s] : -1;
      if (dst[s] >= 0 && !idx_ok(dst[s], a.rmax, a.status)) dst[s] = -1;
    }
    const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(t) * a.d);
    for (int v0 = lane; v0 < nvec; v0 += 32 * kGatherUnroll) {
      uint4 val[kGatherUnroll];
#pragma unroll
      for (int u = 0; u < kGatherUnroll; ++u)
        if (v0 + 32 * u < nvec) val[u] = __ldg(src + v0 + 32 * u);
#pragma unroll
      for (int u = 0; u < kGatherUnroll; ++u) {
        if (v0 + 32 * u < nvec) {
#pragma unroll
          for (int s = 0; s < kMaxTopK; ++s)
            if (dst[s] >= 0)
              reinterpret_cast<uint4*>(a.x_perm + static_cast<int64_t>(dst[s]) * a.d)[v0 + 32 * u] =
                  val[u];
        }
      }
    }
  }
}

}  // namespace

int launch_tile_hist(const int32_t* ids, int32_t T, int32_t k, int32_t E, int32_t* tile_hist,
                     int* status, cudaStream_t stream) {
  const int ntiles = (T + kTileTokens - 1) / kTileTokens;
  if (ntiles == 0) return 0;
  tile_hist_kernel<<<ntiles, 256, 0, stream>>>(ids, T, k, E, tile_hist, status);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_finalize(const FinalizeArgs& args, cudaStream_t stream) {
  if (args.E > kFinThreads) return -2;
  finalize_kernel<<<args.E, kFinThreads, 0, stream>>>(args);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_scatter(const ScatterArgs& args, cudaStream_t stream) {
  const int ntiles = (args.T + kTileTokens - 1) / kTileTokens;
  if (ntiles == 0 || args.k == 0) return 0;
  // enough CTAs to keep every SM streaming rows (about 4 per SM)
  int G = (4 * args.num_sms + ntiles - 1) / ntiles;
  G = G < 1 ? 1 : (G > 16 ? 16 : G);
  if (args.stage_q || args.x_perm == nullptr) G = 1;  // indices only, no row copies
  if (launch_kernel(scatter_kernel, dim3(ntiles, G), dim3(kScatterThreads), 0, stream,
                    args.pdl != 0, 1u, args) != cudaSuccess)
    return -3;
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace moe
