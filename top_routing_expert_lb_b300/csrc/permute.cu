// Dispatch: loads, capacity cut and the permutation into expert-contiguous
// rows, plus the reduction of the router's per-tile partials.
//
// The CSDN note's moe_infer (DeepseekV3MoE excerpt) builds tokens_per_expert
// from a one-hot scatter, argsorts the flattened ids and gathers the token
// rows; the toy MoE demo keeps the first C tokens of each expert in token
// order.  Here the same result comes from integer work only:
//   1. per 128-token tile, an expert histogram (from the router, or
//      tile_hist_kernel);
//   2. finalize_kernel: counts n_e, kept_e = min(n_e, C)
//      (C = ceil(c k T / E), "MoE：条件计算与路由" §3), offsets = exclusive scan
//      of kept_e, and per-tile exclusive bases tile_base[tile][e];
//   3. scatter_kernel: the rank of pair (t, s) among its expert's pairs in
//      token-major order is tile_base + rank inside the tile (warp match +
//      per-warp counts); the pair is kept iff rank < C and lands on row
//      offsets[e] + rank.  Each token row is read once and written to each of
//      its kept rows.
// Every step is deterministic and bit-reproducible.
//
// finalize_kernel also reduces the side outputs in a fixed order:
// f_e = n_e / (k T), P_e = (1/T) sum_t p_e(t), L_bal = lambda E sum f_e P_e
// ("MoE：条件计算与路由" balance loss; P as in "MOE大模型对比篇" §2.1) and
// L_z = (1/T) sum_t lse_t^2 ("MOE大模型对比篇" §2.2).
#include <cuda_runtime.h>

#include "moe_internal.h"

namespace moe {

namespace {

__global__ void tile_hist_kernel(const int32_t* __restrict__ ids, int32_t T, int32_t k,
                                 int32_t E, int32_t* __restrict__ tile_hist) {
  __shared__ int hist[256];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int tile = blockIdx.x;
  const int t0 = tile * kTileTokens;
  const int pairs = min(kTileTokens, T - t0) * k;
  const int32_t* tid = ids + static_cast<int64_t>(t0) * k;
  for (int q = threadIdx.x; q < pairs; q += blockDim.x) atomicAdd(&hist[tid[q]], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    tile_hist[static_cast<int64_t>(tile) * E + e] = hist[e];
}

__global__ void __launch_bounds__(256) finalize_kernel(const FinalizeArgs a) {
  __shared__ double fp[256];
  __shared__ int kept[256];
  const int E = a.E;
  const int ntiles = (a.T + kTileTokens - 1) / kTileTokens;
  const int e = threadIdx.x;
  if (e < E) {
    int run = 0;
    double psum = 0.0;
    for (int tl = 0; tl < ntiles; ++tl) {
      const int64_t idx = static_cast<int64_t>(tl) * E + e;
      if (a.tile_base) a.tile_base[idx] = run;
      run += a.tile_hist[idx];
      if (a.tile_psum) psum += static_cast<double>(a.tile_psum[idx]);
    }
    if (a.counts) a.counts[e] = run;
    const double fe = (a.T > 0 && a.k > 0) ? static_cast<double>(run) /
                                                 (static_cast<double>(a.k) * a.T)
                                           : 0.0;
    const double Pe = (a.T > 0) ? psum / a.T : 0.0;
    if (a.f) a.f[e] = static_cast<float>(fe);
    if (a.P) a.P[e] = static_cast<float>(Pe);
    fp[e] = fe * Pe;
    kept[e] = (a.C >= 0 && run > a.C) ? static_cast<int>(a.C) : run;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (a.offsets) {
      int acc = 0;
      for (int j = 0; j < E; ++j) {
        a.offsets[j] = acc;
        acc += kept[j];
      }
      a.offsets[E] = acc;
    }
    if (a.bal_loss) {
      double s = 0.0;
      for (int j = 0; j < E; ++j) s += fp[j];
      *a.bal_loss = static_cast<float>(static_cast<double>(a.balance_coef) * E * s);
    }
    if (a.z_loss) {
      double z = 0.0;
      if (a.tile_lse2)
        for (int tl = 0; tl < ntiles; ++tl) z += static_cast<double>(a.tile_lse2[tl]);
      *a.z_loss = (a.T > 0) ? static_cast<float>(z / a.T) : 0.0f;
    }
  }
}

constexpr int kScatterThreads = 256;
constexpr int kScatterWarps = kScatterThreads / 32;

__global__ void __launch_bounds__(kScatterThreads) scatter_kernel(const ScatterArgs a) {
  __shared__ int run[256];                      // pairs of e seen in earlier rounds
  __shared__ int wcnt[kScatterWarps][256];      // pairs of e per warp, this round
  __shared__ int base[256];                     // tile_base + offsets
  __shared__ int rows[kTileTokens * kMaxTopK];  // destination row per pair (-1 dropped)
  const int E = a.E, k = a.k;
  const int tile = blockIdx.x;
  const int t0 = tile * kTileTokens;
  const int ntok = min(kTileTokens, a.T - t0);
  const int pairs = ntok * k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    run[e] = 0;
    base[e] = a.tile_base[static_cast<int64_t>(tile) * E + e];
#pragma unroll
    for (int w = 0; w < kScatterWarps; ++w) wcnt[w][e] = 0;
  }
  __syncthreads();
  const int32_t* tid = a.ids + static_cast<int64_t>(t0) * k;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int q0 = 0; q0 < pairs; q0 += kScatterThreads) {
    const int q = q0 + threadIdx.x;
    const bool active = q < pairs;
    const int e = active ? tid[q] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank_w = __popc(peers & lt_mask);
    if (active && rank_w == 0) wcnt[warp][e] = __popc(peers);
    __syncthreads();
    if (active) {
      int r = run[e] + rank_w;
      for (int w = 0; w < warp; ++w) r += wcnt[w][e];
      const int64_t rank = static_cast<int64_t>(base[e]) + r;  // rank within expert
      const bool kept = (a.C < 0) || (rank < a.C);
      rows[q] = kept ? static_cast<int>(a.offsets[e] + rank) : -1;
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
  // slot rows, drop mask, row -> token
  for (int q = threadIdx.x; q < pairs; q += blockDim.x) {
    const int row = rows[q];
    const int64_t gq = static_cast<int64_t>(t0) * k + q;
    a.slot_row[gq] = row;
    if (a.drop_mask) a.drop_mask[gq] = row < 0 ? 1 : 0;
    if (row >= 0) a.row_token[row] = t0 + q / k;
  }
  // gather: warp per token, the token row is read once
  const int nvec = a.d / 8;  // 16-byte vectors per row
  for (int tl = warp; tl < ntok; tl += kScatterWarps) {
    const int t = t0 + tl;
    int dst[kMaxTopK];
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s) dst[s] = (s < k) ? rows[tl * k + s] : -1;
    const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(t) * a.d);
    for (int v = lane; v < nvec; v += 32) {
      const uint4 val = src[v];
#pragma unroll
      for (int s = 0; s < kMaxTopK; ++s)
        if (dst[s] >= 0)
          reinterpret_cast<uint4*>(a.x_perm + static_cast<int64_t>(dst[s]) * a.d)[v] = val;
    }
  }
}

}  // namespace

int launch_tile_hist(const int32_t* ids, int32_t T, int32_t k, int32_t E, int32_t* tile_hist,
                     cudaStream_t stream) {
  const int ntiles = (T + kTileTokens - 1) / kTileTokens;
  if (ntiles == 0) return 0;
  tile_hist_kernel<<<ntiles, 256, 0, stream>>>(ids, T, k, E, tile_hist);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_finalize(const FinalizeArgs& args, cudaStream_t stream) {
  finalize_kernel<<<1, 256, 0, stream>>>(args);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_scatter(const ScatterArgs& args, cudaStream_t stream) {
  const int ntiles = (args.T + kTileTokens - 1) / kTileTokens;
  if (ntiles == 0 || args.k == 0) return 0;
  scatter_kernel<<<ntiles, kScatterThreads, 0, stream>>>(args);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace moe
