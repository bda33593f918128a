// Score-ordered selection: probability-priority capacity and expert-choice
// routing, plus the row gather and the expert-choice combine they feed.
//
// Priority capacity ("深入理解 MoE" §4.2.2, the capacity-bounded router: an
// over-full expert keeps its highest-probability tokens).  The pairs of each
// expert arrive in a staging list in token-major (t, s) order together with
// their unbiased router scores.  An expert with n_e > C keeps its C largest
// scores; equal scores at the cut are taken in list order, i.e. (t, s).
// Kept pairs land on rows offsets[e] + (their rank among the kept pairs in
// list order), so rows inside an expert stay in (t, s) order.
//
// Expert choice ("深入理解 MoE" §9.2; the routing table of "MoE：条件计算与
// 路由": every expert takes its top-r tokens).  Expert e scans the column
// scores[e][0..T) and takes its r largest, equal scores to the lower token;
// row e*r + j holds its j-th chosen token in ascending order, with the score
// as the gate.
//
// Both cuts find the threshold with an MSB-first radix select over the fp32
// bit patterns of the (non-negative) scores, 8 bits per pass: a 256-bin
// shared-memory histogram of the keys that match the prefix found so far, then
// a suffix scan over the bins.  After four passes the threshold is exact and
// the number of keys strictly above it is known; one ordered pass with a
// paired block scan (keys above, keys equal) places the kept entries.
// Integer work only, deterministic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "bounds.cuh"
#include "moe_internal.h"
#include "sm100_primitives.cuh"

namespace moe {

namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;

struct SelectShared {
  int hist[256];
  int warp_tot[2][kSelWarps];
  uint32_t prefix;
  int rem;
  int gt;
};

// Exclusive scans of two ints per thread over the block, in thread order;
// totals returned through *tot_a, *tot_b.
__device__ __forceinline__ void block_scan2(int a, int b, int* ex_a, int* ex_b, int* tot_a,
                                            int* tot_b, SelectShared* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int xa = a, xb = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ya = __shfl_up_sync(0xffffffffu, xa, o);
    const int yb = __shfl_up_sync(0xffffffffu, xb, o);
    if (lane >= o) {
      xa += ya;
      xb += yb;
    }
  }
  if (lane == 31) {
    sh->warp_tot[0][warp] = xa;
    sh->warp_tot[1][warp] = xb;
  }
  __syncthreads();
  if (warp == 0) {
    int wa = lane < kSelWarps ? sh->warp_tot[0][lane] : 0;
    int wb = lane < kSelWarps ? sh->warp_tot[1][lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ya = __shfl_up_sync(0xffffffffu, wa, o);
      const int yb = __shfl_up_sync(0xffffffffu, wb, o);
      if (lane >= o) {
        wa += ya;
        wb += yb;
      }
    }
    if (lane < kSelWarps) {
      sh->warp_tot[0][lane] = wa;
      sh->warp_tot[1][lane] = wb;
    }
  }
  __syncthreads();
  *ex_a = (warp > 0 ? sh->warp_tot[0][warp - 1] : 0) + xa - a;
  *ex_b = (warp > 0 ? sh->warp_tot[1][warp - 1] : 0) + xb - b;
  *tot_a = sh->warp_tot[0][kSelWarps - 1];
  *tot_b = sh->warp_tot[1][kSelWarps - 1];
  __syncthreads();
}

// The want-th largest (1 <= want <= n) of the n keys key_at(0..n): returns the
// key and, through *n_gt, how many keys are strictly larger.
template <typename KeyAt>
__device__ uint32_t radix_select_desc(int n, int want, KeyAt key_at, int* n_gt,
                                      SelectShared* sh) {
  uint32_t prefix = 0, mask = 0;
  int rem = want, gt = 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < 256; b += blockDim.x) sh->hist[b] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const uint32_t key = key_at(i);
      if ((key & mask) == prefix) atomicAdd(&sh->hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins [8l, 8l + 8); suffix sums over higher lanes
      int cnt[8];
      int own = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cnt[j] = sh->hist[8 * lane + j];
        own += cnt[j];
      }
      int incl = own;  // sum over lanes >= lane
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += y;
      }
      int above = incl - own;  // keys in bins owned by higher lanes
      // the crossing bin: the highest b with (keys in bins > b) < rem <= (keys in bins >= b)
      if (above < rem && above + own >= rem) {
        int acc = above;
        for (int j = 7; j >= 0; --j) {
          if (acc + cnt[j] >= rem) {
            sh->prefix = prefix | (static_cast<uint32_t>(8 * lane + j) << shift);
            sh->rem = rem - acc;
            sh->gt = gt + acc;
            break;
          }
          acc += cnt[j];
        }
      }
    }
    __syncthreads();
    prefix = sh->prefix;
    rem = sh->rem;
    gt = sh->gt;
    mask |= 255u << shift;
    __syncthreads();
  }
  *n_gt = gt;
  return prefix;
}

// ---------------------------------------------------------------------------
// Probability-priority capacity: one CTA per expert over its staging segment.
__global__ void __launch_bounds__(kSelThreads) priority_select_kernel(const PrioritySelectArgs a) {
  __shared__ SelectShared sh;
  const int e = blockIdx.x;
  const int base = a.all_offsets[e];
  const int n = a.all_offsets[e + 1] - base;
  const int out0 = a.offsets[e];
  const int32_t* list = a.stage_q + base;
  const float* keys = a.stage_key + base;
  const int k = a.k;
  const bool cut = a.C >= 0 && n > a.C;
  uint32_t thr = 0u;
  int n_gt = 0, ties = 0;
  if (cut) {
    thr = radix_select_desc(
        n, static_cast<int>(a.C), [&](int i) { return __float_as_uint(__ldg(keys + i)); }, &n_gt,
        &sh);
    ties = static_cast<int>(a.C) - n_gt;
  }
  // kept: every key above the threshold, and the first `ties` keys equal to
  // it; a kept entry's position = kept-above before it + min(equal before, ties)
  int carry_gt = 0, carry_eq = 0;
  for (int c0 = 0; c0 < n; c0 += kSelThreads) {
    const int i = c0 + threadIdx.x;
    const bool in = i < n;
    const uint32_t key = in ? __float_as_uint(__ldg(keys + i)) : 0u;
    const int gt = (in && (!cut || key > thr)) ? 1 : 0;
    const int eq = (in && cut && key == thr) ? 1 : 0;
    int ex_gt, ex_eq, tot_gt, tot_eq;
    block_scan2(gt, eq, &ex_gt, &ex_eq, &tot_gt, &tot_eq, &sh);
    const int eq_before = carry_eq + ex_eq;
    const bool keep = gt || (eq && eq_before < ties);
    if (in) {
      const int q = __ldg(list + i);
      if (!idx_ok(q, a.n_pairs, a.status)) {
        // a staged pair number outside [0, T k): nothing to place
      } else if (keep) {
        const int row = out0 + carry_gt + ex_gt + min(eq_before, ties);
        a.slot_row[q] = row;
        if (a.drop_mask) a.drop_mask[q] = 0;
        if (idx_ok(row, a.rmax, a.status)) {
          a.row_token[row] = q / k;
          if (a.row_gate) a.row_gate[row] = a.gates[q];
        }
      } else {
        a.slot_row[q] = -1;
        if (a.drop_mask) a.drop_mask[q] = 1;
      }
    }
    carry_gt += tot_gt;
    carry_eq += tot_eq;
  }
}

// ---------------------------------------------------------------------------
// Expert choice: one CTA per expert over its score column.
__global__ void __launch_bounds__(kSelThreads) ec_select_kernel(const EcSelectArgs a) {
  __shared__ SelectShared sh;
  const int e = blockIdx.x;
  const int T = a.T;
  const int r = a.r;
  const float* col = a.scores_t + static_cast<int64_t>(e) * T;
  int32_t* sel = a.sel_t + static_cast<int64_t>(e) * T;
  const bool cut = r < T;
  uint32_t thr = 0u;
  int n_gt = 0, ties = 0;
  if (cut && r > 0) {
    thr = radix_select_desc(
        T, r, [&](int i) { return __float_as_uint(__ldg(col + i)); }, &n_gt, &sh);
    ties = r - n_gt;
  }
  int carry_gt = 0, carry_eq = 0;
  const int64_t row0 = static_cast<int64_t>(e) * r;
  for (int c0 = 0; c0 < T; c0 += kSelThreads) {
    const int t = c0 + threadIdx.x;
    const bool in = t < T;
    const float s = in ? __ldg(col + t) : 0.0f;
    const uint32_t key = __float_as_uint(s);
    const int gt = (in && r > 0 && (!cut || key > thr)) ? 1 : 0;
    const int eq = (in && r > 0 && cut && key == thr) ? 1 : 0;
    int ex_gt, ex_eq, tot_gt, tot_eq;
    block_scan2(gt, eq, &ex_gt, &ex_eq, &tot_gt, &tot_eq, &sh);
    const int eq_before = carry_eq + ex_eq;
    const bool keep = gt || (eq && eq_before < ties);
    if (in) {
      if (keep) {
        const int64_t row = row0 + carry_gt + ex_gt + min(eq_before, ties);
        sel[t] = static_cast<int32_t>(row);
        a.row_token[row] = t;
        a.row_gate[row] = s;
      } else {
        sel[t] = -1;
      }
    }
    carry_gt += tot_gt;
    carry_eq += tot_eq;
  }
}

// ---------------------------------------------------------------------------
// x_perm[row] = x[row_token[row]] for row < offsets[E]; one warp per row.
constexpr int kGatherWarps = 8;
constexpr int kGatherU = 4;

__global__ void __launch_bounds__(kGatherWarps * 32)
    gather_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ row_token,
                       const int32_t* __restrict__ offsets, int32_t E, int32_t d,
                       uint16_t* __restrict__ x_perm, int64_t max_rows, int64_t x_rows,
                       int* status) {
  int R = __ldg(offsets + E);
  if (kBoundsChecked && R > max_rows) {
    idx_ok(R - 1, max_rows, status);  // records the overflow
    R = static_cast<int>(max_rows);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = d / 8;
  for (int row = blockIdx.x * kGatherWarps + warp; row < R; row += gridDim.x * kGatherWarps) {
    const int t = __ldg(row_token + row);
    if (!idx_ok(t, x_rows, status)) continue;
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * d);
    uint4* dst = reinterpret_cast<uint4*>(x_perm + static_cast<int64_t>(row) * d);
    for (int v0 = lane; v0 < nvec; v0 += 32 * kGatherU) {
      uint4 val[kGatherU];
#pragma unroll
      for (int u = 0; u < kGatherU; ++u)
        if (v0 + 32 * u < nvec) val[u] = __ldg(src + v0 + 32 * u);
#pragma unroll
      for (int u = 0; u < kGatherU; ++u)
        if (v0 + 32 * u < nvec) dst[v0 + 32 * u] = val[u];
    }
  }
}

// ---------------------------------------------------------------------------
// Expert-choice combine: y[t] = sum over experts e that picked t (e ascending)
// of gate * y_perm[row] + y_shared[t]; fp32 accumulation, bf16 store.  One
// warp per token; the warp first lists (row, gate) of its token's experts.
constexpr int kEcCombineWarps = 8;

__device__ __forceinline__ void fma_bf16x8(float (&acc)[8], const uint4 v, float g) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    acc[2 * i] = fmaf(g, f.x, acc[2 * i]);
    acc[2 * i + 1] = fmaf(g, f.y, acc[2 * i + 1]);
  }
}

// kU vectors of the row per lane and kR rows at a time: kU * kR 16-byte loads
// in flight before the first FMA.  Tokens with few rows (about E r / T) take
// kU = 4, kR = 2, so that the vectors supply the parallelism; tokens with
// many rows take kU = 1, kR = 8 (fewer registers, more resident warps).  Rows
// are accumulated in ascending expert order either way.
template <int kU, int kR>
__global__ void __launch_bounds__(kEcCombineWarps * 32)
    ec_combine_kernel(int32_t T, int32_t d, int32_t E, const int32_t* __restrict__ sel_t,
                      const float* __restrict__ row_gate, const uint16_t* __restrict__ y_perm,
                      const uint16_t* __restrict__ y_shared, uint16_t* __restrict__ y,
                      int64_t rmax, int* status) {
  __shared__ int lrow[kEcCombineWarps][256];
  __shared__ float lgate[kEcCombineWarps][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kEcCombineWarps + warp;
  if (t >= T) return;
  int n = 0;
  for (int e0 = 0; e0 < E; e0 += 32) {
    const int e = e0 + lane;
    int row = e < E ? __ldg(sel_t + static_cast<int64_t>(e) * T + t) : -1;
    if (row >= 0 && !idx_ok(row, rmax, status)) row = -1;
    const unsigned m = __ballot_sync(0xffffffffu, row >= 0);
    if (row >= 0) {
      const int pos = n + __popc(m & ((1u << lane) - 1u));
      lrow[warp][pos] = row;
      lgate[warp][pos] = row_gate ? __ldg(row_gate + row) : 1.0f;  // null: applied upstream
    }
    n += __popc(m);
  }
  __syncwarp();
  const int nvec = d / 8;
  const uint4* ys =
      y_shared ? reinterpret_cast<const uint4*>(y_shared + static_cast<int64_t>(t) * d) : nullptr;
  uint4* out = reinterpret_cast<uint4*>(y + static_cast<int64_t>(t) * d);
  for (int v0 = lane; v0 < nvec; v0 += 32 * kU) {
    float acc[kU][8];
    uint4 sv[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[u][i] = 0.0f;
      sv[u] = make_uint4(0u, 0u, 0u, 0u);
      if (ys && v0 + 32 * u < nvec) sv[u] = __ldg(ys + v0 + 32 * u);
    }
    for (int j0 = 0; j0 < n; j0 += kR) {
      uint4 val[kU][kR];
#pragma unroll
      for (int rr = 0; rr < kR; ++rr) {
        if (j0 + rr >= n) continue;
        const uint4* src =
            reinterpret_cast<const uint4*>(y_perm + static_cast<int64_t>(lrow[warp][j0 + rr]) * d);
#pragma unroll
        for (int u = 0; u < kU; ++u)
          if (v0 + 32 * u < nvec) val[u][rr] = __ldg(src + v0 + 32 * u);
      }
#pragma unroll
      for (int rr = 0; rr < kR; ++rr) {  // experts in ascending order
        if (j0 + rr >= n) continue;
        const float gate = lgate[warp][j0 + rr];
#pragma unroll
        for (int u = 0; u < kU; ++u)
          if (v0 + 32 * u < nvec) fma_bf16x8(acc[u], val[u][rr], gate);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = v0 + 32 * u;
      if (v >= nvec) continue;
      if (ys) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&sv[u]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(h[i]);
          acc[u][2 * i] += f.x;
          acc[u][2 * i + 1] += f.y;
        }
      }
      out[v] = make_uint4(pack_bf16x2(acc[u][0], acc[u][1]), pack_bf16x2(acc[u][2], acc[u][3]),
                          pack_bf16x2(acc[u][4], acc[u][5]), pack_bf16x2(acc[u][6], acc[u][7]));
    }
  }
}

}  // namespace

int launch_priority_select(const PrioritySelectArgs& args, cudaStream_t stream) {
  if (args.E <= 0) return 0;
  priority_select_kernel<<<args.E, kSelThreads, 0, stream>>>(args);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_ec_select(const EcSelectArgs& args, cudaStream_t stream) {
  if (args.E <= 0 || args.T <= 0) return 0;
  ec_select_kernel<<<args.E, kSelThreads, 0, stream>>>(args);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_gather_rows(const uint16_t* x, const int32_t* row_token, const int32_t* offsets,
                       int32_t E, int32_t d, int64_t max_rows, uint16_t* x_perm, int num_sms,
                       int64_t x_rows, int* status, cudaStream_t stream) {
  if (max_rows <= 0) return 0;
  int64_t grid = (max_rows + kGatherWarps - 1) / kGatherWarps;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (grid > cap) grid = cap;
  gather_rows_kernel<<<static_cast<unsigned>(grid), kGatherWarps * 32, 0, stream>>>(
      x, row_token, offsets, E, d, x_perm, max_rows, x_rows, status);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_ec_combine(int32_t T, int32_t d, int32_t E, const int32_t* sel_t,
                      const float* row_gate, const uint16_t* y_perm, const uint16_t* y_shared,
                      uint16_t* y, int64_t rmax, int* status, cudaStream_t stream) {
  if (T == 0) return 0;
  if (E > 256) return -2;
  const int grid = (T + kEcCombineWarps - 1) / kEcCombineWarps;
  // rmax = E r rows: tokens average rmax / T of them
  if (rmax <= 3 * static_cast<int64_t>(T))
    ec_combine_kernel<4, 2><<<grid, kEcCombineWarps * 32, 0, stream>>>(
        T, d, E, sel_t, row_gate, y_perm, y_shared, y, rmax, status);
  else
    ec_combine_kernel<1, 8><<<grid, kEcCombineWarps * 32, 0, stream>>>(
        T, d, E, sel_t, row_gate, y_perm, y_shared, y, rmax, status);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace moe
