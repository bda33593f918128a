// Fused router: logits tile GEMM on tcgen05 + per-token softmax, selection
// bias, Top-k and renormalisation.
//
// Computes, for 128 tokens per tile ("MoE：条件计算与路由": router
// g(x) = softmax(W_r x), ALF-LB bias b_e added before Top-k, §7 Eqs.(1)-(2);
// the router bias of the CSDN note's toy gate is the optional logit offset):
//   l_e   = W_r[e] . x + o_e                     (fp32 accumulate in TMEM)
//   p_e   = exp(l_e - max l) / sum exp(l - max l) (max subtraction: "MoE"
//                                                 page, training instability)
//   S     = the k largest keys p_e + b_e, descending, ties to the lower index
//   g~    = p_S / sum p_S                         (unbiased p)
// and per-tile partials for the side outputs: expert histogram (n_e), sum of
// p_e over the tile's tokens (P_e) and sum of lse^2 (z-loss, "MOE大模型对比篇"
// §2.2).  Reductions over tokens run in a fixed order, so results are
// bitwise reproducible.
//
// Layout of the work.  The logits tile is 128 x N (N = E rounded up to 16;
// W_r rows past E are zero-filled by TMA); TMEM lane i holds token i, so one
// epilogue thread owns one token.  When there are few tiles, S CTAs of a
// thread-block cluster split the d (K) dimension of one tile: each runs its
// share of the k-blocks, copies its partial logits TMEM -> shared memory, and
// the cluster's rank-0 CTA adds the peers' partials over distributed shared
// memory in rank order (deterministic) before the softmax / Top-k passes,
// which all read the row from shared memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include "moe_internal.h"
#include "sm100_primitives.cuh"

namespace moe {

namespace {

constexpr int kBK = 64;
constexpr int kMaxStages = 8;
constexpr int kThreads = 192;

struct RouterSmemTail {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull;
  uint32_t tmem_base;
  int abort_flag;
  int hist[256];
  float off[256];
  float bias[256];
  float lse[128];
  float zw[4];
};

struct RouterGeom {
  int N;             // MMA N (E rounded up to 16)
  int stages;        // pipeline depth
  int stage_bytes;   // A tile + B tile
  int part_floats;   // one [128][E+1] logits tile, rounded up to 4 floats
  size_t main_bytes;  // stage ring, reused afterwards for S logits tiles
};

__host__ __device__ inline RouterGeom router_geom(int E, int stages, int S) {
  RouterGeom g;
  g.N = (E + 15) / 16 * 16;
  g.stages = stages;
  g.stage_bytes = 128 * kBK * 2 + g.N * kBK * 2;
  g.part_floats = (128 * (E + 1) + 3) / 4 * 4;
  const size_t ring = static_cast<size_t>(stages) * g.stage_bytes;
  // S partial tiles, then [4][E] per-warp column sums
  const size_t parts = (static_cast<size_t>(S) * g.part_floats + 4 * static_cast<size_t>(E)) * 4;
  g.main_bytes = ring > parts ? ring : parts;
  return g;
}

__host__ __device__ inline uint32_t router_tmem_cols(int N) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(N)) c <<= 1;
  return c;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_peer(uint32_t local_addr, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  return remote;
}

__device__ __forceinline__ void st_dsmem_v4(uint32_t remote_addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(remote_addr), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    router_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                  const RouterArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const int E = p.E, k = p.k;
  const int S = p.split;
  const RouterGeom geo = router_geom(E, p.stages, S);
  const int a_bytes = 128 * kBK * 2;
  RouterSmemTail* st = reinterpret_cast<RouterSmemTail*>(smem + geo.main_bytes);
  volatile int* abort_flag = &st->abort_flag;
  const uint32_t tmem_cols = router_tmem_cols(geo.N);
  float* lg = reinterpret_cast<float*>(smem);  // [128][E+1] after the main loop
  const int ldl = E + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = S > 1 ? cluster_rank() : 0u;
  const int tile = blockIdx.x / S;
  const int nk = p.d / kBK;
  const int kb0 = static_cast<int>(rank) * nk / S;
  const int kb1 = (static_cast<int>(rank) + 1) * nk / S;

  if (threadIdx.x == 0) {
    for (int s = 0; s < geo.stages; ++s) {
      mbar_init(&st->full[s], 1);
      mbar_init(&st->empty[s], 1);
    }
    mbar_init(&st->tfull, 1);
    st->abort_flag = 0;
    fence_barrier_init();
  }
  for (int e = threadIdx.x; e < 256; e += blockDim.x) {
    st->hist[e] = 0;
    st->off[e] = (e < E && p.logit_offset) ? p.logit_offset[e] : 0.0f;
    st->bias[e] = (e < E && p.sel_bias) ? p.sel_bias[e] : 0.0f;
  }
  if (warp == 1) tmem_alloc(&st->tmem_base, tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = st->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmX);
      tma_prefetch_desc(&tmW);
      uint32_t uses = 0;  // loads issued; stage = uses % stages
      for (int kb = kb0; kb < kb1; ++kb, ++uses) {
        const int stage = static_cast<int>(uses % geo.stages);
        const uint32_t phase = (uses / geo.stages) & 1u;
        if (!mbar_wait_bounded(&st->empty[stage], phase ^ 1u, p.timeout_ns, p.status,
                               abort_flag))
          break;
        uint8_t* sa = smem + stage * geo.stage_bytes;
        mbar_arrive_expect_tx(&st->full[stage], static_cast<uint32_t>(geo.stage_bytes));
        tma_load_2d(sa, &tmX, &st->full[stage], kb * kBK, tile * 128);
        tma_load_2d(sa + a_bytes, &tmW, &st->full[stage], kb * kBK, 0);
      }
      // drain: the last copy into each used stage must land before exit
      for (uint32_t s = 0; s < static_cast<uint32_t>(geo.stages) && s < uses; ++s) {
        const uint32_t n_s = (uses - 1u - s) / geo.stages + 1u;  // uses of stage s
        mbar_wait_bounded(&st->full[s], (n_s - 1u) & 1u, p.timeout_ns, p.status, nullptr);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, static_cast<uint32_t>(geo.N));
      uint32_t uses = 0;
      for (int kb = kb0; kb < kb1; ++kb, ++uses) {
        const int stage = static_cast<int>(uses % geo.stages);
        const uint32_t phase = (uses / geo.stages) & 1u;
        if (!mbar_wait_bounded(&st->full[stage], phase, p.timeout_ns, p.status, abort_flag))
          break;
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + stage * geo.stage_bytes);
        const uint32_t sb = sa + a_bytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          tc_mma_bf16(tmem_base, smem_desc_sw128(sa + kk * 32), smem_desc_sw128(sb + kk * 32),
                      idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
        tc_commit(&st->empty[stage]);
      }
      tc_commit(&st->tfull);
      // every issued MMA must retire before TMEM is freed (also on abort)
      mbar_wait_bounded(&st->tfull, 0, p.timeout_ns, p.status, nullptr);
    }
    __syncwarp();
  } else {
    // -------------------------------------------- epilogue, part 1: TMEM -> smem
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const bool ok = mbar_wait_bounded(&st->tfull, 0, p.timeout_ns, p.status, abort_flag);
    tc_fence_after();
    if (ok) {
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
      for (int c = 0; c < (E + 31) / 32; ++c) {
        float v[32];
        tmem_ld32(taddr + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c * 32 + i < E) lg[r * ldl + c * 32 + i] = v[i];
      }
    }
    tc_fence_before();
  }

  // Partial logits of every CTA are in its own shared memory and every MMA of
  // the cluster has retired (so the leader's stage ring is free).  Peers push
  // their tile into slot `rank` of the leader's ring with vector DSMEM stores;
  // the second cluster barrier makes them visible to the leader.
  __syncthreads();
  if (S > 1) {
    cluster_sync_all();
    if (rank != 0 && !*abort_flag) {
      const uint32_t dst = map_peer(smem_u32(lg + static_cast<size_t>(rank) * geo.part_floats), 0);
      const uint4* src = reinterpret_cast<const uint4*>(lg);
      for (int i = threadIdx.x; i < geo.part_floats / 4; i += blockDim.x)
        st_dsmem_v4(dst + 16u * i, src[i]);
    }
    cluster_sync_all();
  }

  if (rank == 0 && warp >= 2 && !*abort_flag) {
    // -------------------------------------------- epilogue, part 2 (leader)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int t = tile * 128 + r;
    const bool valid = t < p.T;
    float* row = lg + r * ldl;
    // full logits: partials summed in rank order, + offset
    float m = -INFINITY;
    for (int e = 0; e < E; ++e) {
      float v = row[e];
      for (int q = 1; q < S; ++q) v += row[static_cast<size_t>(q) * geo.part_floats + e];
      v += st->off[e];
      row[e] = v;
      m = fmaxf(m, v);
    }
    float s = 0.0f;
#pragma unroll 4
    for (int e = 0; e < E; ++e) s += expf(row[e] - m);
    const float inv_s = 1.0f / s;
    float top_key[kMaxTopK];
    float top_p[kMaxTopK];
    int top_id[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      top_key[j] = -INFINITY;
      top_p[j] = 0.0f;
      top_id[j] = -1;
    }
    float thresh = -INFINITY;  // k-th largest key so far
#pragma unroll 2
    for (int e = 0; e < E; ++e) {
      const float pe = expf(row[e] - m) * inv_s;
      row[e] = valid ? pe : 0.0f;  // the row now holds p (for the P partial)
      const float key = pe + st->bias[e];
      // Insertion into the descending list.  Experts arrive in index order,
      // so a new key goes after every equal key already listed (strict '>');
      // entries below the insertion point shift down.
      if (k > 0 && key > thresh) {
        float ck = key, cp = pe;
        int ci = e;
        bool placed = false;
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
          if (j < k && (placed || ck > top_key[j])) {
            const float tk = top_key[j], tp = top_p[j];
            const int ti = top_id[j];
            top_key[j] = ck;
            top_p[j] = cp;
            top_id[j] = ci;
            ck = tk;
            cp = tp;
            ci = ti;
            placed = true;
          }
        }
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j)
          if (j == k - 1) thresh = top_key[j];
      }
    }
    st->lse[r] = valid ? (m + logf(s)) : 0.0f;
    if (valid && k > 0) {
      float denom = 0.0f;
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j)
        if (j < k) denom += top_p[j];
      const float inv_d = 1.0f / denom;
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {
        if (j < k) {
          p.ids[static_cast<int64_t>(t) * k + j] = top_id[j];
          p.gates[static_cast<int64_t>(t) * k + j] = top_p[j] * inv_d;
          atomicAdd(&st->hist[top_id[j]], 1);
        }
      }
    }
    // the 128 epilogue threads meet, then reduce the tile partials in a fixed
    // order: warp w sums rows 32w..32w+31 per expert, then the four warp sums
    asm volatile("bar.sync 1, 128;" ::: "memory");
    const int rows_valid = min(128, p.T - tile * 128);
    float* wsum = lg + static_cast<size_t>(S) * geo.part_floats;  // [4][E] (after the parts)
    for (int e = lane; e < E; e += 32) {
      float acc = 0.0f;
      const int r1 = min(rows_valid, quarter * 32 + 32);
      for (int rr = quarter * 32; rr < r1; ++rr) acc += lg[rr * ldl + e];
      wsum[quarter * E + e] = acc;
    }
    float z = st->lse[r] * st->lse[r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane == 0) st->zw[quarter] = z;
    asm volatile("bar.sync 1, 128;" ::: "memory");
    const int et = threadIdx.x - 64;
    for (int e = et; e < E; e += 128) {
      p.tile_psum[static_cast<int64_t>(tile) * E + e] =
          ((wsum[e] + wsum[E + e]) + wsum[2 * E + e]) + wsum[3 * E + e];
      p.tile_hist[static_cast<int64_t>(tile) * E + e] = st->hist[e];
    }
    if (et == 0) p.tile_lse2[tile] = ((st->zw[0] + st->zw[1]) + st->zw[2]) + st->zw[3];
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, tmem_cols);
}

}  // namespace

int launch_router(const CUtensorMap& x_map, const CUtensorMap& wr_map, RouterArgs args,
                  int num_sms, cudaStream_t stream) {
  const int ntiles = (args.T + 127) / 128;
  if (ntiles == 0) return 0;
  const int nk = args.d / kBK;
  const size_t tail = sizeof(RouterSmemTail) + 1024;
  // Split K over a cluster while the grid still fits one wave (one CTA per
  // SM), each CTA keeps >= 2 k-blocks and the S partial tiles fit the ring.
  int S = 1;
  while (S < 8 && ntiles * 2 * S <= num_sms && nk / (2 * S) >= 2 &&
         router_geom(args.E, 1, 2 * S).main_bytes + tail <= 200 * 1024)
    S *= 2;
  const int nk_local = (nk + S - 1) / S;
  const int stage_bytes = router_geom(args.E, 1, S).stage_bytes;
  // With more tiles than SMs, size shared memory for two CTAs per SM.
  const size_t budget = (ntiles * S > num_sms) ? 110 * 1024 : 200 * 1024;
  int stages = static_cast<int>((budget - tail) / stage_bytes);
  stages = stages > kMaxStages ? kMaxStages : stages;
  stages = stages > nk_local ? nk_local : stages;
  stages = stages < 1 ? 1 : stages;
  args.split = S;
  args.stages = stages;
  const RouterGeom geo = router_geom(args.E, stages, S);
  const size_t smem = tail + geo.main_bytes;
  if (smem > 227 * 1024) return -2;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             227 * 1024) != cudaSuccess)
      return -3;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ntiles * S);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = S;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, router_kernel, x_map, wr_map, args) != cudaSuccess) return -3;
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace moe
