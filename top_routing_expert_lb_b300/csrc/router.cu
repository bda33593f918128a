// Fused router: logits tile GEMM on tcgen05 + per-token softmax, selection
// bias, Top-k and renormalisation.
//
// Computes, for 128 tokens per CTA ("MoE：条件计算与路由": router
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
// The logits tile is 128 x N (N = E rounded up to 16, W_r rows past E are
// zero-filled by TMA); TMEM lane i holds token i's logits, so one epilogue
// thread owns one token and reads its row in 32-column chunks.
#include <cuda.h>
#include <cuda_runtime.h>

#include "moe_internal.h"
#include "sm100_primitives.cuh"

namespace moe {

namespace {

constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kThreads = 192;

struct RouterSmemTail {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull;
  uint32_t tmem_base;
  int abort_flag;
  int hist[256];
  float off[256];
  float bias[256];
  float lse[128];
};

__host__ __device__ inline int router_n(int E) { return (E + 15) / 16 * 16; }
__host__ __device__ inline uint32_t router_tmem_cols(int N) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(N)) c <<= 1;
  return c;
}
__host__ __device__ inline size_t router_main_bytes(int E) {
  const size_t stages = static_cast<size_t>(kStages) * (128 * kBK * 2 + router_n(E) * kBK * 2);
  const size_t psm = static_cast<size_t>(128) * (E + 1) * 4;
  return stages > psm ? stages : psm;
}
inline size_t router_smem_bytes(int E) {
  return 1024 + router_main_bytes(E) + sizeof(RouterSmemTail);
}

__global__ void __launch_bounds__(kThreads, 1)
    router_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                  const RouterArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const int E = p.E, k = p.k;
  const int N = router_n(E);
  const int a_bytes = 128 * kBK * 2;
  const int stage_bytes = a_bytes + N * kBK * 2;
  RouterSmemTail* st = reinterpret_cast<RouterSmemTail*>(smem + router_main_bytes(E));
  volatile int* abort_flag = &st->abort_flag;
  const uint32_t tmem_cols = router_tmem_cols(N);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tile = blockIdx.x;
  const int nk = p.d / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
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
      uint32_t uses[kStages] = {0, 0, 0, 0};
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait_bounded(&st->empty[stage], phase ^ 1u, p.timeout_ns, p.status,
                               abort_flag))
          break;
        uint8_t* sa = smem + stage * stage_bytes;
        mbar_arrive_expect_tx(&st->full[stage], static_cast<uint32_t>(stage_bytes));
        tma_load_2d(sa, &tmX, &st->full[stage], kb * kBK, tile * 128);
        tma_load_2d(sa + a_bytes, &tmW, &st->full[stage], kb * kBK, 0);
        uses[stage] += 1;
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      for (int s = 0; s < kStages; ++s)
        if (uses[s] > 0)
          mbar_wait_bounded(&st->full[s], (uses[s] - 1u) & 1u, p.timeout_ns, p.status, nullptr);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, static_cast<uint32_t>(N));
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait_bounded(&st->full[stage], phase, p.timeout_ns, p.status, abort_flag))
          break;
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + stage * stage_bytes);
        const uint32_t sb = sa + a_bytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          tc_mma_bf16(tmem_base, smem_desc_sw128(sa + kk * 32), smem_desc_sw128(sb + kk * 32),
                      idesc, (kb | kk) != 0 ? 1u : 0u);
        tc_commit(&st->empty[stage]);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      tc_commit(&st->tfull);
      // every issued MMA must retire before TMEM is freed (also on abort)
      mbar_wait_bounded(&st->tfull, 0, p.timeout_ns, p.status, nullptr);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int t = tile * 128 + r;
    const bool valid = t < p.T;
    float* p_smem = reinterpret_cast<float*>(smem);  // [128][E+1], reuses the stage ring
    const bool ok = mbar_wait_bounded(&st->tfull, 0, p.timeout_ns, p.status, abort_flag);
    tc_fence_after();
    if (ok && !*abort_flag) {
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
      const int nchunks = (E + 31) / 32;
      float m = -INFINITY;
      for (int c = 0; c < nchunks; ++c) {
        float v[32];
        tmem_ld32(taddr + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = c * 32 + i;
          if (e < E) m = fmaxf(m, v[i] + st->off[e]);
        }
      }
      float s = 0.0f;
      for (int c = 0; c < nchunks; ++c) {
        float v[32];
        tmem_ld32(taddr + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = c * 32 + i;
          if (e < E) s += expf(v[i] + st->off[e] - m);
        }
      }
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
      for (int c = 0; c < nchunks; ++c) {
        float v[32];
        tmem_ld32(taddr + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = c * 32 + i;
          if (e < E) {
            const float pe = expf(v[i] + st->off[e] - m) * inv_s;
            p_smem[r * (E + 1) + e] = valid ? pe : 0.0f;
            const float key = pe + st->bias[e];
            // Insertion into the descending list.  Experts arrive in index
            // order, so a new key goes after every equal key already listed
            // (strict '>'); entries below the insertion point shift down.
            if (k > 0 && key > thresh) {
              float ck = key, cp = pe;
              int ci = e;
              bool placed = false;
#pragma unroll
              for (int j = 0; j < kMaxTopK; ++j) {
                if (j < k && (placed || ck > top_key[j])) {
                  const float tk = top_key[j], tp = top_p[j];
                  const int tid = top_id[j];
                  top_key[j] = ck;
                  top_p[j] = cp;
                  top_id[j] = ci;
                  ck = tk;
                  cp = tp;
                  ci = tid;
                  placed = true;
                }
              }
#pragma unroll
              for (int j = 0; j < kMaxTopK; ++j)
                if (j == k - 1) thresh = top_key[j];
            }
          }
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
    }
    tc_fence_before();
    // the 128 epilogue threads meet, then reduce the tile partials
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (ok && !*abort_flag) {
      const int et = threadIdx.x - 64;
      const int rows_valid = min(128, p.T - tile * 128);
      for (int e = et; e < E; e += 128) {
        float acc = 0.0f;
        for (int rr = 0; rr < rows_valid; ++rr) acc += p_smem[rr * (E + 1) + e];
        p.tile_psum[static_cast<int64_t>(tile) * E + e] = acc;
        p.tile_hist[static_cast<int64_t>(tile) * E + e] = st->hist[e];
      }
      if (et == 0) {
        float z = 0.0f;
        for (int rr = 0; rr < rows_valid; ++rr) z += st->lse[rr] * st->lse[rr];
        p.tile_lse2[tile] = z;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, tmem_cols);
}

}  // namespace

int launch_router(const CUtensorMap& x_map, const CUtensorMap& wr_map, const RouterArgs& args,
                  cudaStream_t stream) {
  const int ntiles = (args.T + 127) / 128;
  if (ntiles == 0) return 0;
  const size_t smem = router_smem_bytes(args.E);
  if (smem > 227 * 1024) return -2;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             227 * 1024) != cudaSuccess)
      return -3;
    attr = true;
  }
  router_kernel<<<ntiles, kThreads, smem, stream>>>(x_map, wr_map, args);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace moe
