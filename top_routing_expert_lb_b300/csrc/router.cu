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
// §2.2).  Every reduction runs in a fixed order, so results are bitwise
// reproducible for a given shape.
//
// Layout of the work.  The logits tile is 128 x N (N = E rounded up to 16;
// W_r rows past E are zero-filled by TMA) in TMEM, lane i = token i.  When
// there are few tiles, the S CTAs of a thread-block cluster split the d (K)
// dimension of one tile.  After the main loop every CTA copies its partial
// logits to shared memory; CTA q of the cluster owns rows [q*128/S,
// (q+1)*128/S) and receives the peers' partials for them over distributed
// shared memory (a reduce-scatter), sums them in rank order and runs the
// softmax / Top-k epilogue for its rows with 8 warps: 2S threads per token,
// each over a strided subset of the experts, combined by xor butterflies
// (max, sum) and a merge of per-thread Top-k lists under the total order
// (key descending, expert index ascending).  Per-CTA column sums, histograms
// and lse^2 sums go to the cluster's rank-0 CTA, which adds them in rank order.
// Optional outputs: the unbiased score of every selected pair (priority
// capacity) and the whole score matrix, expert-major (expert-choice routing,
// launched with k = 0).
#include <cuda.h>
#include <cuda_runtime.h>

#include "moe_internal.h"
#include "sm100_primitives.cuh"

namespace moe {

namespace {

constexpr int kBK = 64;
constexpr int kMaxStages = 8;
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = 64 + kEpiThreads;  // producer, MMA, 8 epilogue warps
constexpr int kMaxSplit = 8;

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
  // per-CTA contributions to the tile partials, one slot per cluster rank
  // (the per-expert slots follow the struct: router_slots, S x 256 each)
  float slot_lse2[kMaxSplit];
  float slot_ent[kMaxSplit];
  float ent[128];
};

// Per-expert tile-partial slots after the tail struct, sized by the cluster
// split S (a split of 1 needs one slot, which leaves room for another ring
// stage when two CTAs share an SM): column sums, histograms, importance.
struct RouterSlots {
  float* colsum;  // [S][256]
  int* hist;      // [S][256]
  float* imp;     // [S][256]
};
__host__ __device__ inline size_t router_slot_bytes(int S) {
  return static_cast<size_t>(S) * 256 * 3 * 4;
}
__device__ inline RouterSlots router_slots(RouterSmemTail* st, int S) {
  RouterSlots r;
  r.colsum = reinterpret_cast<float*>(st + 1);
  r.hist = reinterpret_cast<int*>(r.colsum + S * 256);
  r.imp = reinterpret_cast<float*>(r.hist + S * 256);
  return r;
}

struct RouterGeom {
  int N;             // MMA N (E rounded up to 16)
  int stages;        // pipeline depth
  int stage_bytes;   // A tile + B tile
  int ldl;           // row pitch of a logits row (floats)
  int rpc;           // rows owned per CTA (128 / S)
  size_t main_bytes;  // stage ring, reused afterwards for the logits tiles
};

__host__ __device__ inline RouterGeom router_geom(int E, int stages, int S) {
  RouterGeom g;
  g.N = (E + 15) / 16 * 16;
  g.stages = stages;
  g.stage_bytes = 128 * kBK * 2 + g.N * kBK * 2;
  // Row pitch = 2S (mod 32) floats: the 2S threads that share a row in the
  // epilogue read consecutive experts, so one warp's 32 lanes hit 32 banks.
  g.ldl = E + (((2 * S - E) % 32) + 32) % 32;
  g.rpc = 128 / S;
  const size_t ring = static_cast<size_t>(stages) * g.stage_bytes;
  // own partial [128][ldl] + receive slots [S][rpc][ldl] (= another 128 rows)
  const size_t tiles = static_cast<size_t>(S > 1 ? 256 : 128) * g.ldl * 4;
  g.main_bytes = ring > tiles ? ring : tiles;
  return g;
}

__host__ __device__ inline uint32_t router_tmem_cols(int N) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(N)) c <<= 1;
  return c;
}

__device__ __forceinline__ void st_dsmem_f32(uint32_t remote_addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote_addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_dsmem_s32(uint32_t remote_addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(remote_addr), "r"(v) : "memory");
}

// (key desc, index asc): true when (ka, ia) comes before (kb, ib).
__device__ __forceinline__ bool before(float ka, int ia, float kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

template <int K>
__global__ void __launch_bounds__(kThreads, 1)
    router_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                  const RouterArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const int E = p.E;
  const int S = p.split;
  const RouterGeom geo = router_geom(E, p.stages, S);
  const int a_bytes = 128 * kBK * 2;
  RouterSmemTail* st = reinterpret_cast<RouterSmemTail*>(smem + geo.main_bytes);
  const RouterSlots slots = router_slots(st, S);
  volatile int* abort_flag = &st->abort_flag;
  const uint32_t tmem_cols = router_tmem_cols(geo.N);
  const int ldl = geo.ldl;
  const int rpc = geo.rpc;
  float* lg = reinterpret_cast<float*>(smem);          // own partial [128][ldl]
  float* recv = lg + static_cast<size_t>(128) * ldl;   // [S][rpc][ldl], slot q from rank q

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = S > 1 ? cluster_ctarank() : 0u;
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
  } else if (warp < 6) {
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

  // Partial logits of every CTA are in its shared memory and every MMA of the
  // cluster has retired.  Reduce-scatter: rows owned by CTA q go to slot
  // [this rank] of q's receive area.
  __syncthreads();
  const int eidx = static_cast<int>(threadIdx.x) - 64;  // epilogue thread index, or < 0
  if (S > 1) {
    cluster_arrive_wait();
    if (eidx >= 0 && !*abort_flag) {
      const int per = rpc * E;  // values per destination
      for (int q = 0; q < S; ++q) {
        if (q == static_cast<int>(rank)) continue;
        const uint32_t dst =
            mapa_shared(smem_u32(recv + static_cast<size_t>(rank) * rpc * ldl), q);
        for (int i = eidx; i < per; i += kEpiThreads) {
          const int rl = i / E, e = i - rl * E;
          st_dsmem_f32(dst + 4u * (rl * ldl + e), lg[(q * rpc + rl) * ldl + e]);
        }
      }
    }
    cluster_arrive_wait();
  }

  const int tpr = kEpiThreads / rpc;  // threads per token row (2S)
  if (eidx >= 0 && !*abort_flag) {
    // -------------------------------------------- epilogue, part 2 (owned rows)
    const int rl = eidx / tpr;        // local row
    const int sub = eidx - rl * tpr;  // this thread's expert subset: e = sub (mod tpr)
    const int r = static_cast<int>(rank) * rpc + rl;
    const int t = tile * 128 + r;
    const bool valid = t < p.T;
    float* row = lg + r * ldl;  // receives the full logits, then exp, then the scores
    const bool sigmoid = (p.flags & kRouteSigmoid) != 0;
    // The three passes over the row below handle four experts per step:
    // their loads and arithmetic overlap, while every sum and the Top-k
    // insertion still take the experts in ascending order (same results as
    // one expert at a time).
    float m = -INFINITY;
    auto full_logit = [&](int e) {
      float v = 0.0f;
      for (int q = 0; q < S; ++q)  // partials in rank order
        v += (q == static_cast<int>(rank))
                 ? row[e]
                 : recv[(static_cast<size_t>(q) * rpc + rl) * ldl + e];
      return v + st->off[e];
    };
    int e = sub;
    for (; e + 3 * tpr < E; e += 4 * tpr) {
      float v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = full_logit(e + u * tpr);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        row[e + u * tpr] = v[u];
        m = fmaxf(m, v[u]);
      }
    }
    for (; e < E; e += tpr) {
      const float v = full_logit(e);
      row[e] = v;
      m = fmaxf(m, v);
    }
    for (int o = 1; o < tpr; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    // softmax normaliser (also the z-loss's lse); with sigmoid scores the row
    // keeps the logits for the next pass
    float s = 0.0f, hs = 0.0f;  // hs: sum of ex * (l - m), for the entropy
    for (e = sub; e + 3 * tpr < E; e += 4 * tpr) {
      float v[4], ex[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        v[u] = row[e + u * tpr];
        ex[u] = __expf(v[u] - m);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (!sigmoid) row[e + u * tpr] = ex[u];
        s += ex[u];
        hs += ex[u] * (v[u] - m);
      }
    }
    for (; e < E; e += tpr) {
      const float v = row[e];
      const float ex = __expf(v - m);
      if (!sigmoid) row[e] = ex;
      s += ex;
      hs += ex * (v - m);
    }
    for (int o = 1; o < tpr; o <<= 1) {
      s += __shfl_xor_sync(0xffffffffu, s, o);
      hs += __shfl_xor_sync(0xffffffffu, hs, o);
    }
    const float inv_s = 1.0f / s;
    float top_key[K > 0 ? K : 1];
    int top_id[K > 0 ? K : 1];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      top_key[j] = -INFINITY;
      top_id[j] = 0x7fffffff;
    }
    float thresh = -INFINITY;  // K-th largest key of this thread so far
    float ssum = 0.0f, slog = 0.0f;  // sigmoid: sum s, sum s log s (entropy)
    // score of expert e (and its sigmoid entropy term), independent per expert
    auto score = [&](int e, float* term) {
      if (sigmoid) {
        const float en = __expf(-row[e]);
        const float pe = 1.0f / (1.0f + en);
        *term = pe > 0.0f ? pe * log1pf(en) : 0.0f;  // s log s = -s log(1 + e^-l)
        return pe;
      }
      *term = 0.0f;
      return row[e] * inv_s;
    };
    // in ascending expert order: the sums, the row's score and the Top-k list
    auto commit = [&](int e, float pe, float term) {
      if (sigmoid) {
        ssum += pe;
        if (pe > 0.0f) slog -= term;
      }
      row[e] = valid ? pe : 0.0f;  // the row now holds the scores (gates, P partial)
      const float key = pe + st->bias[e];
      // experts arrive in index order: strict '>' keeps equal keys in index order
      if (K > 0 && key > thresh) {
        float ck = key;
        int ci = e;
        bool placed = false;
#pragma unroll
        for (int j = 0; j < K; ++j) {
          if (placed || ck > top_key[j]) {
            const float tk = top_key[j];
            const int ti = top_id[j];
            top_key[j] = ck;
            top_id[j] = ci;
            ck = tk;
            ci = ti;
            placed = true;
          }
        }
        thresh = top_key[K > 0 ? K - 1 : 0];
      }
    };
    for (e = sub; e + 3 * tpr < E; e += 4 * tpr) {
      float pe[4], term[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) pe[u] = score(e + u * tpr, &term[u]);
#pragma unroll
      for (int u = 0; u < 4; ++u) commit(e + u * tpr, pe[u], term[u]);
    }
    for (; e < E; e += tpr) {
      float term;
      const float pe = score(e, &term);
      commit(e, pe, term);
    }
    if (sigmoid) {
      for (int o = 1; o < tpr; o <<= 1) {
        ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
        slog += __shfl_xor_sync(0xffffffffu, slog, o);
      }
    }
    __syncwarp();  // the row's p values (written by the whole group) are visible
    // merge the group's lists: each level inserts the partner's K entries
    for (int o = 1; o < tpr; o <<= 1) {
      float pk[K > 0 ? K : 1];
      int pi[K > 0 ? K : 1];
#pragma unroll
      for (int j = 0; j < K; ++j) {
        pk[j] = __shfl_xor_sync(0xffffffffu, top_key[j], o);
        pi[j] = __shfl_xor_sync(0xffffffffu, top_id[j], o);
      }
#pragma unroll
      for (int i = 0; i < K; ++i) {
        float ck = pk[i];
        int ci = pi[i];
        bool placed = false;
#pragma unroll
        for (int j = 0; j < K; ++j) {
          if (placed || before(ck, ci, top_key[j], top_id[j])) {
            const float tk = top_key[j];
            const int ti = top_id[j];
            top_key[j] = ck;
            top_id[j] = ci;
            ck = tk;
            ci = ti;
            placed = true;
          }
        }
      }
    }
    // entropy of the router distribution: softmax log s - sum ex (l-m) / s;
    // sigmoid q = s / sum s: log sum s - sum s log s / sum s
    const float ent = sigmoid ? (logf(ssum) - slog / ssum) : (logf(s) - hs * inv_s);
    const bool renorm = (p.flags & kRouteNoRenorm) == 0;
    if (sub == 0) {
      st->lse[rl] = valid ? (m + logf(s)) : 0.0f;
      st->ent[rl] = valid ? ent : 0.0f;
      if (valid && K > 0) {
        float denom = 0.0f;
#pragma unroll
        for (int j = 0; j < K; ++j) denom += row[top_id[j]];
        const float inv_d = renorm ? 1.0f / denom : 1.0f;
#pragma unroll
        for (int j = 0; j < K; ++j) {
          p.ids[static_cast<int64_t>(t) * K + j] = top_id[j];
          p.gates[static_cast<int64_t>(t) * K + j] = row[top_id[j]] * inv_d;
          if (p.pair_score) p.pair_score[static_cast<int64_t>(t) * K + j] = row[top_id[j]];
          atomicAdd(&st->hist[top_id[j]], 1);
        }
      }
    }
    // this CTA's contribution to the tile partials, into slot [rank] of the
    // cluster's rank-0 CTA (fixed row order inside, rank order across)
    asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory");
    const int rows_valid =
        max(0, min(rpc, p.T - (tile * 128 + static_cast<int>(rank) * rpc)));
    const bool remote = rank != 0;
    if (p.scores_t != nullptr) {
      // every score, expert-major: consecutive threads write consecutive tokens
      const int t0 = tile * 128 + static_cast<int>(rank) * rpc;
      for (int i = eidx; i < rows_valid * E; i += kEpiThreads) {
        const int e = i / rows_valid, rr = i - e * rows_valid;
        p.scores_t[static_cast<int64_t>(e) * p.T + t0 + rr] =
            lg[(static_cast<int>(rank) * rpc + rr) * ldl + e];
      }
    }
    for (int e = eidx; e < E; e += kEpiThreads) {
      float acc = 0.0f;
      for (int rr = 0; rr < rows_valid; ++rr)
        acc += lg[(static_cast<int>(rank) * rpc + rr) * ldl + e];
      if (remote) {
        st_dsmem_f32(mapa_shared(smem_u32(&slots.colsum[rank * 256 + e]), 0), acc);
        st_dsmem_s32(mapa_shared(smem_u32(&slots.hist[rank * 256 + e]), 0), st->hist[e]);
      } else {
        slots.colsum[e] = acc;
        slots.hist[e] = st->hist[e];
      }
    }
    if (eidx == 0) {
      float z = 0.0f, h = 0.0f;
      for (int rr = 0; rr < rows_valid; ++rr) {
        z += st->lse[rr] * st->lse[rr];
        h += st->ent[rr];
      }
      if (remote) {
        st_dsmem_f32(mapa_shared(smem_u32(&st->slot_lse2[rank]), 0), z);
        st_dsmem_f32(mapa_shared(smem_u32(&st->slot_ent[rank]), 0), h);
      } else {
        st->slot_lse2[0] = z;
        st->slot_ent[0] = h;
      }
    }
    if (p.tile_imp != nullptr && K > 0) {
      // importance: each row becomes its sparse gate vector (gates on the
      // selected experts, 0 elsewhere), then the same fixed-order column sums
      asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory");
      for (int e = sub; e < E; e += tpr) row[e] = 0.0f;
      __syncwarp();
      if (sub == 0 && valid) {
#pragma unroll
        for (int j = 0; j < K; ++j)
          row[top_id[j]] = p.gates[static_cast<int64_t>(t) * K + j];
      }
      asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory");
      for (int e = eidx; e < E; e += kEpiThreads) {
        float acc = 0.0f;
        for (int rr = 0; rr < rows_valid; ++rr)
          acc += lg[(static_cast<int>(rank) * rpc + rr) * ldl + e];
        if (remote)
          st_dsmem_f32(mapa_shared(smem_u32(&slots.imp[rank * 256 + e]), 0), acc);
        else
          slots.imp[e] = acc;
      }
    }
  }
  if (S > 1)
    cluster_arrive_wait();
  else
    __syncthreads();
  if (rank == 0 && eidx >= 0 && !*abort_flag) {
    for (int e = eidx; e < E; e += kEpiThreads) {
      float acc = 0.0f;
      int h = 0;
      for (int q = 0; q < S; ++q) {
        acc += slots.colsum[q * 256 + e];
        h += slots.hist[q * 256 + e];
      }
      p.tile_psum[static_cast<int64_t>(tile) * E + e] = acc;
      p.tile_hist[static_cast<int64_t>(tile) * E + e] = h;
    }
    if (eidx == 0) {
      float z = 0.0f, h = 0.0f;
      for (int q = 0; q < S; ++q) {
        z += st->slot_lse2[q];
        h += st->slot_ent[q];
      }
      p.tile_lse2[tile] = z;
      if (p.tile_ent) p.tile_ent[tile] = h;
    }
    if (p.tile_imp != nullptr && K > 0) {
      for (int e = eidx; e < E; e += kEpiThreads) {
        float acc = 0.0f;
        for (int q = 0; q < S; ++q) acc += slots.imp[q * 256 + e];
        p.tile_imp[static_cast<int64_t>(tile) * E + e] = acc;
      }
    }
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
  // Split K over a cluster while the grid still fits one wave (one CTA per
  // SM) and each CTA keeps >= 2 k-blocks.
  int S = 1;
  while (S < kMaxSplit && ntiles * 2 * S <= num_sms && nk / (2 * S) >= 2) S *= 2;
  const size_t tail = sizeof(RouterSmemTail) + router_slot_bytes(S) + 1024;
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
  void (*kern)(const CUtensorMap, const CUtensorMap, const RouterArgs) = nullptr;
  switch (args.k) {
    case 0: kern = router_kernel<0>; break;
    case 1: kern = router_kernel<1>; break;
    case 2: kern = router_kernel<2>; break;
    case 3: kern = router_kernel<3>; break;
    case 4: kern = router_kernel<4>; break;
    case 5: kern = router_kernel<5>; break;
    case 6: kern = router_kernel<6>; break;
    case 7: kern = router_kernel<7>; break;
    case 8: kern = router_kernel<8>; break;
    default: return -2;
  }
  static bool attr[kMaxTopK + 1] = {false};
  if (!attr[args.k]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
        cudaSuccess)
      return -3;
    attr[args.k] = true;
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
  if (cudaLaunchKernelEx(&cfg, kern, x_map, wr_map, args) != cudaSuccess) return -3;
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace moe
