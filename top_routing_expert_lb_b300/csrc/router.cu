// Fused router: logits GEMM on tcgen05 + per-token softmax, selection bias,
// Top-k and renormalisation, plus the reduction of the side outputs.
//
// Computes, for every token ("MoE：条件计算与路由": router g(x) = softmax(W_r x),
// ALF-LB bias b_e added before Top-k, §7 Eqs.(1)-(2); the router bias of the
// CSDN note's toy gate is the optional logit offset):
//   l_e   = W_r[e] . x + o_e                      (fp32 accumulate in TMEM)
//   p_e   = exp(l_e - max l) / sum exp(l - max l)  (max subtraction: "MoE"
//                                                  page, training instability)
//   S     = the k largest keys p_e + b_e, descending, ties to the lower index
//   g~    = p_S / sum p_S                          (unbiased p)
// and the side outputs: n_e, f_e = n_e / (k T), P_e = (1/T) sum_t p_e(t),
// L_bal = lambda E sum f_e P_e, L_z = (1/T) sum_t lse_t^2 ("MOE大模型对比篇"
// §2.1-§2.2), optionally the importance and its CV^2 (CSDN note) and the mean
// router entropy ("MoE：条件计算与路由" §9), and for the layer the offsets of the
// kept rows and the per-chunk bases of the permutation.
//
// Work layout.  Units are (tile of 128 tokens, K slice): with few tiles the
// d dimension of each tile is split into S slices so that every SM streams.
// A persistent grid (one CTA per SM) takes units round-robin; per CTA a TMA
// warp fills a ring of (x, W_r) stages, an MMA warp accumulates each unit into
// one of two TMEM buffers, and sixteen epilogue warps drain the other buffer
// (handing it back right after their last TMEM read), so a unit's epilogue
// overlaps the next unit's loads.  A K-split unit stores its
// partial logits to the workspace (coalesced, [expert][row] per tile); the
// CTA that stores a tile's last slice sums the S partials in slice order,
// writes the sums back into its TMEM buffer and runs the tile's epilogue.
//
// The epilogue reads the logits straight from TMEM.  Sixteen warps share a
// tile: thread (row r, part c) owns the 16-column groups c, c+4, c+8, ... of
// row r.  Two passes over the groups: an online max and sum of exponentials
// (rescaled whenever a group raises the running max), then the scores, the
// keys and a per-thread Top-k list; the four parts of a row combine max, sum
// and lists through shared memory in part order.  Column sums over the
// tile's rows (P, importance) are reduced inside each warp by a fixed shuffle
// tree and then over the four row quarters in order.  Every cross-tile total
// is either a 64-bit integer atomic on fixed-point values (P and importance at 2^-32,
// entropy at 2^-32, counts exact) or a per-tile value summed in tile order
// (lse^2), so all results are bitwise reproducible whichever CTA runs which
// tile.  The CTA that completes the last tile reduces the totals (f, P, both
// losses, importance, entropy), scans the kept counts into row offsets and
// the per-chunk expert counts into chunk bases, and puts every accumulator
// back to zero for the next call.
#include <cuda.h>
#include <cuda_runtime.h>

#include "moe_internal.h"
#include "sm100_primitives.cuh"

namespace moe {

namespace {

constexpr int kBK = 64;
constexpr int kMaxStages = 8;
constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = 64 + kEpiThreads;  // TMA warp, MMA warp, 16 epilogue warps
constexpr int kParts = kEpiWarps / 4;       // threads per row (TMEM lane quarters x parts)
constexpr int kMaxSplit = 8;
constexpr float kFix = 4294967296.0f;       // 2^32: fixed-point scale of P, importance, entropy
constexpr int kBarEpi = 1;                  // named barrier of the epilogue warps

struct RouterSmem {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t fin;
  uint32_t tmem_base;
  int abort_flag;
  int flag;                 // broadcast of a last-arrival decision
  int go;                   // broadcast: the unit's accumulator is ready (0: stop)
  int hist[256];            // this tile's expert counts
  alignas(16) float off[256];
  alignas(16) float bias[256];
  float xm[kParts][128];    // per-part running row max
  float xs[kParts][128];    // per-part sum of exponentials relative to it
  float xh[kParts][128];    // per-part sum ex (l - m) (softmax entropy)
  float xq[kParts][128];    // sigmoid: per-part sum s
  float xg[kParts][128];    // sigmoid: per-part sum s log s
  // the Top-k lists of parts 1..3 per row (score and id; the key is
  // recomputed as score + bias); after the merge by the row's part-0 thread,
  // list 0 holds the merged selection (ids, gates)
  float tk_p[kParts - 1][kMaxTopK][128];
  int tk_id[kParts - 1][kMaxTopK][128];
  float rowv[2][128];       // per-row lse^2 and entropy, for the tile sums
  float colsum[4][256];     // [row quarter][expert]: column sums over 32 rows
  float fred[kEpiWarps];    // finalize: per-warp sums
  float fred2[kEpiWarps];
  int wtot[kEpiWarps];
};

struct RouterGeom {
  int N;             // MMA N (E rounded up to 16)
  int stages;        // pipeline depth
  int stage_bytes;   // A tile + B tile
  uint32_t buf_cols;  // TMEM columns per accumulator buffer (power of two >= N)
};

__host__ __device__ inline RouterGeom router_geom(int E, int stages) {
  RouterGeom g;
  g.N = (E + 15) / 16 * 16;
  g.stages = stages;
  g.stage_bytes = 128 * kBK * 2 + g.N * kBK * 2;
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(g.N)) c <<= 1;
  g.buf_cols = c;
  return g;
}

// (key desc, index asc): true when (ka, ia) comes before (kb, ib).
__device__ __forceinline__ bool before(float ka, int ia, float kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

// Inserts (key, id, p) into the descending list (tk, ti, tp) of K entries
// under the order of before(); the last entry falls off.
template <int K>
__device__ __forceinline__ void topk_insert(float (&tk)[K > 0 ? K : 1], int (&ti)[K > 0 ? K : 1],
                                            float (&tp)[K > 0 ? K : 1], float key, int id,
                                            float pv) {
  bool placed = false;
#pragma unroll
  for (int i = 0; i < K; ++i) {
    if (placed || before(key, id, tk[i], ti[i])) {
      const float k0 = tk[i], p0 = tp[i];
      const int i0 = ti[i];
      tk[i] = key;
      ti[i] = id;
      tp[i] = pv;
      key = k0;
      id = i0;
      pv = p0;
      placed = true;
    }
  }
}

// Inserts (key, id, p) into the descending list (tk, ti, tp), the last entry
// falling off, for a scan in ascending id order: the caller has checked that
// key beats the last entry, and an equal key never moves above an entry
// already listed (it has a higher id).  Every slot is updated from the old
// values of its own slot and the one above, without a dependency chain.
template <int K>
__device__ __forceinline__ void topk_push_ascending(float (&tk)[K > 0 ? K : 1],
                                                    int (&ti)[K > 0 ? K : 1],
                                                    float (&tp)[K > 0 ? K : 1], float key,
                                                    int id, float pv) {
#pragma unroll
  for (int i = K - 1; i > 0; --i) {
    const bool above = key > tk[i - 1];  // the new entry goes above slot i - 1
    const bool here = key > tk[i];
    tk[i] = above ? tk[i - 1] : (here ? key : tk[i]);
    ti[i] = above ? ti[i - 1] : (here ? id : ti[i]);
    tp[i] = above ? tp[i - 1] : (here ? pv : tp[i]);
  }
  if (K > 0 && key > tk[0]) {
    tk[0] = key;
    ti[0] = id;
    tp[0] = pv;
  }
}

// Counter increment with release and acquire semantics at GPU scope.  After a
// CTA barrier, one thread's increment publishes every earlier write of the
// CTA (release is cumulative over the barrier); the thread that sees the
// final count then observes every other CTA's writes (acquire), and a barrier
// passes that on to the rest of its CTA.
__device__ __forceinline__ int atom_add_acq_rel(int* ptr, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(ptr), "r"(v)
               : "memory");
  return old;
}

// v * 2^32 is exact in float (a power-of-two scale), so the integer added is
// v's value to 2^-32 with nothing rounded but v itself.  The router does no
// FP64 arithmetic: this part's FP64 units are few, and a few dozen FP64
// operations per thread cost microseconds.
__device__ __forceinline__ void add_fixed(unsigned long long* acc, float v) {
  atomicAdd(acc, static_cast<unsigned long long>(__float2ll_rn(v * kFix)));
}


// Exclusive scan of one int per epilogue thread (fixed order); *total gets
// the sum.  All 256 epilogue threads call it.
__device__ int epi_exclusive_scan(RouterSmem* st, int eidx, int v, int* total) {
  const int lane = eidx & 31, w = eidx >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) st->wtot[w] = x;
  named_bar_sync(kBarEpi, kEpiThreads);
  int before_w = 0, tot = 0;
  for (int i = 0; i < kEpiWarps; ++i) {
    const int t = st->wtot[i];
    if (i < w) before_w += t;
    tot += t;
  }
  named_bar_sync(kBarEpi, kEpiThreads);
  *total = tot;
  return before_w + x - v;
}

// Sums of two floats per epilogue thread in a fixed order (xor tree in each
// warp, then the warps in order); every thread gets both.
__device__ float2 epi_sum2(RouterSmem* st, int eidx, float a, float b) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  if ((eidx & 31) == 0) {
    st->fred[eidx >> 5] = a;
    st->fred2[eidx >> 5] = b;
  }
  named_bar_sync(kBarEpi, kEpiThreads);
  float ra = 0.0f, rb = 0.0f;
#pragma unroll
  for (int w = 0; w < kEpiWarps; ++w) {
    ra += st->fred[w];
    rb += st->fred2[w];
  }
  named_bar_sync(kBarEpi, kEpiThreads);
  return make_float2(ra, rb);
}

// Column sums of a warp's 32 rows: lane l holds 16 values (columns 0..15 of
// its row); afterwards lanes 2c and 2c+1 hold the total of column c.  Four
// halving exchanges (xor 16, 8, 4, 2) then a pair sum (xor 1), all in a fixed
// order.
__device__ __forceinline__ float warp_column_sums16(const float (&a)[16], int lane) {
  float b8[8], b4[4], b2[2];
  const bool u16 = (lane & 16) != 0, u8 = (lane & 8) != 0, u4 = (lane & 4) != 0,
             u2 = (lane & 2) != 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float send = u16 ? a[i] : a[i + 8];
    const float keep = u16 ? a[i + 8] : a[i];
    b8[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = u8 ? b8[i] : b8[i + 4];
    const float keep = u8 ? b8[i + 4] : b8[i];
    b4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = u4 ? b4[i] : b4[i + 2];
    const float keep = u4 ? b4[i + 2] : b4[i];
    b2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  const float send = u2 ? b2[0] : b2[1];
  const float keep = u2 ? b2[1] : b2[0];
  const float c = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  return c + __shfl_xor_sync(0xffffffffu, c, 1);
}

// The reductions across tiles, run by the epilogue warps of the CTA that
// completed the last tile (epilogue thread e handles expert e).  Every global
// read is issued first; every accumulator is left at zero.
__device__ void finalize_all(const RouterArgs& p, RouterSmem* st, int eidx, int ntiles) {
  const int E = p.E;
  const int e = eidx;
  const bool ec = p.fixed_count >= 0;
  const bool in = e < E;
  // ---- loads
  const int n = in ? (ec ? p.fixed_count : __ldcg(p.acc_count + e)) : 0;
  const long long ps = in ? static_cast<long long>(__ldcg(p.acc_psum + e)) : 0ll;
  const bool want_imp = p.importance != nullptr || p.importance_cv2 != nullptr;
  const long long is = (in && want_imp) ? static_cast<long long>(__ldcg(p.acc_imp + e)) : 0ll;
  const long long es = (e == 0 && p.entropy_mean) ? static_cast<long long>(__ldcg(p.acc_ent)) : 0ll;
  float zf = 0.0f;
  for (int t = eidx; t < ntiles; t += kEpiThreads) zf += __ldcg(p.tile_lse2 + t);
  int cv[8];
  const bool chunks = p.chunk_acc != nullptr && in;
#pragma unroll
  for (int i = 0; i < 8; ++i) cv[i] = (chunks && i < p.n_chunks) ? __ldcg(p.chunk_acc + i * E + e) : 0;
  // ---- per-expert outputs
  // pair and token counts stay below 2^24, exact in float
  const float n_pairs = p.n_pairs >= 0.0 ? static_cast<float>(p.n_pairs)
                                         : static_cast<float>(p.k) * static_cast<float>(p.T);
  const float inv_T = p.T > 0 ? 1.0f / static_cast<float>(p.T) : 0.0f;
  const float fe = (in && p.T > 0 && n_pairs > 0.0f) ? static_cast<float>(n) / n_pairs : 0.0f;
  const float Pe = (in && p.T > 0) ? static_cast<float>(ps) * (1.0f / kFix) * inv_T : 0.0f;
  if (in) {
    if (p.counts) p.counts[e] = n;
    if (p.f) p.f[e] = fe;
    if (p.P) p.P[e] = Pe;
  }
  // ---- per-chunk bases of the permutation: exclusive scan over chunks
  if (chunks) {
    int run = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < p.n_chunks) {
        p.chunk_base[i * E + e] = run;
        p.chunk_acc[i * E + e] = 0;
      }
      run += cv[i];
    }
    for (int c = 8; c < p.n_chunks; ++c) {  // more than 8 chunks: T > 32768 tokens
      const int v = __ldcg(p.chunk_acc + c * E + e);
      p.chunk_base[c * E + e] = run;
      p.chunk_acc[c * E + e] = 0;
      run += v;
    }
  }
  // ---- scans over experts: offsets of the kept rows (and before capacity)
  if (p.offsets) {
    const int kept = in ? ((p.C >= 0 && n > p.C) ? static_cast<int>(p.C) : n) : 0;
    int R = 0;
    const int off = epi_exclusive_scan(st, eidx, kept, &R);
    if (in) p.offsets[e] = off;
    if (e == 0) p.offsets[E] = R;
  }
  if (p.all_offsets) {
    int n_all = 0;
    const int off = epi_exclusive_scan(st, eidx, n, &n_all);
    if (in) p.all_offsets[e] = off;
    if (e == 0) p.all_offsets[E] = n_all;
  }
  // ---- losses (fixed-order float sums)
  const float imp = static_cast<float>(is) * (1.0f / kFix);
  const float2 s1 = epi_sum2(st, eidx, fe * Pe, zf);
  if (want_imp) {
    if (in && p.importance) p.importance[e] = imp;
    const float mean = epi_sum2(st, eidx, imp, 0.0f).x / E;
    const float var = epi_sum2(st, eidx, in ? (imp - mean) * (imp - mean) : 0.0f, 0.0f).x / E;
    if (e == 0 && p.importance_cv2) *p.importance_cv2 = mean != 0.0f ? var / (mean * mean) : 0.0f;
  }
  if (e == 0) {
    if (p.bal_loss) *p.bal_loss = p.balance_coef * static_cast<float>(E) * s1.x;
    if (p.z_loss) *p.z_loss = (p.T > 0) ? static_cast<float>(s1.y * inv_T) : 0.0f;
    if (p.entropy_mean)
      *p.entropy_mean =
          (p.T > 0) ? static_cast<float>(es) * (1.0f / kFix) * inv_T : 0.0f;
  }
  // ---- every accumulator back to zero (all of them were read above)
  if (in) {
    p.acc_count[e] = 0;
    p.acc_psum[e] = 0ull;
    if (p.acc_imp) p.acc_imp[e] = 0ull;
  }
  if (e == 0) {
    if (p.acc_ent) *p.acc_ent = 0ull;
    *p.tiles_done = 0;
  }
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
  const RouterGeom geo = router_geom(E, p.stages);
  const int a_bytes = 128 * kBK * 2;
  RouterSmem* st =
      reinterpret_cast<RouterSmem*>(smem + static_cast<size_t>(geo.stages) * geo.stage_bytes);
  volatile int* abort_flag = &st->abort_flag;
  const uint32_t tmem_cols = 2 * geo.buf_cols;
  const int ntiles = (p.T + 127) / 128;
  const int units = ntiles * S;
  const int nk = p.d / kBK;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < geo.stages; ++s) {
      mbar_init(&st->full[s], 1);
      mbar_init(&st->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&st->tfull[b], 1);
      mbar_init(&st->tempty[b], kEpiWarps);
    }
    mbar_init(&st->fin, 1);
    st->abort_flag = 0;
    fence_barrier_init();
  }
  // x, the offsets and the bias may come from the previous kernel in the stream
  pdl_wait();
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
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      if (static_cast<int>(blockIdx.x) < units) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
      }
      uint32_t uses = 0;  // loads issued; stage = uses % stages
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok && !*abort_flag; u += gridDim.x) {
        const int t = u / S, s = u - t * S;
        const int kb0 = s * nk / S, kb1 = (s + 1) * nk / S;
        for (int kb = kb0; kb < kb1; ++kb, ++uses) {
          const int stage = static_cast<int>(uses % geo.stages);
          const uint32_t phase = (uses / geo.stages) & 1u;
          if (!mbar_wait_bounded(&st->empty[stage], phase ^ 1u, p.timeout_ns, p.status,
                                 abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * geo.stage_bytes;
          mbar_arrive_expect_tx(&st->full[stage], static_cast<uint32_t>(geo.stage_bytes));
          tma_load_2d(sa, &tmX, &st->full[stage], kb * kBK, t * 128);
          tma_load_2d(sa + a_bytes, &tmW, &st->full[stage], kb * kBK, 0);
        }
      }
      // drain: the last copy into each used stage must land before exit
      for (uint32_t s = 0; s < static_cast<uint32_t>(geo.stages) && s < uses; ++s) {
        const uint32_t n_s = (uses - 1u - s) / geo.stages + 1u;  // uses of stage s
        mbar_wait_bounded(&st->full[s], (n_s - 1u) & 1u, p.timeout_ns, p.status, nullptr);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, static_cast<uint32_t>(geo.N));
      uint32_t uses = 0;
      int local = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok && !*abort_flag; u += gridDim.x, ++local) {
        const int t = u / S, s = u - t * S;
        (void)t;
        const int kb0 = s * nk / S, kb1 = (s + 1) * nk / S;
        const int b = local & 1;
        const uint32_t q = static_cast<uint32_t>(local >> 1);
        if (!mbar_wait_bounded(&st->tempty[b], (q & 1u) ^ 1u, p.timeout_ns, p.status,
                               abort_flag))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b) * geo.buf_cols;
        for (int kb = kb0; kb < kb1; ++kb, ++uses) {
          const int stage = static_cast<int>(uses % geo.stages);
          const uint32_t phase = (uses / geo.stages) & 1u;
          if (!mbar_wait_bounded(&st->full[stage], phase, p.timeout_ns, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * geo.stage_bytes);
          const uint32_t sb = sa + a_bytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            tc_mma_bf16(d_tmem, smem_desc_sw128(sa + kk * 32), smem_desc_sw128(sb + kk * 32),
                        idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
          tc_commit(&st->empty[stage]);
        }
        if (!ok) break;
        tc_commit(&st->tfull[b]);
      }
      // every issued MMA must retire before TMEM is freed (also on abort)
      tc_commit(&st->fin);
      mbar_wait_bounded(&st->fin, 0, p.timeout_ns, p.status, nullptr);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue
    const int eidx = static_cast<int>(threadIdx.x) - 64;  // 0..511
    const int c = eidx >> 7;                             // column part
    const int quarter = warp & 3;                        // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;                   // this thread's tile row
    const int ng = (E + 15) / 16;  // 16-column groups; part c owns groups c, c+4, ...
    const int nparts = ng < kParts ? ng : kParts;  // parts that own a group
    const bool sigmoid = (p.flags & kRouteSigmoid) != 0;
    const bool renorm = (p.flags & kRouteNoRenorm) == 0;
    const bool want_imp = p.acc_imp != nullptr && K > 0;
    const bool want_ent = p.acc_ent != nullptr;
    // hands the TMEM buffer back to the MMA warp (one arrival per warp)
    auto release = [&](int b) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&st->tempty[b]);
    };
    // totals of colsum[0..3][e] in quarter order, added to acc[e] (fixed point)
    auto add_column_totals = [&](unsigned long long* acc, int e) {
      if (e < E) {
        const float tot =
            ((st->colsum[0][e] + st->colsum[1][e]) + st->colsum[2][e]) + st->colsum[3][e];
        add_fixed(acc + e, tot);
      }
    };
    // this warp's 32-row column sums of group g (lanes 2j, 2j+1 hold column j)
    auto stage_columns = [&](int g, const float (&a)[16]) {
      const float s = warp_column_sums16(a, lane);
      const int e = g * 16 + (lane >> 1);
      if ((lane & 1) == 0 && e < E) st->colsum[quarter][e] = s;
    };
    int local = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++local) {
      const int t = u / S, s = u - t * S;
      const int b = local & 1;
      const uint32_t q = static_cast<uint32_t>(local >> 1);
      // one thread waits for the accumulator and every epilogue warp follows
      // its decision, so that all of them take the same path through the
      // named barriers below
      if (eidx == 0)
        st->go = mbar_wait_bounded(&st->tfull[b], q & 1u, p.timeout_ns, p.status, abort_flag);
      named_bar_sync(kBarEpi, kEpiThreads);
      if (!st->go) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(b) * geo.buf_cols;
      bool run_tile = true;
      if (S > 1) {
        // partial logits of slice s, [slice][tile][expert][row] (coalesced per expert)
        float* part = p.part_logits + ((static_cast<size_t>(s) * ntiles + t) * E) * 128 + r;
#pragma unroll 1
        for (int g = c; g < ng; g += kParts) {
          float v[16];
          tmem_ld16(taddr + g * 16, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (g * 16 + j < E) part[static_cast<size_t>(g * 16 + j) * 128] = v[j];
        }
        named_bar_sync(kBarEpi, kEpiThreads);
        if (eidx == 0) {
          const int last = atom_add_acq_rel(p.tile_arrive + t, 1) == S - 1;
          if (last) p.tile_arrive[t] = 0;  // ready for the next call
          st->flag = last;
        }
        named_bar_sync(kBarEpi, kEpiThreads);
        run_tile = st->flag != 0;
        if (run_tile) {
          // the S partials summed in slice order (two slices per round trip)
          // into this unit's TMEM buffer
          const float* part0 = p.part_logits + (static_cast<size_t>(t) * E) * 128 + r;
          const size_t slice = static_cast<size_t>(ntiles) * E * 128;
#pragma unroll 1
          for (int g = c; g < ng; g += kParts) {
            const float* src = part0 + static_cast<size_t>(g * 16) * 128;
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = 0.0f;
#pragma unroll 1
            for (int ss = 0; ss < S; ss += 2) {
              float a0[16], a1[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const bool in = g * 16 + j < E;
                a0[j] = in ? __ldcg(src + ss * slice + j * 128) : 0.0f;
                a1[j] = in ? __ldcg(src + (ss + 1) * slice + j * 128) : 0.0f;
              }
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] = (v[j] + a0[j]) + a1[j];
            }
            tmem_st16(taddr + g * 16, v);
          }
          tmem_st_wait();
        } else {
          release(b);
        }
      }
      if (run_tile) {
        // ------------------------------------------------ the tile's epilogue
        const int tok = t * 128 + r;
        const bool valid = tok < p.T;
        // pass 1: running max m and, relative to it, the sum of exponentials
        // and sum ex (l - m); a group that raises m rescales both first
        float m = -INFINITY, sx = 0.0f, hs = 0.0f;
#pragma unroll 1
        for (int g = c; g < ng; g += kParts) {
          float v[16];
          tmem_ld16(taddr + g * 16, v);
          tmem_ld_wait();
          float gm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            v[j] += st->off[g * 16 + j];
            if (g * 16 + j < E) gm[j & 3] = fmaxf(gm[j & 3], v[j]);
          }
          const float mg = fmaxf(fmaxf(gm[0], gm[1]), fmaxf(gm[2], gm[3]));
          if (mg > m) {
            if (m != -INFINITY) {
              const float a = __expf(m - mg);
              hs = a * fmaf(m - mg, sx, hs);
              sx *= a;
            }
            m = mg;
          }
          float sp[4] = {0.0f, 0.0f, 0.0f, 0.0f}, hp[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (g * 16 + j < E) {
              const float l = v[j] - m;
              const float ex = __expf(l);
              sp[j & 3] += ex;
              hp[j & 3] = fmaf(ex, l, hp[j & 3]);
            }
          sx += (sp[0] + sp[1]) + (sp[2] + sp[3]);
          hs += (hp[0] + hp[1]) + (hp[2] + hp[3]);
        }
        st->xm[c][r] = m;
        st->xs[c][r] = sx;
        st->xh[c][r] = hs;
        named_bar_sync(kBarEpi, kEpiThreads);
        // the parts in order: row max, then the sums moved to it
        m = st->xm[0][r];
        for (int i = 1; i < nparts; ++i) m = fmaxf(m, st->xm[i][r]);
        sx = 0.0f;
        hs = 0.0f;
        for (int i = 0; i < nparts; ++i) {
          const float mi = st->xm[i][r], si = st->xs[i][r];
          const float a = __expf(mi - m);
          sx = fmaf(a, si, sx);
          hs = fmaf(a, fmaf(mi - m, si, st->xh[i][r]), hs);
        }
        const float inv_s = 1.0f / sx;
        const float lse = m + logf(sx);
        // pass 2: scores, keys, this thread's Top-k list, column sums of P
        float top_key[K > 0 ? K : 1];
        int top_id[K > 0 ? K : 1];
        float top_p[K > 0 ? K : 1];
#pragma unroll
        for (int j = 0; j < K; ++j) {
          top_key[j] = -INFINITY;
          top_id[j] = 0x7fffffff;
          top_p[j] = 0.0f;
        }
        float thresh = -INFINITY;
        float ssum = 0.0f, slog = 0.0f;  // sigmoid: sum s, sum s log s
#pragma unroll 1
        for (int g = c; g < ng; g += kParts) {
          float v[16];
          tmem_ld16(taddr + g * 16, v);
          tmem_ld_wait();
          float pe[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int e = g * 16 + j;
            pe[j] = 0.0f;
            if (e < E) {
              const float l = v[j] + st->off[e];
              if (sigmoid) {
                const float en = __expf(-l);
                pe[j] = 1.0f / (1.0f + en);
                ssum += pe[j];
                if (pe[j] > 0.0f) slog -= pe[j] * log1pf(en);  // s log s = -s log(1 + e^-l)
              } else {
                pe[j] = __expf(l - m) * inv_s;
              }
            }
          }
          // candidates in ascending expert order (equal keys keep the lower
          // index first); the threshold rises as entries go in
          if (K > 0) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int e = g * 16 + j;
              const float key = pe[j] + st->bias[e];
              if (e < E && key > thresh) {
                topk_push_ascending<K>(top_key, top_id, top_p, key, e, pe[j]);
                thresh = top_key[K > 0 ? K - 1 : 0];
              }
            }
          }
          if (p.scores_t != nullptr && valid) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (g * 16 + j < E) p.scores_t[static_cast<size_t>(g * 16 + j) * p.T + tok] = pe[j];
          }
          if (!valid) {
#pragma unroll
            for (int j = 0; j < 16; ++j) pe[j] = 0.0f;
          }
          stage_columns(g, pe);
        }
        // the logits are no longer needed: the next unit may use the buffer
        release(b);
        if (c > 0 && c < nparts) {
#pragma unroll
          for (int j = 0; j < K; ++j) {
            st->tk_p[c - 1][j][r] = top_p[j];
            st->tk_id[c - 1][j][r] = top_id[j];
          }
        }
        st->xq[c][r] = ssum;
        st->xg[c][r] = slog;
        named_bar_sync(kBarEpi, kEpiThreads);
        if (c >= 2) {
          add_column_totals(p.acc_psum, eidx - 256);  // parts 2, 3: expert eidx - 256
        } else if (c == 0) {
          // merge the other parts' lists (each descending: stop at the first
          // entry that does not make it)
#pragma unroll 1
          for (int i = 1; i < nparts; ++i) {
#pragma unroll 1
            for (int j = 0; j < K; ++j) {
              const int id = st->tk_id[i - 1][j][r];
              if (id >= E) break;
              const float pv = st->tk_p[i - 1][j][r];
              const float key = pv + st->bias[id];
              if (!before(key, id, top_key[K > 0 ? K - 1 : 0], top_id[K > 0 ? K - 1 : 0])) break;
              topk_insert<K>(top_key, top_id, top_p, key, id, pv);
            }
          }
          // entropy of the router distribution: softmax log s - sum ex (l-m) / s;
          // sigmoid q = s / sum s: log sum s - sum s log s / sum s
          float ent = 0.0f;
          if (sigmoid) {
            float ss = 0.0f, sl = 0.0f;
            for (int i = 0; i < nparts; ++i) {
              ss += st->xq[i][r];
              sl += st->xg[i][r];
            }
            ent = logf(ss) - sl / ss;
          } else {
            ent = logf(sx) - hs * inv_s;
          }
          st->rowv[0][r] = valid ? lse * lse : 0.0f;
          st->rowv[1][r] = valid ? ent : 0.0f;
          if (K > 0) {
            float denom = 0.0f;
#pragma unroll
            for (int j = 0; j < K; ++j) denom += top_p[j];
            const float inv_d = renorm ? 1.0f / denom : 1.0f;
#pragma unroll
            for (int j = 0; j < K; ++j) {
              const float gj = top_p[j] * inv_d;
              st->tk_id[0][j][r] = valid ? top_id[j] : -1;  // the merged selection
              st->tk_p[0][j][r] = gj;
              if (valid) {
                p.ids[static_cast<int64_t>(tok) * K + j] = top_id[j];
                p.gates[static_cast<int64_t>(tok) * K + j] = gj;
                if (p.pair_score) p.pair_score[static_cast<int64_t>(tok) * K + j] = top_p[j];
                // a slot left unfilled (only with NaN scores) names no expert
                if (top_id[j] < E) atomicAdd(&st->hist[top_id[j]], 1);
              }
            }
          }
        }
        named_bar_sync(kBarEpi, kEpiThreads);
        // tile totals: expert counts, lse^2 (per tile, summed in tile order by
        // the finalize), entropy (fixed point)
        for (int e = eidx; e < E; e += kEpiThreads) {
          const int hcount = st->hist[e];
          if (K > 0 && hcount != 0) atomicAdd(p.acc_count + e, hcount);
          if (p.tile_hist) p.tile_hist[static_cast<int64_t>(t) * E + e] = hcount;
          if (p.chunk_acc && hcount != 0)
            atomicAdd(p.chunk_acc + (t / p.chunk_tiles) * E + e, hcount);
          st->hist[e] = 0;
        }
        if (warp == 2 + 8) {  // one warp (eidx 256..287): the two row sums in a fixed order
          float z = 0.0f, hsum = 0.0f;
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            z += st->rowv[0][lane * 4 + x];
            hsum += st->rowv[1][lane * 4 + x];
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            z += __shfl_xor_sync(0xffffffffu, z, o);
            hsum += __shfl_xor_sync(0xffffffffu, hsum, o);
          }
          if (lane == 0) {
            p.tile_lse2[t] = z;
            if (want_ent) add_fixed(p.acc_ent, hsum);
          }
        }
        if (want_imp) {
          // importance: each row's sparse gate vector (gates on the selected
          // experts, 0 elsewhere), column sums as for P
#pragma unroll 1
          for (int g = c; g < ng; g += kParts) {
            float gv[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) gv[j] = 0.0f;
#pragma unroll
            for (int j = 0; j < K; ++j) {
              const int id = st->tk_id[0][j][r];
              const float gate = st->tk_p[0][j][r];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                if (id == g * 16 + i) gv[i] = gate;
            }
            stage_columns(g, gv);
          }
          named_bar_sync(kBarEpi, kEpiThreads);
          if (c >= 2) add_column_totals(p.acc_imp, eidx - 256);
        }
        // this tile is done: the CTA that completes the last tile reduces
        named_bar_sync(kBarEpi, kEpiThreads);
        if (eidx == 0) st->flag = atom_add_acq_rel(p.tiles_done, 1) == ntiles - 1;
        named_bar_sync(kBarEpi, kEpiThreads);
        if (st->flag) finalize_all(p, st, eidx, ntiles);
      }
    }
    if (ntiles == 0 && blockIdx.x == 0) finalize_all(p, st, eidx, 0);
  }

  tc_fence_before();
  __syncthreads();
  pdl_trigger();  // this CTA's work is done: the next kernel's CTAs may come up
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, tmem_cols);
}

}  // namespace

int router_split(int T, int d, int num_sms, int max_split) {
  const int ntiles = (T + 127) / 128;
  const int nk = d / kBK;
  // Split K while every slice still gets its own SM and keeps >= 2 k-blocks.
  int S = 1;
  while (S < kMaxSplit && 2 * S <= max_split && ntiles * 2 * S <= num_sms && nk / (2 * S) >= 2)
    S *= 2;
  return S;
}

int launch_router(const CUtensorMap& x_map, const CUtensorMap& wr_map, RouterArgs args,
                  int num_sms, cudaStream_t stream) {
  const int ntiles = (args.T + 127) / 128;
  if (args.E > 256 || args.k > kMaxTopK || args.k < 0) return -2;
  const int S = router_split(args.T, args.d, num_sms, args.max_split);
  if (S > 1 && (args.part_logits == nullptr || args.tile_arrive == nullptr)) return -2;
  if (args.acc_count == nullptr || args.acc_psum == nullptr || args.tiles_done == nullptr ||
      args.tile_lse2 == nullptr)
    return -2;
  if ((args.importance != nullptr || args.importance_cv2 != nullptr) && args.acc_imp == nullptr)
    return -2;
  if (args.entropy_mean != nullptr && args.acc_ent == nullptr) return -2;
  if ((args.chunk_acc == nullptr) != (args.chunk_base == nullptr) || args.chunk_tiles < 1) return -2;
  const size_t tail = sizeof(RouterSmem) + 1024;
  const int stage_bytes = router_geom(args.E, 1).stage_bytes;
  const int nk_unit = (args.d / kBK + S - 1) / S;
  int stages = static_cast<int>((227 * 1024 - tail) / stage_bytes);
  stages = stages > kMaxStages ? kMaxStages : stages;
  const int units = ntiles * S;
  const int grid = units < num_sms ? (units > 0 ? units : 1) : num_sms;
  const int units_per_cta = (units + grid - 1) / grid;
  const int max_useful = nk_unit * (units_per_cta > 0 ? units_per_cta : 1);
  stages = stages > max_useful ? max_useful : stages;
  stages = stages < 1 ? 1 : stages;
  if (stages < 2 && max_useful >= 2) return -2;  // W_r too wide for two stages
  args.split = S;
  args.stages = stages;
  const size_t smem = tail + static_cast<size_t>(stages) * stage_bytes;
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
  if (launch_kernel(kern, dim3(grid), dim3(kThreads), smem, stream, args.pdl != 0, 1u, x_map,
                    wr_map, args) != cudaSuccess)
    return -3;
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace moe
