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
// one of two TMEM buffers, and eight epilogue warps drain the other buffer, so
// a unit's epilogue overlaps the next unit's loads.  A K-split unit stores its
// partial logits to the workspace (coalesced, [expert][row] per tile); the
// CTA that stores a tile's last slice sums the S partials in slice order,
// writes the sums back into its TMEM buffer and runs the tile's epilogue.
//
// The epilogue reads the logits straight from TMEM: thread (row r, half h)
// owns 32-column chunks h, h+2, ... of row r.  Three passes over the chunks:
// row max, sum of exponentials, then the scores, the keys and a per-thread
// Top-k list; the two halves exchange max, sum and lists through shared
// memory.  Column sums over the tile's rows (P, importance) go through a
// transposition buffer in a fixed order.  Every cross-tile total is either a
// 64-bit integer atomic on fixed-point values (P and importance at 2^-32,
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
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = 64 + kEpiThreads;  // TMA warp, MMA warp, 8 epilogue warps
constexpr int kMaxSplit = 8;
constexpr int kTbPitch = 129;               // transposition buffer row pitch (floats)
constexpr double kFix = 4294967296.0;       // 2^32: fixed-point scale of P, importance, entropy
constexpr int kBarEpi = 1;                  // named barrier of the 8 epilogue warps
constexpr int kBarHalf = 2;                 // + h: named barrier of epilogue half h

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
  float off[256];
  float bias[256];
  float xm[2][128];         // per-half row max
  float xs[2][128];         // per-half sum of exponentials
  float xh[2][128];         // per-half entropy partial (softmax: sum ex (l - m); sigmoid: sum s)
  float xq[2][128];         // sigmoid: per-half sum s
  float xg[2][128];         // sigmoid: per-half sum s log s
  // half 1's Top-k list per row; after the merge (by the same row's half-0
  // thread) the merged selection: ids in tk_id, gates in tk_p
  float tk_key[kMaxTopK][128];
  int tk_id[kMaxTopK][128];
  float tk_p[kMaxTopK][128];
  float rowv[2][128];       // per-row lse^2 and entropy, for the tile sums
  float red[2][4][16];      // column-sum partials: [half][row quarter][column]
  double dred[kEpiWarps];   // finalize: per-warp sums
  double dred2[kEpiWarps];
  int wtot[kEpiWarps];
  float tb[2][16 * kTbPitch];  // transposition buffers (16 columns), one per half
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

__device__ __forceinline__ void add_fixed(unsigned long long* acc, double v) {
  atomicAdd(acc, static_cast<unsigned long long>(__double2ll_rn(v * kFix)));
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

// Sums of two doubles per epilogue thread in a fixed order (xor tree in each
// warp, then the warps in order); every thread gets both.
__device__ double2 epi_sum2(RouterSmem* st, int eidx, double a, double b) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  if ((eidx & 31) == 0) {
    st->dred[eidx >> 5] = a;
    st->dred2[eidx >> 5] = b;
  }
  named_bar_sync(kBarEpi, kEpiThreads);
  double ra = 0.0, rb = 0.0;
#pragma unroll
  for (int w = 0; w < kEpiWarps; ++w) {
    ra += st->dred[w];
    rb += st->dred2[w];
  }
  named_bar_sync(kBarEpi, kEpiThreads);
  return make_double2(ra, rb);
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
  const double n_pairs = p.n_pairs >= 0.0 ? p.n_pairs
                                          : static_cast<double>(p.k) * static_cast<double>(p.T);
  const double inv_pairs = n_pairs > 0.0 ? 1.0 / n_pairs : 0.0;
  const double inv_T = p.T > 0 ? 1.0 / p.T : 0.0;
  const double fe = (in && p.T > 0) ? static_cast<double>(n) * inv_pairs : 0.0;
  const double Pe = (in && p.T > 0) ? static_cast<double>(ps) * (1.0 / kFix) * inv_T : 0.0;
  if (in) {
    if (p.counts) p.counts[e] = n;
    if (p.f) p.f[e] = static_cast<float>(fe);
    if (p.P) p.P[e] = static_cast<float>(Pe);
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
  // ---- losses
  const double imp = static_cast<double>(is) * (1.0 / kFix);
  const double2 s1 = epi_sum2(st, eidx, fe * Pe, static_cast<double>(zf));
  if (want_imp) {
    if (in && p.importance) p.importance[e] = static_cast<float>(imp);
    const double mean = epi_sum2(st, eidx, imp, 0.0).x / E;
    const double var = epi_sum2(st, eidx, in ? (imp - mean) * (imp - mean) : 0.0, 0.0).x / E;
    if (e == 0 && p.importance_cv2)
      *p.importance_cv2 = static_cast<float>(mean != 0.0 ? var / (mean * mean) : 0.0);
  }
  if (e == 0) {
    if (p.bal_loss) *p.bal_loss = static_cast<float>(static_cast<double>(p.balance_coef) * E * s1.x);
    if (p.z_loss) *p.z_loss = (p.T > 0) ? static_cast<float>(s1.y * inv_T) : 0.0f;
    if (p.entropy_mean)
      *p.entropy_mean =
          (p.T > 0) ? static_cast<float>(static_cast<double>(es) * (1.0 / kFix) * inv_T) : 0.0f;
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
    const int eidx = static_cast<int>(threadIdx.x) - 64;  // 0..255
    const int h = eidx >> 7;                             // column half
    const int quarter = warp & 3;                        // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;                   // this thread's tile row
    const int ng = (E + 15) / 16;  // 16-column groups; half h owns groups h, h+2, ...
    const bool sigmoid = (p.flags & kRouteSigmoid) != 0;
    const bool renorm = (p.flags & kRouteNoRenorm) == 0;
    const bool want_imp = p.acc_imp != nullptr && K > 0;
    const bool want_ent = p.acc_ent != nullptr;
    float* tb = st->tb[h];
    // Column sums of the 16 values per row this half staged in tb: the warp of
    // each row quarter sums its 32 rows (lane = column), then the quarters in
    // order; the total of column j goes to acc[g*16 + j] (fixed point).
    auto column_sums = [&](int g, unsigned long long* acc) {
      named_bar_sync(kBarHalf + h, 128);
      if (lane < 16) {
        float x = 0.0f;
#pragma unroll 8
        for (int i = 0; i < 32; ++i) x += tb[lane * kTbPitch + quarter * 32 + i];
        st->red[h][quarter][lane] = x;
      }
      named_bar_sync(kBarHalf + h, 128);
      if (quarter == 0 && lane < 16 && g * 16 + lane < E) {
        const float tot =
            ((st->red[h][0][lane] + st->red[h][1][lane]) + st->red[h][2][lane]) + st->red[h][3][lane];
        add_fixed(acc + g * 16 + lane, static_cast<double>(tot));
      }
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
        for (int g = h; g < ng; g += 2) {
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
          for (int g = h; g < ng; g += 2) {
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
        }
      }
      if (run_tile) {
        // ------------------------------------------------ the tile's epilogue
        const int tok = t * 128 + r;
        const bool valid = tok < p.T;
        // pass 1: row max (four independent maxima)
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
        for (int g = h; g < ng; g += 2) {
          float v[16];
          tmem_ld16(taddr + g * 16, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (g * 16 + j < E) mx[j & 3] = fmaxf(mx[j & 3], v[j] + st->off[g * 16 + j]);
        }
        float m = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        st->xm[h][r] = m;
        named_bar_sync(kBarEpi, kEpiThreads);
        m = fmaxf(st->xm[0][r], st->xm[1][r]);
        // pass 2: sum of exponentials (and sum ex (l - m) for the entropy)
        // (four independent partial sums per thread, combined in a fixed order)
        float sp[4] = {0.0f, 0.0f, 0.0f, 0.0f}, hp[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 1
        for (int g = h; g < ng; g += 2) {
          float v[16];
          tmem_ld16(taddr + g * 16, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (g * 16 + j < E) {
              const float l = v[j] + st->off[g * 16 + j] - m;
              const float ex = __expf(l);
              sp[j & 3] += ex;
              hp[j & 3] = fmaf(ex, l, hp[j & 3]);
            }
        }
        float sx = (sp[0] + sp[1]) + (sp[2] + sp[3]);
        float hs = (hp[0] + hp[1]) + (hp[2] + hp[3]);
        st->xs[h][r] = sx;
        st->xh[h][r] = hs;
        named_bar_sync(kBarEpi, kEpiThreads);
        sx = st->xs[0][r] + st->xs[1][r];
        hs = st->xh[0][r] + st->xh[1][r];
        const float inv_s = 1.0f / sx;
        const float lse = m + logf(sx);
        // pass 3: scores, keys, this thread's Top-k list, column sums of P
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
        for (int g = h; g < ng; g += 2) {
          float v[16];
          tmem_ld16(taddr + g * 16, v);
          tmem_ld_wait();
          // scores into the transposition buffer (0 for rows past T) and a
          // mask of the experts whose key beats the list's current last entry
          uint32_t cand = 0u;
          if (sigmoid) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int e = g * 16 + j;
              float pe = 0.0f;
              if (e < E) {
                const float en = __expf(-(v[j] + st->off[e]));
                pe = 1.0f / (1.0f + en);
                ssum += pe;
                if (pe > 0.0f) slog -= pe * log1pf(en);  // s log s = -s log(1 + e^-l)
                if (pe + st->bias[e] > thresh) cand |= 1u << j;
              }
              tb[j * kTbPitch + r] = valid ? pe : 0.0f;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int e = g * 16 + j;
              float pe = 0.0f;
              if (e < E) {
                pe = __expf(v[j] + st->off[e] - m) * inv_s;
                if (pe + st->bias[e] > thresh) cand |= 1u << j;
              }
              tb[j * kTbPitch + r] = valid ? pe : 0.0f;
            }
          }
          // candidates in ascending expert order (equal keys keep the lower
          // index first); the threshold rises as entries go in
          if (K > 0) {
            while (cand != 0u) {
              const int j = __ffs(cand) - 1;
              cand &= cand - 1u;
              const int e = g * 16 + j;
              const float pe = tb[j * kTbPitch + r];
              const float key = pe + st->bias[e];
              if (key > thresh) {
                topk_push_ascending<K>(top_key, top_id, top_p, key, e, pe);
                thresh = top_key[K > 0 ? K - 1 : 0];
              }
            }
          }
          if (p.scores_t != nullptr && valid) {
#pragma unroll 1
            for (int j = 0; j < 16 && g * 16 + j < E; ++j)
              p.scores_t[static_cast<size_t>(g * 16 + j) * p.T + tok] = tb[j * kTbPitch + r];
          }
          column_sums(g, p.acc_psum);
        }
        // merge the two halves' Top-k lists (half 0 keeps the result)
        if (h == 1) {
#pragma unroll
          for (int j = 0; j < K; ++j) {
            st->tk_key[j][r] = top_key[j];
            st->tk_id[j][r] = top_id[j];
            st->tk_p[j][r] = top_p[j];
          }
        }
        st->xq[h][r] = ssum;
        st->xg[h][r] = slog;
        named_bar_sync(kBarEpi, kEpiThreads);
        if (h == 0) {
#pragma unroll 1
          for (int i = 0; i < K; ++i)
            topk_insert<K>(top_key, top_id, top_p, st->tk_key[i][r], st->tk_id[i][r],
                           st->tk_p[i][r]);
          // entropy of the router distribution: softmax log s - sum ex (l-m) / s;
          // sigmoid q = s / sum s: log sum s - sum s log s / sum s
          float ent = 0.0f;
          if (sigmoid) {
            const float ss = st->xq[0][r] + st->xq[1][r];
            const float sl = st->xg[0][r] + st->xg[1][r];
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
              st->tk_id[j][r] = valid ? top_id[j] : -1;  // the merged selection
              st->tk_p[j][r] = gj;
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
        if (warp == 2 + 4) {  // one warp (eidx 128..159): the two row sums in a fixed order
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
            if (want_ent) add_fixed(p.acc_ent, static_cast<double>(hsum));
          }
        }
        if (want_imp) {
          // importance: each row's sparse gate vector (gates on the selected
          // experts, 0 elsewhere), column sums as for P
#pragma unroll 1
          for (int g = h; g < ng; g += 2) {
#pragma unroll
            for (int j = 0; j < 16; ++j) tb[j * kTbPitch + r] = 0.0f;
#pragma unroll
            for (int j = 0; j < K; ++j) {
              const int id = st->tk_id[j][r];
              if (id >= g * 16 && id < g * 16 + 16 && id < E)
                tb[(id - g * 16) * kTbPitch + r] = st->tk_p[j][r];
            }
            column_sums(g, p.acc_imp);
          }
        }
        // this tile is done: the CTA that completes the last tile reduces
        named_bar_sync(kBarEpi, kEpiThreads);
        if (eidx == 0) st->flag = atom_add_acq_rel(p.tiles_done, 1) == ntiles - 1;
        named_bar_sync(kBarEpi, kEpiThreads);
        if (st->flag) finalize_all(p, st, eidx, ntiles);
      }
      // release the TMEM buffer to the MMA warp
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&st->tempty[b]);
    }
    if (ntiles == 0 && blockIdx.x == 0) finalize_all(p, st, eidx, 0);
  }

  tc_fence_before();
  __syncthreads();
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
  kern<<<grid, kThreads, smem, stream>>>(x_map, wr_map, args);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace moe
