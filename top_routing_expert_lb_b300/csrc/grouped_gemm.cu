// Ragged grouped GEMM on tcgen05 tensor cores for the expert FFNs.
//
// out_g = A_g * B_g^T for every group g, where the routed groups are the
// experts (rows [offsets[e], offsets[e+1]) of the permuted activations, one
// weight slice per expert) and an optional shared group covers every token
// with the shared-expert weights.  This replaces the per-expert Python loop
// over contiguous slices of the CSDN note's moe_infer (DeepseekV3MoE excerpt)
// with one persistent kernel.  With `swiglu`, the first projection's
// epilogue computes h = SiLU(W1 x) * (W3 x) ("深入理解 MoE" §10.2) from a
// 256-column tile holding 128 gate and the matching 128 up columns.
//
// Design (sm_103a):
//   * 192 threads: warp 0 = TMA producer, warp 1 = TMEM owner + MMA issuer,
//     warps 2-5 = epilogue (warp w reads TMEM lanes 32*(w%4) .. +31).
//   * 128 x BN x 64 tiles per stage, TMA with 128-byte swizzle, kStages-deep
//     mbarrier ring (full: TMA bytes landed; empty: MMAs reading it retired).
//   * Accumulators in TMEM, two buffers of BN fp32 columns so the epilogue of
//     one tile overlaps the main loop of the next.  The epilogue writes 32 x 32
//     output blocks through shared memory with TMA tile stores.
//   * Persistent grid (one CTA per SM).  Tiles are numbered group by group,
//     n-tile major / m-tile minor inside a group, so CTAs running at the same
//     time share a weight tile through L2 (groups with many rows go in blocks
//     of a few n-tiles, m-tile major inside a block, so a wave also shares
//     its A rows instead of sweeping the whole group); row counts come from device
//     offsets (no host synchronisation), ragged m-tiles are masked in the
//     epilogue, and rows past a group's end are computed but never stored.
//   * Every wait is bounded; on expiry the kernel records a timeout in the
//     status word, drains its copies and MMAs, frees TMEM and returns.
//   * Launched with programmatic dependent launch: the prologue (barriers,
//     descriptor prefetch, TMEM) runs while the previous kernel finishes, and
//     griddepcontrol.wait precedes the first read of the row offsets.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdio>

#include "bounds.cuh"
#include "moe_internal.h"
#include "sm100_primitives.cuh"

namespace moe {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreads = 192;
constexpr int kMaxGroups = 257;

struct GemmSmemTail {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t fin;
  uint32_t tmem_base;
  int abort_flag;
  int prefix[kMaxGroups + 1];
  int row0[kMaxGroups];
  int rows[kMaxGroups];
};

// Epilogue output staging.  Each of the four epilogue warps owns kBufs 2 KB
// buffers (two with one CTA per SM, one with two CTAs per SM), each holding one
// block of 32 rows x 32 bf16 columns in the 64-byte-swizzled layout of the
// output tensor maps, and writes a block with one TMA tile store: the block
// reaches L2 as whole 64-byte row segments, where direct stores send 32
// scattered 16-byte pieces per instruction.  On the dense 8192 x 4096 x 28672
// gate/up shape the direct stores alone cost 8 % of the launch.
constexpr int kOutBlockBytes = 32 * 32 * 2;
__host__ __device__ constexpr int out_stage_bytes(int bufs) { return 4 * bufs * kOutBlockBytes; }
constexpr int kOutStageBytes = out_stage_bytes(2);

template <int BN, int kStages, int kOutBufs = 2>
constexpr size_t gemm_smem_bytes() {
  return 1024 + static_cast<size_t>(kStages) * (kBM * kBK * 2 + BN * kBK * 2) +
         out_stage_bytes(kOutBufs) + sizeof(GemmSmemTail);
}

struct OutStage {
  uint32_t buf0;  // shared address of this warp's first buffer (1024-byte aligned)
  uint32_t n;     // blocks issued so far; block n uses buffer n % kBufs
};

// Writes one 32 x 32 output block whose top-left element is (row, col) of the
// tensor behind `map`; lane l holds row l's 32 values as packed bf16 pairs.
// Row l's 16-byte piece i goes to piece i ^ ((l >> 1) & 3) of the row's 64
// bytes in the buffer (the 64-byte swizzle), so each quarter-warp's writes
// cover all 32 banks.
template <int kBufs>
__device__ __forceinline__ void store_block_tma(OutStage& o, const uint32_t (&packed)[16],
                                                const CUtensorMap* map, int col, int64_t row,
                                                int lane) {
  static_assert(kBufs == 1 || kBufs == 2, "one or two buffers per warp");
  const uint32_t buf = o.buf0 + (o.n & static_cast<uint32_t>(kBufs - 1)) *
                                    static_cast<uint32_t>(kOutBlockBytes);
  if (lane == 0) bulk_wait_read<kBufs - 1>();  // the store that used this buffer has read it
  __syncwarp();
  const uint32_t r = buf + static_cast<uint32_t>(lane) * 64u;
  const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
#pragma unroll
  for (uint32_t i = 0; i < 4; ++i)
    st_shared_v4(r + ((i ^ sw) << 4), packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                 packed[4 * i + 3]);
  fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, buf, col, static_cast<int32_t>(row));
    bulk_commit_group();
  }
  ++o.n;
}

struct TileInfo {
  int g;        // group (0 = shared when present)
  int shared;   // 1 for the shared group
  int a_row;    // first A / output row of the tile
  int rows_left;  // valid rows in this tile (may exceed 128)
  int b_row;    // first B row of the tile
  int n;        // n-tile index within the group
  int nk;       // K blocks
};

// Tail tiles.  The last m-tile of a group often holds few rows; a 128-row
// MMA would spend most of its work on rows that are never stored.  When the
// tile has r <= 112 valid rows it is computed transposed instead: D^T = B A^T
// with the weight rows as the MMA's M (128 per half of the B tile) and the
// r token rows, rounded up to 16, as its N.  The staged shared-memory tiles
// are the same (both are K-major, 128-byte swizzled); only the descriptors
// swap roles, and the epilogue reads TMEM lane = output column, TMEM column =
// token row.  Returns that N, or 0 for a normal tile.
template <int BN>
__device__ __forceinline__ int swapped_n(int rows_left, int max_n) {
  if (BN < 128 || rows_left >= kBM) return 0;
  const int n = (rows_left + 15) & ~15;
  return n <= max_n ? n : 0;
}

// Which tails may run transposed.  The tail of a group that also has full
// m-tiles finds its weight tile in L2 (its full tiles read it) and is bound by
// the MMA, where two M = 128 MMAs of N = r cost more than one padded 128-row
// MMA: transposing those tails made the Mixtral layer 33 us slower (1.4 %),
// DeepSeek-V2 9 us.  A group of one m-tile streams its weights and gains, and
// so does every tail of a short reduction (swap_all_tails, set for K <= 1024).
template <typename Tail>
__device__ __forceinline__ bool swap_tail(const Tail* st, const GroupedGemmArgs& p,
                                          const TileInfo& ti) {
  return p.swap_all_tails || ti.rows_left == st->rows[ti.g];
}

template <typename Tail>
__device__ __forceinline__ TileInfo decode_tile(const Tail* st, const GroupedGemmArgs& p, int G,
                                                int tile, int bn, int bm = kBM) {
  int lo = 0, hi = G;  // largest g with prefix[g] <= tile
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (st->prefix[mid] <= tile) lo = mid; else hi = mid;
  }
  TileInfo ti;
  ti.g = lo;
  const int has_shared = p.shared_rows > 0 ? 1 : 0;
  ti.shared = (has_shared && lo == 0) ? 1 : 0;
  const int rows = st->rows[lo];
  const int mt = (rows + bm - 1) / bm;
  const int local = tile - st->prefix[lo];
  const int ncols = ti.shared ? p.n_cols_shared : p.n_cols_routed;
  const int nt = ncols / bn;
  int m;
  if (p.n_block > 1 && rows > p.block_min_rows && nt > 1) {
    // long group: blocks of n_block n-tiles, m-tile major inside a block, so
    // the CTAs of one wave share a few A rows and a few weight tiles instead of
    // sweeping every A row of the group once per n-tile
    const int nb = p.n_block;
    const int b = local / (mt * nb);
    const int n0 = b * nb;
    const int w = min(nb, nt - n0);
    const int j = local - b * (mt * nb);
    m = j / w;
    ti.n = n0 + (j - m * w);
  } else {
    ti.n = local / mt;
    m = local - ti.n * mt;
  }
  ti.a_row = st->row0[lo] + m * bm;
  ti.rows_left = rows - m * bm;
  const int e = lo - has_shared;
  ti.b_row = (ti.shared ? 0 : e * ncols) + ti.n * bn;
  ti.nk = (ti.shared ? p.k_shared : p.k_routed) / kBK;
  return ti;
}

// kRowScale (plain projections only): every routed output row r is multiplied
// by p.row_scale[r] in fp32 before rounding (the combine's gate, applied here).
// kAcc = 2: one CTA per SM, two TMEM accumulators (a tile's epilogue runs
// under the next tile's MMAs).  kAcc = 1: two CTAs per SM with one accumulator
// and a shorter ring each, so that one CTA's MMAs run while the other waits
// for its operands or drains its accumulator.
template <int BN, bool kSwiGLU, int kStages, bool kRowScale = false, int kAcc = 2>
__global__ void __launch_bounds__(kThreads, 3 - kAcc)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA0,
                        const __grid_constant__ CUtensorMap tmA1,
                        const __grid_constant__ CUtensorMap tmB0,
                        const __grid_constant__ CUtensorMap tmB1,
                        const __grid_constant__ CUtensorMap tmO0,
                        const __grid_constant__ CUtensorMap tmO1, const GroupedGemmArgs p) {
  static_assert(!kSwiGLU || BN == 256, "SwiGLU tiles pair 128 gate with 128 up columns");
  constexpr int kABytes = kBM * kBK * 2;
  constexpr int kBBytes = BN * kBK * 2;
  constexpr int kStageBytes = kABytes + kBBytes;
  constexpr uint32_t kTmemCols = kAcc * BN;
  constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, BN);
  static_assert(!(kRowScale && kSwiGLU), "row scaling applies to the plain projection");
  static_assert(kAcc == 1 || kAcc == 2, "one or two accumulators");
  // two CTAs per SM fit one output buffer per epilogue warp each
  constexpr int kOutBufs = kAcc == 2 ? 2 : 1;
  constexpr int kOutBytes = out_stage_bytes(kOutBufs);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  GemmSmemTail* st = reinterpret_cast<GemmSmemTail*>(smem + kStages * kStageBytes + kOutBytes);
  volatile int* abort_flag = &st->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int has_shared = p.shared_rows > 0 ? 1 : 0;
  const int G = p.n_routed + has_shared;
  const int item0 = static_cast<int>(blockIdx.x);
  const int stride = static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&st->full[s], 1);
      mbar_init(&st->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&st->tfull[a], 1);
      mbar_init(&st->tempty[a], 4);
    }
    mbar_init(&st->fin, 1);
    st->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA0);
    tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB0);
    tma_prefetch_desc(&tmB1);
  }
  if (warp == 1) tmem_alloc(&st->tmem_base, kTmemCols);
  // the row offsets and the A rows come from earlier kernels in the stream
  pdl_wait();
  if (threadIdx.x == 0) {
    int acc = 0;
    st->prefix[0] = 0;
    for (int g = 0; g < G; ++g) {
      const int sh = (has_shared && g == 0);
      int r0, rows;
      if (sh) {
        r0 = 0;
        rows = p.shared_rows;
      } else {
        const int e = g - has_shared;
        r0 = p.offsets[e];
        rows = p.offsets[e + 1] - r0;
        if (rows < 0) rows = 0;
      }
      if (p.row_split != 0) {  // whole 256-row blocks, or the rows after them
        const int whole = rows & ~255;
        if (p.row_split == 1) {
          rows = whole;
        } else {
          r0 += whole;
          rows -= whole;
        }
      }
      st->row0[g] = r0;
      st->rows[g] = rows;
      const int ncols = sh ? p.n_cols_shared : p.n_cols_routed;
      const int mt = (rows + kBM - 1) / kBM;
      acc += mt * (ncols / BN);
      st->prefix[g + 1] = acc;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = st->tmem_base;
  const int total = st->prefix[G];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (p.gather_rows == nullptr) {
      // box loads: lane 0 alone runs the ring
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        uint32_t uses[kStages];
#pragma unroll
        for (int s = 0; s < kStages; ++s) uses[s] = 0;
        for (int tile = item0; tile < total && !*abort_flag; tile += stride) {
          const TileInfo ti = decode_tile(st, p, G, tile, BN);
          const CUtensorMap* am = ti.shared ? &tmA1 : &tmA0;
          const CUtensorMap* bm = ti.shared ? &tmB1 : &tmB0;
          bool ok = true;
          for (int kb = 0; kb < ti.nk; ++kb) {
            if (!mbar_wait_bounded(&st->empty[stage], phase ^ 1u, p.timeout_ns, p.status,
                                   abort_flag)) {
              ok = false;
              break;
            }
            uint8_t* sa = smem + stage * kStageBytes;
            mbar_arrive_expect_tx(&st->full[stage], kStageBytes);
            tma_load_2d(sa, am, &st->full[stage], kb * kBK, ti.a_row);
            tma_load_2d(sa + kABytes, bm, &st->full[stage], kb * kBK, ti.b_row);
            uses[stage] += 1;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
        }
        // Drain: the last copy issued into each stage must have landed before
        // the CTA may exit.
#pragma unroll
        for (int s = 0; s < kStages; ++s)
          if (uses[s] > 0)
            mbar_wait_bounded(&st->full[s], (uses[s] - 1u) & 1u, p.timeout_ns, p.status,
                              nullptr);
      }
      __syncwarp();
    } else {
      // Gathered A rows: the whole warp runs the loop (control flow is uniform:
      // lane 0 waits and broadcasts) and every lane issues one 4-row gather per
      // k-block: lane l loads tile rows 4l .. 4l+3, whose token rows it looked
      // up once per tile.  Lane 0 issues the box loads (B, and A of the
      // shared group).
      int stage = 0;
      uint32_t phase = 0;
      uint32_t uses[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) uses[s] = 0;
      for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        int stop = (lane == 0) ? *abort_flag : 0;
        if (__shfl_sync(0xffffffffu, stop, 0)) break;
        const TileInfo ti = decode_tile(st, p, G, tile, BN);
        const CUtensorMap* am = ti.shared ? &tmA1 : &tmA0;
        const CUtensorMap* bm = ti.shared ? &tmB1 : &tmB0;
        const bool gathered = !ti.shared;
        int rr[4] = {0, 0, 0, 0};
        if (gathered) {
          // rows past the tile's valid rows repeat its last valid row (their
          // results are never stored)
          const int nvalid = ti.rows_left < kBM ? ti.rows_left : kBM;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int i = 4 * lane + j;
            rr[j] = __ldg(p.gather_rows + ti.a_row + (i < nvalid ? i : nvalid - 1));
            if (!idx_ok(rr[j], p.gather_limit, p.status)) rr[j] = 0;
          }
        }
        bool ok = true;
        for (int kb = 0; kb < ti.nk; ++kb) {
          int waited = 1;
          if (lane == 0) {
            waited = mbar_wait_bounded(&st->empty[stage], phase ^ 1u, p.timeout_ns, p.status,
                                       abort_flag) ? 1 : 0;
            if (waited) mbar_arrive_expect_tx(&st->full[stage], kStageBytes);
          }
          if (!__shfl_sync(0xffffffffu, waited, 0)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * kStageBytes;
          if (gathered)
            tma_gather4(sa + lane * 4 * (kBK * 2), am, &st->full[stage], kb * kBK, rr[0], rr[1],
                        rr[2], rr[3]);
          else if (lane == 0)
            tma_load_2d(sa, am, &st->full[stage], kb * kBK, ti.a_row);
          if (lane == 0) {
            tma_load_2d(sa + kABytes, bm, &st->full[stage], kb * kBK, ti.b_row);
          }
          uses[stage] += 1;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      // Drain: the last copy issued into each stage must have landed before
      // the CTA may exit.
      if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kStages; ++s)
          if (uses[s] > 0)
            mbar_wait_bounded(&st->full[s], (uses[s] - 1u) & 1u, p.timeout_ns, p.status, nullptr);
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      for (int tile = item0; tile < total && !*abort_flag; tile += stride, ++local) {
        const TileInfo ti = decode_tile(st, p, G, tile, BN);
        const int a = local % kAcc;
        const uint32_t q = static_cast<uint32_t>(local / kAcc);
        if (!mbar_wait_bounded(&st->tempty[a], (q & 1u) ^ 1u, p.timeout_ns, p.status,
                               abort_flag))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * BN);
        const int nsw = swap_tail(st, p, ti) ? swapped_n<BN>(ti.rows_left, p.tail_max_n) : 0;
        const uint32_t idesc_sw = idesc_bf16_f32(kBM, static_cast<uint32_t>(nsw > 0 ? nsw : 16));
        bool ok = true;
        for (int kb = 0; kb < ti.nk; ++kb) {
          if (!mbar_wait_bounded(&st->full[stage], phase, p.timeout_ns, p.status,
                                 abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * kStageBytes);
          const uint32_t sb = sa + kABytes;
          if (nsw == 0) {
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              tc_mma_bf16(d_tmem, smem_desc_sw128(sa + kk * 32), smem_desc_sw128(sb + kk * 32),
                          kIdesc, (kb | kk) != 0 ? 1u : 0u);
            }
          } else {
            // transposed tail: half h of the B tile (weight rows 128h ..) as M,
            // the first nsw rows of the A tile as N; result columns
            // [h * nsw, (h + 1) * nsw) of the accumulator buffer
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
#pragma unroll
              for (int h = 0; h < BN / 128; ++h)
                tc_mma_bf16(d_tmem + static_cast<uint32_t>(h * nsw),
                            smem_desc_sw128(sb + h * (128 * kBK * 2) + kk * 32),
                            smem_desc_sw128(sa + kk * 32), idesc_sw, (kb | kk) != 0 ? 1u : 0u);
            }
          }
          tc_commit(&st->empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&st->tfull[a]);
      }
      // Every MMA issued by this thread must retire before TMEM is freed.
      tc_commit(&st->fin);
      mbar_wait_bounded(&st->fin, 0, p.timeout_ns, p.status, nullptr);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int r_in_tile = quarter * 32 + lane;
    OutStage ostage{smem_u32(smem + kStages * kStageBytes) +
                        static_cast<uint32_t>(quarter * kOutBufs * kOutBlockBytes),
                    0u};
    int local = 0;
    for (int tile = item0; tile < total && !*abort_flag; tile += stride, ++local) {
      const TileInfo ti = decode_tile(st, p, G, tile, BN);
      const int a = local % kAcc;
      const uint32_t q = static_cast<uint32_t>(local / kAcc);
      if (!mbar_wait_bounded(&st->tfull[a], q & 1u, p.timeout_ns, p.status, abort_flag)) break;
      tc_fence_after();
      const int64_t out_rows = ti.shared ? p.out_rows_shared : p.out_rows_routed;
      const int64_t row = static_cast<int64_t>(ti.a_row) + r_in_tile;
      const bool valid = r_in_tile < ti.rows_left && idx_ok(row, out_rows, p.status);
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(a * BN);
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(ti.shared ? p.out_shared
                                                                      : p.out_routed);
      const int64_t ld = ti.shared ? p.ld_shared : p.ld_routed;
      const int nsw = swap_tail(st, p, ti) ? swapped_n<BN>(ti.rows_left, p.tail_max_n) : 0;
      if (nsw > 0) {
        // transposed tail: this thread's TMEM lane is output column r_in_tile
        // of each 128-wide half; TMEM column j of a half is token row j
        __nv_bfloat16* base = out + static_cast<int64_t>(ti.a_row) * ld;
        if constexpr (kSwiGLU) {
          __nv_bfloat16* dst = base + static_cast<int64_t>(ti.n) * 128 + r_in_tile;
#pragma unroll 1
          for (int c = 0; c < nsw; c += 32) {
            float g[32], u[32];
            tmem_ld32(taddr + c, g);
            tmem_ld32(taddr + nsw + c, u);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c + j < ti.rows_left && idx_ok(ti.a_row + c + j, out_rows, p.status))
                dst[static_cast<int64_t>(c + j) * ld] = __float2bfloat16_rn(silu_f32(g[j]) * u[j]);
          }
        } else {
#pragma unroll 1
          for (int h = 0; h < BN / 128; ++h) {
            __nv_bfloat16* dst = base + static_cast<int64_t>(ti.n) * BN + h * 128 + r_in_tile;
#pragma unroll 1
            for (int c = 0; c < nsw; c += 32) {
              float v[32];
              tmem_ld32(taddr + h * nsw + c, v);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (c + j < ti.rows_left && idx_ok(ti.a_row + c + j, out_rows, p.status)) {
                  float o = v[j];
                  if constexpr (kRowScale)
                    if (!ti.shared) o *= __ldg(p.row_scale + ti.a_row + c + j);
                  dst[static_cast<int64_t>(c + j) * ld] = __float2bfloat16_rn(o);
                }
            }
          }
        }
      } else if constexpr (kSwiGLU) {
        __nv_bfloat16* dst = out + row * ld + static_cast<int64_t>(ti.n) * 128;
        // a warp whose 32 rows are all stored writes through the tensor map
        const bool via_tma = __all_sync(0xffffffffu, valid);
        const CUtensorMap* om = ti.shared ? &tmO1 : &tmO0;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float g[32], u[32];
          tmem_ld32(taddr + c * 32, g);
          tmem_ld32(taddr + 128 + c * 32, u);
          tmem_ld_wait();
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            packed[i] = pack_bf16x2(silu_f32(g[2 * i]) * u[2 * i],
                                    silu_f32(g[2 * i + 1]) * u[2 * i + 1]);
          if (via_tma) {
            store_block_tma<kOutBufs>(ostage, packed, om, ti.n * 128 + c * 32, row - lane, lane);
          } else if (valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              d4[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                 packed[4 * i + 3]);
          }
        }
      } else {
        __nv_bfloat16* dst = out + row * ld + static_cast<int64_t>(ti.n) * BN;
        float sc = 1.0f;
        if constexpr (kRowScale) sc = (valid && !ti.shared) ? __ldg(p.row_scale + row) : 1.0f;
        const bool via_tma = __all_sync(0xffffffffu, valid);
        const CUtensorMap* om = ti.shared ? &tmO1 : &tmO0;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(taddr + c * 32, v);
          tmem_ld_wait();
          if constexpr (kRowScale) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= sc;
          }
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) packed[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
          if (via_tma) {
            store_block_tma<kOutBufs>(ostage, packed, om, ti.n * BN + c * 32, row - lane, lane);
          } else if (valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              d4[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                 packed[4 * i + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&st->tempty[a]);
    }
    // every output block written before the CTA (and its buffers) goes away
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  pdl_trigger();  // this CTA's tiles are done: the next kernel's CTAs may come up
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}


// ---------------------------------------------------------------------------
// Paired (2-SM) variant: a cluster of two CTAs computes 256 x 256 tiles with
// tcgen05 cta_group::2.  Each CTA stages its 128 rows of A and its 128 rows of
// B (half of N) per k-block, so one SM moves 32 KB per 64-deep k-block instead
// of 48 KB and the ring holds 6 stages.  The even CTA issues the MMAs; its
// full barrier collects the TMA bytes of both CTAs; each MMA completion
// arrives on the empty / accumulator-full barriers of both CTAs; both CTAs'
// epilogue warps release an accumulator buffer on the even CTA's barrier.
// ---------------------------------------------------------------------------
constexpr int kPairBM = 256;
constexpr int kPairStages = 6;
constexpr int kTileQ = 4;  // tile queue depth (dynamic schedule)
// consumers of a queue slot, counted on the even CTA's q_empty: its MMA warp
// and 4 epilogue warps, the odd CTA's producer and 4 epilogue warps
constexpr int kTileQConsumers = 10;

struct PairSmemTail {
  uint64_t full[kPairStages];
  uint64_t empty[kPairStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t fin;
  uint64_t q_full[kTileQ];
  uint64_t q_empty[kTileQ];
  int qtile[kTileQ];
  uint32_t tmem_base;
  int abort_flag;
  int prefix[kMaxGroups + 1];
  int row0[kMaxGroups];
  int rows[kMaxGroups];
};

constexpr size_t pair_smem_bytes() {
  return 1024 + static_cast<size_t>(kPairStages) * (128 * kBK * 2 + 128 * kBK * 2) +
         kOutStageBytes + sizeof(PairSmemTail);
}

// Dynamic schedule of the pair kernel.  The even CTA's producer takes the
// next tile number from a global counter when it is ready to load it and
// publishes it in slot q of both CTAs' tile queues; every other role reads the
// same sequence from its own queue.  Pairs thus take tiles in the order they
// free up, so the pairs sharing a weight tile start it together however far
// their speeds drift apart.  Consumer side: returns the tile (>= total ends
// the loop) or -1 when the wait ran out.
__device__ __forceinline__ int pair_next_tile(PairSmemTail* st, int q_pos,
                                              const GroupedGemmArgs& p,
                                              volatile int* abort_flag) {
  const int q = q_pos % kTileQ;
  const uint32_t ph = static_cast<uint32_t>(q_pos / kTileQ) & 1u;
  if (!mbar_wait_bounded<true>(&st->q_full[q], ph, p.timeout_ns, p.status, abort_flag))
    return -1;
  const int t = *reinterpret_cast<volatile int*>(&st->qtile[q]);
  mbar_arrive_cluster(mapa_shared(smem_u32(&st->q_empty[q]), 0));
  return t;
}

template <bool kSwiGLU, bool kRowScale = false>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA0,
                             const __grid_constant__ CUtensorMap tmA1,
                             const __grid_constant__ CUtensorMap tmB0,
                             const __grid_constant__ CUtensorMap tmB1,
                             const __grid_constant__ CUtensorMap tmB0h,
                             const __grid_constant__ CUtensorMap tmB1h,
                             const __grid_constant__ CUtensorMap tmO0,
                             const __grid_constant__ CUtensorMap tmO1, const GroupedGemmArgs p) {
  constexpr int BN = 256;                 // N of the pair tile
  constexpr int kABytes = 128 * kBK * 2;  // this CTA's A rows
  constexpr int kBBytes = 128 * kBK * 2;  // this CTA's half of B
  // Half tiles: a group's last tile with at most 128 rows runs as one M = 128
  // pair MMA (64 A rows per CTA).  Its accumulator puts row i of CTA r
  // (tile row 64 r + i) in TMEM lanes i and 64 + i: lanes 0-63 hold the
  // tile's columns 0-127, lanes 64-127 columns 128-255, 128 TMEM columns in
  // all.  With SwiGLU each CTA then loads 64 gate rows and the matching 64 up
  // rows of B (tmB0h / tmB1h: 64-row boxes), so that every lane holds the
  // gate and the up values of the same output columns.
  constexpr uint32_t kIdescHalf = idesc_bf16_f32(128, BN);
  constexpr int kStageBytes = kABytes + kBBytes;
  constexpr uint32_t kTmemCols = 2 * BN;
  constexpr uint32_t kIdesc = idesc_bf16_f32(kPairBM, BN);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  PairSmemTail* st =
      reinterpret_cast<PairSmemTail*>(smem + kPairStages * kStageBytes + kOutStageBytes);
  volatile int* abort_flag = &st->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0 = even CTA (issues the MMAs)
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  const int has_shared = p.shared_rows > 0 ? 1 : 0;
  const int G = p.n_routed + has_shared;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&st->full[s], 1);
      mbar_init(&st->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&st->tfull[a], 1);
      mbar_init(&st->tempty[a], 8);  // 4 epilogue warps in each CTA of the pair
    }
    mbar_init(&st->fin, 1);
    for (int q = 0; q < kTileQ; ++q) {
      mbar_init(&st->q_full[q], 1);
      mbar_init(&st->q_empty[q], kTileQConsumers);
    }
    st->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA0);
    tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB0);
    tma_prefetch_desc(&tmB1);
  }
  if (warp == 1) tmem_alloc_pair(&st->tmem_base, kTmemCols);
  // the row offsets and the A rows come from earlier kernels in the stream
  pdl_wait();
  if (threadIdx.x == 0) {
    int acc = 0;
    st->prefix[0] = 0;
    for (int g = 0; g < G; ++g) {
      const int sh = (has_shared && g == 0);
      int r0, rows;
      if (sh) {
        r0 = 0;
        rows = p.shared_rows;
      } else {
        const int e = g - has_shared;
        r0 = p.offsets[e];
        rows = p.offsets[e + 1] - r0;
        if (rows < 0) rows = 0;
      }
      if (p.row_split != 0) {  // whole 256-row blocks, or the rows after them
        const int whole = rows & ~255;
        if (p.row_split == 1) {
          rows = whole;
        } else {
          r0 += whole;
          rows -= whole;
        }
      }
      st->row0[g] = r0;
      st->rows[g] = rows;
      const int ncols = sh ? p.n_cols_shared : p.n_cols_routed;
      acc += ((rows + kPairBM - 1) / kPairBM) * (ncols / BN);
      st->prefix[g + 1] = acc;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_arrive_wait();  // both CTAs' barriers initialised before any remote signal
  tc_fence_after();
  const uint32_t tmem_base = st->tmem_base;
  const int total = st->prefix[G];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t uses[kPairStages];
#pragma unroll
      for (int s = 0; s < kPairStages; ++s) uses[s] = 0;
      const bool dyn = p.tile_counter != nullptr;
      // Even CTA, dynamic schedule: publishes tile number `t` in queue
      // position `pos` of both CTAs once every reader has freed that slot.
      auto publish = [&](int pos, int t) -> bool {
        const int q = pos % kTileQ;
        const uint32_t ph = static_cast<uint32_t>(pos / kTileQ) & 1u;
        if (!mbar_wait_bounded<true>(&st->q_empty[q], ph ^ 1u, p.timeout_ns, p.status,
                                     abort_flag))
          return false;
        st->qtile[q] = t;
        st_shared_cluster_u32(mapa_shared(smem_u32(&st->qtile[q]), 1), static_cast<uint32_t>(t));
        mbar_arrive_cluster(mapa_shared(smem_u32(&st->q_full[q]), 0));
        mbar_arrive_cluster(mapa_shared(smem_u32(&st->q_full[q]), 1));
        return true;
      };
      int cur = 0;  // even CTA, dynamic: the tile published at q_pos
      if (dyn && leader) {
        cur = atomicAdd(p.tile_counter, 1);
        if (!publish(0, cur)) cur = total;
      }
      for (int tile = pair, q_pos = 0; !*abort_flag; tile += npairs, ++q_pos) {
        if (dyn) {
          if (leader) {
            tile = cur;
          } else if ((tile = pair_next_tile(st, q_pos, p, abort_flag)) < 0) {
            break;
          }
        }
        if (tile >= total) break;
        // the next tile number is taken now and published during this tile's
        // first k-blocks, so neither CTA waits for it at the tile boundary
        int next = 0;
        if (dyn && leader) next = atomicAdd(p.tile_counter, 1);
        bool published = !(dyn && leader);
        const TileInfo ti = decode_tile(st, p, G, tile, BN, kPairBM);
        const CUtensorMap* am = ti.shared ? &tmA1 : &tmA0;
        const CUtensorMap* bm = ti.shared ? &tmB1 : &tmB0;
        const CUtensorMap* bmh = ti.shared ? &tmB1h : &tmB0h;
        const bool half = (p.half_tiles && ti.rows_left <= 128);
        const int a_row = ti.a_row + static_cast<int>(rank) * (half ? 64 : 128);
        const int b_row = ti.b_row + static_cast<int>(rank) * 128;
        // half SwiGLU tile: this CTA's 64 gate rows, then the matching 64 up rows
        const int g_row = ti.b_row + static_cast<int>(rank) * 64;
        bool ok = true;
        for (int kb = 0; kb < ti.nk; ++kb) {
          if (!mbar_wait_bounded(&st->empty[stage], phase ^ 1u, p.timeout_ns, p.status,
                                 abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * kStageBytes;
          const uint32_t full_leader = mapa_shared(smem_u32(&st->full[stage]), 0);
          if (leader) mbar_arrive_expect_tx(&st->full[stage], 2 * kStageBytes);
          tma_load_2d_pair(sa, am, full_leader, kb * kBK, a_row);
          if (kSwiGLU && half) {
            tma_load_2d_pair(sa + kABytes, bmh, full_leader, kb * kBK, g_row);
            tma_load_2d_pair(sa + kABytes + kBBytes / 2, bmh, full_leader, kb * kBK,
                             g_row + 128);
          } else {
            tma_load_2d_pair(sa + kABytes, bm, full_leader, kb * kBK, b_row);
          }
          uses[stage] += 1;
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
          if (!published && (kb == 1 || kb == ti.nk - 1)) {
            if (!publish(q_pos + 1, next)) {
              ok = false;
              break;
            }
            published = true;
          }
        }
        if (ok && !published) ok = publish(q_pos + 1, next);
        if (!ok) break;
        cur = next;
        if (!ok) break;
      }
      // Drain (even CTA): its full barriers count the bytes of both CTAs, so
      // this covers every copy of the pair; the odd CTA stays alive through
      // the final cluster barrier.
      if (leader) {
#pragma unroll
        for (int s = 0; s < kPairStages; ++s)
          if (uses[s] > 0)
            mbar_wait_bounded(&st->full[s], (uses[s] - 1u) & 1u, p.timeout_ns, p.status,
                              nullptr);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      const bool dyn = p.tile_counter != nullptr;
      for (int tile = pair; !*abort_flag; tile += npairs, ++local) {
        if (dyn && (tile = pair_next_tile(st, local, p, abort_flag)) < 0) break;
        if (tile >= total) break;
        const TileInfo ti = decode_tile(st, p, G, tile, BN, kPairBM);
        const int a = local & 1;
        const uint32_t q = static_cast<uint32_t>(local >> 1);
        if (!mbar_wait_bounded<true>(&st->tempty[a], (q & 1u) ^ 1u, p.timeout_ns, p.status,
                                     abort_flag))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * BN);
        const uint32_t idesc = (p.half_tiles && ti.rows_left <= 128) ? kIdescHalf : kIdesc;
        bool ok = true;
        for (int kb = 0; kb < ti.nk; ++kb) {
          if (!mbar_wait_bounded(&st->full[stage], phase, p.timeout_ns, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * kStageBytes);
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            tc_mma_bf16_pair(d_tmem, smem_desc_sw128(sa + kk * 32),
                             smem_desc_sw128(sb + kk * 32), idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit_pair_mc(&st->empty[stage], 0x3);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(&st->tfull[a], 0x3);
      }
      // every pair MMA must retire before either CTA frees its TMEM
      tc_commit_pair_mc(&st->fin, 0x1);
      mbar_wait_bounded(&st->fin, 0, p.timeout_ns, p.status, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int r_in_half = quarter * 32 + lane;
    const uint32_t tempty_leader0 = mapa_shared(smem_u32(&st->tempty[0]), 0);
    const uint32_t tempty_leader1 = mapa_shared(smem_u32(&st->tempty[1]), 0);
    OutStage ostage{smem_u32(smem + kPairStages * kStageBytes) +
                        static_cast<uint32_t>(quarter * 2 * kOutBlockBytes),
                    0u};
    int local = 0;
    const bool dyn = p.tile_counter != nullptr;
    for (int tile = pair; !*abort_flag; tile += npairs, ++local) {
      if (dyn) {
        int t = 0;
        if (lane == 0) t = pair_next_tile(st, local, p, abort_flag);
        tile = __shfl_sync(0xffffffffu, t, 0);
        if (tile < 0) break;
      }
      if (tile >= total) break;
      const TileInfo ti = decode_tile(st, p, G, tile, BN, kPairBM);
      const int a = local & 1;
      const uint32_t q = static_cast<uint32_t>(local >> 1);
      if (!mbar_wait_bounded(&st->tfull[a], q & 1u, p.timeout_ns, p.status, abort_flag)) break;
      tc_fence_after();
      // full tile: TMEM lane = this CTA's tile row; half tile: lanes i and
      // 64 + i hold row i, columns [0, 128) and [128, 256) of the tile
      const bool half = (p.half_tiles && ti.rows_left <= 128);
      const int r_in_tile = static_cast<int>(rank) * (half ? 64 : 128) +
                            (half ? (r_in_half & 63) : r_in_half);
      const int col_half = half ? (r_in_half >> 6) : 0;
      const int64_t row = static_cast<int64_t>(ti.a_row) + r_in_tile;
      const bool valid = r_in_tile < ti.rows_left &&
                         idx_ok(row, ti.shared ? p.out_rows_shared : p.out_rows_routed, p.status);
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(a * BN);
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(ti.shared ? p.out_shared
                                                                      : p.out_routed);
      const int64_t ld = ti.shared ? p.ld_shared : p.ld_routed;
      // a warp's 32 lanes hold 32 consecutive rows of one column range; when
      // all of them are stored the warp writes through the tensor map
      const bool via_tma = __all_sync(0xffffffffu, valid);
      const CUtensorMap* om = ti.shared ? &tmO1 : &tmO0;
      if constexpr (kSwiGLU) {
        // full: gate in TMEM columns [0, 128), up in [128, 256); half: this
        // lane's 64 output columns, gate in [0, 64), up in [64, 128)
        __nv_bfloat16* dst =
            out + row * ld + static_cast<int64_t>(ti.n) * 128 + static_cast<int64_t>(col_half) * 64;
        const int nc = half ? 2 : 4;
        const uint32_t up = half ? 64u : 128u;
#pragma unroll 1
        for (int c = 0; c < nc; ++c) {
          float g[32], u[32];
          tmem_ld32(taddr + c * 32, g);
          tmem_ld32(taddr + up + c * 32, u);
          tmem_ld_wait();
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            packed[i] = pack_bf16x2(silu_f32(g[2 * i]) * u[2 * i],
                                    silu_f32(g[2 * i + 1]) * u[2 * i + 1]);
          if (via_tma) {
            store_block_tma<2>(ostage, packed, om, ti.n * 128 + col_half * 64 + c * 32,
                               row - lane, lane);
          } else if (valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              d4[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                 packed[4 * i + 3]);
          }
        }
      } else {
        __nv_bfloat16* dst = out + row * ld + static_cast<int64_t>(ti.n) * BN +
                             static_cast<int64_t>(col_half) * 128;
        float sc = 1.0f;
        if constexpr (kRowScale) sc = (valid && !ti.shared) ? __ldg(p.row_scale + row) : 1.0f;
        const int nc = half ? 4 : BN / 32;
#pragma unroll 1
        for (int c = 0; c < nc; ++c) {
          float v[32];
          tmem_ld32(taddr + c * 32, v);
          tmem_ld_wait();
          if constexpr (kRowScale) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= sc;
          }
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) packed[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
          if (via_tma) {
            store_block_tma<2>(ostage, packed, om, ti.n * BN + col_half * 128 + c * 32,
                               row - lane, lane);
          } else if (valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              d4[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                 packed[4 * i + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(a ? tempty_leader1 : tempty_leader0);
    }
    // every output block written before the CTA (and its buffers) goes away
    if (lane == 0) bulk_wait_all();
  }

  // Both CTAs stay until the even CTA's MMAs and the odd CTA's copies are done.
  tc_fence_before();
  __syncthreads();
  cluster_arrive_wait();
  pdl_trigger();  // this pair's tiles are done: the next kernel's CTAs may come up
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
  // The last CTA out puts the tile counter back to zero for the next launch
  // (every CTA has taken its last tile before it counts itself out).
  if (p.tile_counter != nullptr && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.tile_counter + 1, 1) == static_cast<int>(gridDim.x) - 1) {
      atomicExch(p.tile_counter, 0);
      atomicExch(p.tile_counter + 1, 0);
    }
  }
}

template <bool kSwiGLU, bool kRowScale = false>
int launch_pair_impl(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0,
                     const CUtensorMap& b1, const CUtensorMap& b0h, const CUtensorMap& b1h,
                     const CUtensorMap& o0, const CUtensorMap& o1, const GroupedGemmArgs& args,
                     int num_sms, cudaStream_t stream) {
  constexpr size_t smem = pair_smem_bytes();
  static_assert(smem <= 227 * 1024, "shared memory budget");
  auto kern = grouped_gemm_pair_kernel<kSwiGLU, kRowScale>;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return -3;
    attr_set = true;
  }
  if (launch_kernel(kern, dim3(static_cast<unsigned>(num_sms & ~1)), dim3(kThreads), smem, stream,
                    args.pdl != 0, 2u, a0, a1, b0, b1, b0h, b1h, o0, o1, args) != cudaSuccess)
    return -3;
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

template <int BN, bool kSwiGLU, int kStages, bool kRowScale = false, int kAcc = 2>
int launch_impl(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0,
                const CUtensorMap& b1, const CUtensorMap& o0, const CUtensorMap& o1,
                const GroupedGemmArgs& args, int num_sms, cudaStream_t stream) {
  constexpr size_t smem = gemm_smem_bytes<BN, kStages, kAcc == 2 ? 2 : 1>();
  static_assert(smem <= 227 * 1024, "shared memory budget");
  // two CTAs per SM: both blocks and the 1 KB each reserves fit the SM's 228 KB
  static_assert(kAcc == 2 || 2 * (smem + 1024) <= 228 * 1024, "two CTAs per SM");
  auto kern = grouped_gemm_kernel<BN, kSwiGLU, kStages, kRowScale, kAcc>;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return -3;
    attr_set = true;
  }
  if (launch_kernel(kern, dim3(static_cast<unsigned>(num_sms * (3 - kAcc))), dim3(kThreads), smem,
                    stream, args.pdl != 0, 1u, a0, a1, b0, b1, o0, o1, args) != cudaSuccess)
    return -3;
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

}  // namespace

bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows) {
  auto encode = get_encode_fn();
  if (encode == nullptr || rows == 0 || cols == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_out_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols) {
  auto encode = get_encode_fn();
  if (encode == nullptr || rows == 0 || cols == 0 || cols % 8 != 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int launch_grouped_gemm(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0,
                        const CUtensorMap& b1, const CUtensorMap& o0, const CUtensorMap& o1,
                        const GroupedGemmArgs& args, bool swiglu, int bn, bool paired,
                        int num_sms, cudaStream_t stream, const CUtensorMap* b0h,
                        const CUtensorMap* b1h) {
  if (args.n_routed + (args.shared_rows > 0 ? 1 : 0) > kMaxGroups) return -2;
  const bool scale = args.row_scale != nullptr;
  if (scale && swiglu) return -2;
  if (paired) {
    if (bn != 256 || num_sms < 2) return -2;
    if (scale) return launch_pair_impl<false, true>(a0, a1, b0, b1, b0, b1, o0, o1, args, num_sms, stream);
    if (!swiglu) return launch_pair_impl<false>(a0, a1, b0, b1, b0, b1, o0, o1, args, num_sms, stream);
    if (b0h == nullptr || b1h == nullptr) return -2;  // half tiles need 64-row B boxes
    return launch_pair_impl<true>(a0, a1, b0, b1, *b0h, *b1h, o0, o1, args, num_sms, stream);
  }
  if (args.two_per_sm && bn == 256 && !scale) {
    if (swiglu) return launch_impl<256, true, 2, false, 1>(a0, a1, b0, b1, o0, o1, args, num_sms, stream);
    return launch_impl<256, false, 2, false, 1>(a0, a1, b0, b1, o0, o1, args, num_sms, stream);
  }
  if (swiglu) {
    if (bn != 256) return -2;
    return launch_impl<256, true, 4>(a0, a1, b0, b1, o0, o1, args, num_sms, stream);
  }
  if (scale) {
    switch (bn) {
      case 256: return launch_impl<256, false, 4, true>(a0, a1, b0, b1, o0, o1, args, num_sms, stream);
      case 128: return launch_impl<128, false, 6, true>(a0, a1, b0, b1, o0, o1, args, num_sms, stream);
      case 64: return launch_impl<64, false, 8, true>(a0, a1, b0, b1, o0, o1, args, num_sms, stream);
      default: return -2;
    }
  }
  switch (bn) {
    case 256: return launch_impl<256, false, 4>(a0, a1, b0, b1, o0, o1, args, num_sms, stream);
    case 128: return launch_impl<128, false, 6>(a0, a1, b0, b1, o0, o1, args, num_sms, stream);
    case 64: return launch_impl<64, false, 8>(a0, a1, b0, b1, o0, o1, args, num_sms, stream);
    default: return -2;
  }
}

}  // namespace moe
