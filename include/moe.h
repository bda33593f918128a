/*
 * moe.h - C ABI of libmoe_b300.so: the forward pass of one top-k routed
 * Mixture-of-Experts FFN layer on one NVIDIA B300 (sm_103a).
 *
 * The layer ("MoE：条件计算与路由", llm-knowledge-atlas notes 04-04, core formula
 * and §7 Eqs.(1)-(3)):
 *
 *     y(x) = sum_{e in S(x)} g~_e(x) E_e(x)  +  Ys(x)
 *     p    = softmax(W_r x + o)              router, max-subtracted softmax
 *     S    = TopK_e(p_e + b_e, k)            b_e: optional ALF-LB selection bias
 *     g~_e = p_e / sum_{j in S} p_j          renormalised gates (unbiased p)
 *     E_e(x) = W2_e (SiLU(W1_e x) * W3_e x)  SwiGLU expert ("深入理解 MoE" §10.2)
 *     Ys   = shared experts, width n_shared*M, gate 1 (CSDN note, DeepseekV3MoE)
 *
 * with optional capacity C = ceil(c k T / E) ("MoE：条件计算与路由" §3), pairs
 * beyond C per expert dropped in token-major (t, slot) order, and the side
 * outputs f_e, P_e, L_bal = lambda E sum_e f_e P_e and the z-loss
 * L_z = (1/T) sum_t (log sum_e exp l_te)^2 ("MOE大模型对比篇" §2.1, §2.2).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller, unless a
 *     parameter says "host".  The library never allocates device memory; the
 *     scratch it needs is the caller's workspace (moe_workspace_size).
 *   - bf16 tensors are passed as uint16_t bit patterns.  Layouts are
 *     row-major; weights are [out][in] (nn.Linear layout, K-major).
 *   - Every call enqueues work on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and returns without synchronising, except where stated.
 *   - Every device pointer must be 16-byte aligned; the workspace 256-byte.
 *   - Return value: MOE_OK or a negative MOE_ERR_* code.  Arguments are checked
 *     on the host before anything is enqueued; on an error nothing is
 *     enqueued.  MOE_ERR_CUDA reports a failed launch.  Device-side waits are
 *     bounded; a wait that runs out records MOE_ERR_TIMEOUT in the workspace,
 *     read back by moe_check_status.
 *   - Determinism: for fixed inputs every output is bitwise reproducible (all
 *     reductions run in a fixed order; no floating-point atomics).
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)  /* null/misaligned pointer, bad size, k > E ...  */
#define MOE_ERR_UNSUPPORTED (-2)  /* shape outside the supported limits below       */
#define MOE_ERR_CUDA (-3)         /* a CUDA runtime/driver call failed              */
#define MOE_ERR_TIMEOUT (-4)      /* a bounded device wait ran out                  */
#define MOE_ERR_WORKSPACE (-5)    /* workspace smaller than moe_workspace_size      */
#define MOE_ERR_BOUNDS (-6)       /* a device index out of range; reported only by a
                                     library built with -DMOE_BOUNDS_CHECK, which
                                     checks every data-dependent index and skips
                                     the access instead of faulting               */

/* Supported limits (MOE_ERR_UNSUPPORTED outside them):
 *   1 <= E <= 256;  0 <= k <= min(E, 8);  0 <= T <= 2^24;  d % 64 == 0,
 *   64 <= d <= 16384;  M % 128 == 0, 128 <= M <= 32768;  0 <= n_shared <= 8.  */
#define MOE_MAX_EXPERTS 256
#define MOE_MAX_TOPK 8

/* Routing variants, set in moe_shape_t.flags:
 *   MOE_FLAG_SIGMOID    scores s_e = sigmoid(l_e), each expert on its own,
 *                       instead of the softmax (CSDN note, §9: DeepSeek-V3
 *                       moved the gate from softmax to sigmoid); selection on
 *                       s_e + b_e; P_e is the mean score; the z-loss still
 *                       uses log sum exp of the logits.
 *   MOE_FLAG_NO_RENORM  gates are the selected scores themselves, not divided
 *                       by their sum ("MoE：条件计算与路由" §7).
 *   MOE_FLAG_PRIORITY_CAPACITY
 *                       with a capacity, an over-full expert keeps the C
 *                       pairs with the largest unbiased scores (its softmax
 *                       probability, or sigmoid score, for that token; equal
 *                       scores in token-major (t, slot) order) instead of the
 *                       first C in token order ("深入理解 MoE" §4.2.2, the
 *                       capacity-bounded router).  Kept rows stay in (t, slot)
 *                       order.  Honoured by moe_layer_forward(_host); the
 *                       routers ignore it; moe_permute, which receives no
 *                       scores, returns MOE_ERR_UNSUPPORTED with it.
 *   MOE_FLAG_EXPERT_CHOICE
 *                       expert-choice routing ("深入理解 MoE" §9.2): every
 *                       expert takes the r tokens with the largest scores
 *                       (equal scores to the lower token), r = min(T,
 *                       ceil(c k T / E)) with c <= 0 read as 1, so that c = 1
 *                       computes as many rows as token-choice top-k; the
 *                       gate of a row is its score.  Only the moe_ec_* entry
 *                       points accept it, and they require it; the token-
 *                       choice entry points return MOE_ERR_INVALID_ARG.
 *                       Combining it with MOE_FLAG_PRIORITY_CAPACITY is
 *                       MOE_ERR_UNSUPPORTED; MOE_FLAG_NO_RENORM changes
 *                       nothing (expert-choice gates are never renormalised).*/
#define MOE_FLAG_SIGMOID 1u
#define MOE_FLAG_NO_RENORM 2u
#define MOE_FLAG_PRIORITY_CAPACITY 4u
#define MOE_FLAG_EXPERT_CHOICE 8u

/* How the expert GEMMs and the layer are scheduled: tuning choices, not part
 * of the layer's definition.  Every field at zero selects the measured-
 * fastest default; every choice gives parity-tested results (most of them
 * bit-identical to the default).  Invalid values -> MOE_ERR_INVALID_ARG.
 *   gemm1_tile      gate/up projection tiles.  0 or 128: single-CTA 128 x 256
 *                   tiles; 256: CTA-pair 256 x 256 tiles (then the down
 *                   projection too, unless gemm2_tile is 128)
 *   gemm2_tile      down projection tiles.  0: CTA pairs when d % 256 == 0,
 *                   E <= 16 and experts average >= 512 rows (or gemm1_tile is
 *                   256), else
 *                   single-CTA 128 x BN (BN = 256, 128 or 64 by d); 128:
 *                   single-CTA tiles; 256: CTA pairs (needs d % 256 == 0)
 *   tile_order      CTA-pair launches.  0: tiles from a counter in the
 *                   workspace when K >= 4096, else round-robin; 1: round-robin
 *                   throughout; 2: counter throughout
 *   tail_max_n      single-CTA tiles: a group's only m-tile with r valid rows
 *                   runs transposed (weights as the MMA's M) when r rounded up
 *                   to 16 is at most this.  0: 112; < 0: never; 16..128
 *   n_block         tile order inside a group with more than block_min_rows
 *                   rows: blocks of n_block n-tiles, m-tile major inside a
 *                   block.  0: 8, or 4 for a single-CTA gate/up projection
 *                   of at least 64 n-tiles (2M >= 16384); 1: n-tile major,
 *                   m-tile minor throughout
 *   block_min_rows  0: 2048, or 512 for such a gate/up projection
 *   options         MOE_TUNE_* bits:
 *     MOE_TUNE_NO_HALF_TILES    CTA-pair launches pad a group's last tile of at
 *                               most 128 rows to a 256-row tile instead of one
 *                               M = 128 pair MMA (64 rows per CTA)
 *     MOE_TUNE_GEMM1_SPLIT      gate/up projection: whole 256-row blocks on CTA
 *                               pairs, the remaining rows on single CTAs (two
 *                               launches)
 *     MOE_TUNE_FUSED_GATHER     moe_layer_forward / moe_ec_layer_forward: the
 *                               gate/up projection gathers token rows itself
 *                               (TMA 4-row gathers), no x_perm; not with
 *                               gemm1_tile = 256
 *     MOE_TUNE_GATE_IN_EPILOGUE moe_layer_forward / moe_ec_layer_forward: the
 *                               down projection's epilogue scales each routed
 *                               row by its gate (fp32, before rounding) and
 *                               the combine only adds rows, in the same order
 *     MOE_TUNE_SWAP_ALL_TAILS   single-CTA tiles: the last m-tile of every
 *                               group may run transposed (by tail_max_n), not
 *                               only a group's only m-tile (the default for a
 *                               projection with K <= 1024)
 *     MOE_TUNE_TWO_CTAS_PER_SM  single-CTA expert GEMMs with 256-column tiles run
 *                               two CTAs per SM, each with a 2-stage ring and
 *                               one TMEM accumulator (the default only for a
 *                               down projection with M <= 2048 over experts
 *                               averaging fewer than 512 rows)
 *     MOE_TUNE_NO_PDL           launch the router, scatter, expert GEMMs and
 *                               combine without programmatic dependent launch
 *                               (by default each of them may start while the
 *                               kernel before it in the stream finishes, and
 *                               waits for that kernel before reading its
 *                               outputs; results are the same either way)
 *   wait_timeout_ns limit of this call's bounded device waits; 0: the
 *                   process-wide limit (moe_set_wait_timeout_ns)             */
#define MOE_TUNE_NO_HALF_TILES 1u
#define MOE_TUNE_GEMM1_SPLIT 2u
#define MOE_TUNE_FUSED_GATHER 4u
#define MOE_TUNE_GATE_IN_EPILOGUE 8u
#define MOE_TUNE_SWAP_ALL_TAILS 16u
#define MOE_TUNE_TWO_CTAS_PER_SM 32u
#define MOE_TUNE_NO_PDL 64u
typedef struct moe_tuning {
    int32_t gemm1_tile, gemm2_tile, tile_order, tail_max_n, n_block, block_min_rows;
    uint32_t options;
    uint32_t reserved;  /* must be 0 */
    uint64_t wait_timeout_ns;
} moe_tuning_t;

/* Layer shape.
 *   T  tokens;  d  model width;  M  expert intermediate width;
 *   E  routed experts;  k  experts per token;  n_shared  shared experts,
 *      fused into one SwiGLU MLP of width Ms = n_shared * M;
 *   capacity_factor  c; <= 0 means dropless, otherwise C = ceil(c*k*T/E)
 *      evaluated in double precision;
 *   balance_coef  lambda of the balance loss (0.01 is customary);
 *   flags  routing variants, a combination of the MOE_FLAG_* bits above;
 *   tuning  scheduling choices (all zero: the defaults), see moe_tuning_t.
 * A zero-initialised struct with the first eight fields set is a complete
 * description; the library reads nothing from the environment.              */
typedef struct moe_shape {
    int32_t T, d, M, E, k, n_shared;
    float capacity_factor;
    float balance_coef;
    uint32_t flags;
    uint32_t reserved;  /* must be 0 */
    moe_tuning_t tuning;
} moe_shape_t;

/* Error text for a MOE_* code (static string, never NULL). */
const char *moe_error_string(int code);

/* Bytes of device workspace every other entry point needs for this shape
 * (written to *bytes, a host pointer).  Pure host computation.  Zero the
 * workspace once before its first use (e.g. cudaMemset): it holds a status
 * word and counters that must start at zero; every call leaves them at zero
 * again, so later calls need no clearing.                                    */
int moe_workspace_size(const moe_shape_t *shape, size_t *bytes);

/* Expert capacity C (host pointer *C): ceil(c*k*T/E), or -1 when dropless.  */
int moe_capacity(const moe_shape_t *shape, int64_t *C);

/* Upper bound R_max on routed rows: T*k dropless, else min(T*k, E*C); E*r
 * with MOE_FLAG_EXPERT_CHOICE.                                               */
int moe_max_rows(const moe_shape_t *shape, int64_t *rows);

/* Pack canonical SwiGLU gate/up weights for the grouped GEMM.
 *   w1, w3  [G][Mw][d] bf16 (gate = W1, up = W3; G groups of width Mw)
 *   w13     [G][2*Mw][d] bf16 output: within each group, row block
 *           [256 j, 256 j + 128) holds W1 rows [128 j, 128 j + 128) and
 *           [256 j + 128, 256 j + 256) holds W3 rows [128 j, 128 j + 128),
 *           so one 256-row tile of w13 yields 128 columns of h.
 * Mw % 128 == 0, d % 64 == 0.  One-time preparation, not part of the layer.  */
int moe_pack_w13(int32_t G, int32_t Mw, int32_t d, const uint16_t *w1, const uint16_t *w3,
                 uint16_t *w13, void *stream);

/* Router ("MoE：条件计算与路由" router and ALF-LB; §7 Eqs.(1)-(2); z-loss
 * "MOE大模型对比篇" §2.2).
 *   x           [T][d] bf16 tokens
 *   w_router    [E][d] bf16 router projection W_r
 *   logit_offset [E] fp32 or NULL: added to every token's logits (router bias)
 *   sel_bias    [E] fp32 or NULL: ALF-LB bias b_e, added to the softmax
 *               probabilities for selection only
 * Outputs (device):
 *   ids    [T][k] int32  selected experts, descending key p_e + b_e; equal keys
 *                        go to the lower expert index
 *   gates  [T][k] fp32   p_e / sum_{j in S} p_j (unbiased p)
 *   counts [E]    int32  n_e, pairs routed to e (before any capacity cut)
 *   f, P   [E]    fp32   n_e / (k T) and (1/T) sum_t p_e(t)
 *   bal_loss, z_loss [1] fp32  lambda E sum f P  and  (1/T) sum_t lse_t^2
 * Logits are accumulated in fp32 from bf16 products; softmax in fp32.        */
int moe_route(const moe_shape_t *shape, const uint16_t *x, const uint16_t *w_router,
              const float *logit_offset, const float *sel_bias, int32_t *ids, float *gates,
              int32_t *counts, float *f, float *P, float *bal_loss, float *z_loss, void *ws,
              size_t ws_bytes, void *stream);

/* Router with every output in one struct, including two optional side
 * outputs (NULL = not computed):
 *   importance [E]  sum over tokens of each expert's gate (before capacity),
 *   importance_cv2 [1]  (population std / mean of importance)^2 over experts
 *                   (CSDN note, balancing expert utilization:
 *                   L_importance = w * CV(Importance)^2; w is the caller's),
 *   entropy_mean [1]  mean over tokens of -sum_e q_e log q_e of the router
 *                   distribution q (softmax; normalised sigmoid scores with
 *                   MOE_FLAG_SIGMOID) ("MoE：条件计算与路由" §9).
 * The other fields are those of moe_route (ids/gates may be NULL when k = 0).*/
typedef struct moe_route_out {
    int32_t *ids;
    float *gates;
    int32_t *counts;
    float *f;
    float *P;
    float *bal_loss;
    float *z_loss;
    float *importance;
    float *importance_cv2;
    float *entropy_mean;
} moe_route_out_t;
int moe_route_ex(const moe_shape_t *shape, const uint16_t *x, const uint16_t *w_router,
                 const float *logit_offset, const float *sel_bias, const moe_route_out_t *out,
                 void *ws, size_t ws_bytes, void *stream);

/* ALF-LB selection-bias update ("MoE：条件计算与路由", ALF-LB section: the bias
 * of an overloaded expert decreases, of an underloaded one increases, at rate
 * gamma, outside any backward pass).  The pages give no formula; implemented:
 *     b_e <- b_e + gamma * sign(k T / E - n_e),   sign(0) = 0,
 * in place on sel_bias [E] fp32 (device), from counts [E] int32 (device, the
 * counts output of moe_route for the same shape).  gamma >= 0.             */
int moe_alf_bias_update(const moe_shape_t *shape, const int32_t *counts, float gamma,
                        float *sel_bias, void *stream);

/* Dispatch: capacity cut and permutation into expert-contiguous rows (CSDN
 * note, moe_infer's histogram + argsort; capacity "MoE：条件计算与路由" §3).
 *   x    [T][d] bf16;  ids [T][k] int32 (each in [0, E))
 * Outputs (device):
 *   offsets   [E+1] int32  offsets[e] = first row of expert e; offsets[E] = R
 *   slot_row  [T][k] int32 row of pair (t,s) in x_perm, or -1 if dropped
 *   row_token [R_max] int32 token of each row (entries >= R untouched)
 *   drop_mask [T][k] uint8 1 where the pair was dropped
 *   x_perm    [R_max][d] bf16, row r = x[row_token[r]]
 * Rows of one expert are ordered by (t, s) ascending; a pair is kept iff
 * fewer than C earlier pairs (token-major) went to its expert.  Bit-exact and
 * deterministic.  Ids outside [0, E) are undefined behaviour.                */
int moe_permute(const moe_shape_t *shape, const uint16_t *x, const int32_t *ids,
                int32_t *offsets, int32_t *slot_row, int32_t *row_token, uint8_t *drop_mask,
                uint16_t *x_perm, void *ws, size_t ws_bytes, void *stream);

/* Grouped SwiGLU expert FFNs plus the shared experts ("深入理解 MoE" §10.2;
 * CSDN note, DeepseekV3MoE experts loop and shared_experts).
 *   x_perm   [R_max][d] bf16 rows, expert e owning [offsets[e], offsets[e+1])
 *   offsets  [E+1] int32 (device), non-decreasing, offsets[E] <= R_max
 *   w13      [E][2M][d] bf16, packed by moe_pack_w13 (G = E, Mw = M)
 *   w2       [E][d][M] bf16
 *   y_perm   [R_max][d] bf16 output, row r = E_e(x_perm[r])
 *   x        [T][d] bf16 tokens (read only when n_shared > 0)
 *   w13_shared [2Ms][d] bf16 packed (G = 1, Mw = Ms), w2_shared [d][Ms] bf16,
 *   y_shared [T][d] bf16 output Ys(x); all three NULL when n_shared == 0
 * bf16 tensor-core products accumulated in fp32; h = SiLU(g) * u rounded to
 * bf16 between the two projections; outputs rounded to bf16.                 */
int moe_grouped_ffn(const moe_shape_t *shape, const uint16_t *x_perm, const int32_t *offsets,
                    const uint16_t *w13, const uint16_t *w2, uint16_t *y_perm,
                    const uint16_t *x, const uint16_t *w13_shared, const uint16_t *w2_shared,
                    uint16_t *y_shared, void *ws, size_t ws_bytes, void *stream);

/* Combine ("MoE：条件计算与路由" §7 Eq.(3); CSDN note, moe_infer's un-permute
 * and weighted sum):  y[t] = sum_{s: slot_row[t][s] >= 0} gates[t][s] *
 * y_perm[slot_row[t][s]] + y_shared[t], accumulated in fp32 in slot order,
 * stored as bf16.  Dropped pairs add nothing; gates are not renormalised.
 *   y_perm [R_max][d] bf16; slot_row [T][k] int32; gates [T][k] fp32;
 *   y_shared [T][d] bf16 or NULL; y [T][d] bf16 output.                        */
int moe_combine(const moe_shape_t *shape, const uint16_t *y_perm, const int32_t *slot_row,
                const float *gates, const uint16_t *y_shared, uint16_t *y, void *stream);

/* The whole layer: route -> permute -> grouped FFN (+ shared) -> combine, all
 * on `stream`, no host synchronisation.  Arguments as in the calls above;
 * w13_shared / w2_shared are NULL when n_shared == 0.  Outputs: y [T][d] bf16,
 * ids, gates, counts, drop_mask [T][k] uint8, f, P, bal_loss, z_loss.
 * Intermediate rows live in the workspace.                                   */
int moe_layer_forward(const moe_shape_t *shape, const uint16_t *x, const uint16_t *w_router,
                      const float *logit_offset, const float *sel_bias, const uint16_t *w13,
                      const uint16_t *w2, const uint16_t *w13_shared, const uint16_t *w2_shared,
                      uint16_t *y, int32_t *ids, float *gates, int32_t *counts,
                      uint8_t *drop_mask, float *f, float *P, float *bal_loss, float *z_loss,
                      void *ws, size_t ws_bytes, void *stream);

/* Same layer with HOST token input and HOST outputs: copies x_host (pinned or
 * pageable, [T][d] bf16) to x_dev, runs moe_layer_forward, copies y back to
 * y_host and the two losses to losses_host[0..1] (bal, z), then synchronises
 * `stream`.  x_dev / y_dev are caller device buffers of [T][d] bf16; the
 * remaining device outputs are as in moe_layer_forward.                      */
int moe_layer_forward_host(const moe_shape_t *shape, const uint16_t *x_host, uint16_t *x_dev,
                           const uint16_t *w_router, const float *logit_offset,
                           const float *sel_bias, const uint16_t *w13, const uint16_t *w2,
                           const uint16_t *w13_shared, const uint16_t *w2_shared,
                           uint16_t *y_dev, uint16_t *y_host, float *losses_host,
                           int32_t *ids, float *gates, int32_t *counts, uint8_t *drop_mask,
                           float *f, float *P, float *bal_loss, float *z_loss, void *ws,
                           size_t ws_bytes, void *stream);

/* A stream of n_batches token batches from HOST memory through the layer, with
 * the copies overlapped with the compute (double-buffered device slots):
 *   h2d_stream  copies batch i's tokens into x slot i%2 (after the layer of
 *               batch i-2 has read that slot);
 *   stream      runs moe_layer_forward on slot i%2 (after its copy-in, and
 *               after batch i-2's output has left y slot i%2);
 *   d2h_stream  copies y and the two losses of batch i out.
 * Batch i+1 is copied in and batch i-1 copied out while batch i computes, so
 * with pinned host buffers the copies hide behind the layer.  Returns after
 * all three streams have drained (synchronous for the host).
 * Arguments (all sizes from shape; T tokens per batch):
 *   x_host      [n_batches][T][d] bf16 host (pinned for overlap; pageable works
 *               but copies then block)
 *   y_host      [n_batches][T][d] bf16 host, written
 *   losses_host [n_batches][2] fp32 host, (bal, z) per batch, written
 *   x_dev, y_dev [2][T][d] bf16 device slots, 16-byte aligned
 *   loss_dev    [2][2] fp32 device slots
 *   ids, gates, counts, drop_mask, f, P: device outputs as in
 *               moe_layer_forward; they hold the last batch's values.
 * The three streams may be the same stream (no overlap).  The call creates
 * six CUDA events (no device memory) and destroys them before returning.
 * Errors: as
 * moe_layer_forward; n_batches < 0 or a null host buffer -> MOE_ERR_INVALID_ARG.
 * A failing step stops the loop; what was enqueued is drained before return. */
int moe_layer_forward_host_batches(
    const moe_shape_t *shape, int32_t n_batches, const uint16_t *x_host, uint16_t *y_host,
    float *losses_host, uint16_t *x_dev, uint16_t *y_dev, float *loss_dev,
    const uint16_t *w_router, const float *logit_offset, const float *sel_bias,
    const uint16_t *w13, const uint16_t *w2, const uint16_t *w13_shared,
    const uint16_t *w2_shared, int32_t *ids, float *gates, int32_t *counts,
    uint8_t *drop_mask, float *f, float *P, void *ws, size_t ws_bytes, void *stream,
    void *h2d_stream, void *d2h_stream);

/* Expert-choice routing (MOE_FLAG_EXPERT_CHOICE must be set in shape->flags).
 * Tokens each expert takes, r = min(T, ceil(c k T / E)), c <= 0 read as 1
 * (host pointer *r).                                                          */
int moe_ec_capacity(const moe_shape_t *shape, int64_t *r);

/* Expert-choice router ("深入理解 MoE" §9.2; the routing table of
 * "MoE：条件计算与路由").  Scores as in moe_route (softmax over experts, or
 * sigmoid with MOE_FLAG_SIGMOID; logit_offset added to the logits); expert e
 * takes the r tokens with the largest scores, equal scores to the lower token.
 * Outputs (device):
 *   row_token [E*r] int32  rows e*r .. e*r + r - 1 hold expert e's tokens in
 *                          ascending order
 *   row_gate  [E*r] fp32   the score of that (token, expert), the row's gate
 *   counts    [E]   int32  r
 *   f [E] = 1/E (n_e / (E r)), P [E] (mean score), bal_loss = lambda E sum f P,
 *   z_loss as in moe_route.
 * The cut compares the fp32 scores exactly (a radix select on their bits).  */
int moe_ec_route(const moe_shape_t *shape, const uint16_t *x, const uint16_t *w_router,
                 const float *logit_offset, int32_t *row_token, float *row_gate,
                 int32_t *counts, float *f, float *P, float *bal_loss, float *z_loss,
                 void *ws, size_t ws_bytes, void *stream);

/* The expert-choice layer: moe_ec_route, row gather, the grouped FFN (+ shared
 * experts) and the combine
 *     y[t] = sum over experts e that took t (e ascending) of
 *            row_gate[row] * E_e(x_t)  +  Ys(x_t),
 * fp32 accumulation, bf16 store; a token no expert took gets Ys(x_t) (0
 * without shared experts).  Arguments and outputs as in moe_ec_route and
 * moe_layer_forward.                                                         */
int moe_ec_layer_forward(const moe_shape_t *shape, const uint16_t *x, const uint16_t *w_router,
                         const float *logit_offset, const uint16_t *w13, const uint16_t *w2,
                         const uint16_t *w13_shared, const uint16_t *w2_shared, uint16_t *y,
                         int32_t *row_token, float *row_gate, int32_t *counts, float *f,
                         float *P, float *bal_loss, float *z_loss, void *ws, size_t ws_bytes,
                         void *stream);

/* Reads (and clears) the device status word kept in the workspace; writes
 * MOE_OK, MOE_ERR_TIMEOUT or (bounds-checked builds) MOE_ERR_BOUNDS to *status
 * (host).  Synchronises `stream`.  After MOE_ERR_TIMEOUT the workspace's
 * counters may be left nonzero: zero the workspace again before reusing it.  */
int moe_check_status(void *ws, int *status, void *stream);

/* Default wait limit, in nanoseconds, of the bounded device waits of every
 * call launched after this one whose shape->tuning.wait_timeout_ns is 0
 * (initially 2e9).  Process-wide.                                            */
int moe_set_wait_timeout_ns(uint64_t ns);

/* Launches one CTA that waits on a barrier nothing ever signals, bounded by
 * the current wait limit; it records MOE_ERR_TIMEOUT in the workspace status
 * word and returns.  Exercises the timeout path without faulting anything.   */
int moe_debug_timeout_probe(void *ws, size_t ws_bytes, void *stream);

/* Router for callers that cannot allocate device memory.  No counterpart in
 * the pages: it exists for callers that cannot call cudaMalloc or provide a
 * workspace (code running under a host framework that owns all device memory
 * through its own pool, plug-ins inside such processes, paths where an
 * allocation is not allowed).  Same arguments, kernels and outputs as
 * moe_route, without the workspace: the scratch lives in one static device
 * array of about 1 MiB inside the library, which every GPU that loads the
 * library keeps until the process exits.
 *   Limits: T <= MOE_NOALLOC_MAX_TOKENS (65536) and E <= 256; larger shapes
 *   return MOE_ERR_UNSUPPORTED before anything is enqueued.
 *   Allocates nothing (no cudaMalloc/cudaFree or allocating routine).
 *   All calls share the array, which keeps the last call's contents; each
 *   call clears the words that must start at zero.  Calls that overlap on
 *   the GPU (e.g. on unordered streams) race on it: order them.
 *   The first call on a device looks up the array's device address with that
 *   device current and caches it; make that first call before any stream
 *   capture.  Device-side timeouts are recorded in the array, not reported. */
#define MOE_NOALLOC_MAX_TOKENS 65536
int moe_route_noalloc(const moe_shape_t *shape, const uint16_t *x, const uint16_t *w_router,
                      const float *logit_offset, const float *sel_bias, int32_t *ids,
                      float *gates, int32_t *counts, float *f, float *P, float *bal_loss,
                      float *z_loss, void *stream);

/* Kernel accounting for benchmarks (host-side, process-wide, not thread-safe).
 * Kernel ids reported by moe_profile_collect: */
#define MOE_KERNEL_ROUTER 1       /* router logits + softmax + Top-k            */
#define MOE_KERNEL_FINALIZE 2     /* partial reductions, losses, scan           */
#define MOE_KERNEL_TILE_HIST 3    /* per-tile expert histogram (moe_permute)    */
#define MOE_KERNEL_SCATTER 4      /* capacity cut, permutation, row gather      */
#define MOE_KERNEL_GEMM_SWIGLU 5  /* grouped gate/up projection + SwiGLU        */
#define MOE_KERNEL_GEMM_DOWN 6    /* grouped down projection                    */
#define MOE_KERNEL_COMBINE 7      /* gate-weighted un-permute + shared output   */
#define MOE_KERNEL_OTHER 8        /* packing, probes                            */
#define MOE_KERNEL_SELECT 9       /* priority capacity cut / expert-choice cut  */
#define MOE_KERNEL_GATHER 10      /* row gather after a select                  */

/* on == 1: every subsequent kernel launch is bracketed by two CUDA events on
 * its stream; any other nonzero value is a mask, bit (1 << MOE_KERNEL_*)
 * selecting the kernels to bracket; on == 0 stops recording.  Recording
 * continues until collected.  Inside a stream capture the events become
 * external event nodes of the graph: each replay records them again, and a
 * collect after the replay returns that replay's durations.                 */
int moe_profile_enable(int on);

/* Waits for the recorded events and returns, in launch order, up to `cap`
 * (kernel id, duration in ms) pairs (host arrays); *n receives the count.
 * Clears the record.                                                          */
int moe_profile_collect(int cap, int *n, int32_t *kernel_ids, float *ms);

/* Number of kernels this library has launched in this process (host *n).   */
int moe_launch_count(uint64_t *n);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_H */
