/*
 * Oracle for the forward pass of one top-k routed Mixture-of-Experts FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, fp64 CPU statement of
 * what the layer computes.  It exists so that the tests, the smoke check and the
 * CPU-baseline leg of the benchmark can check the CUDA library against it.  It
 * shares no code, header, table or helper with the CUDA library, and the CUDA
 * library never calls it.
 *
 * Every input arrives as bf16 bit patterns (or fp32 for the per-expert vectors)
 * and is widened exactly to double; all arithmetic below is double precision.
 * Loops are plain; OpenMP only splits independent tokens across threads.
 *
 * Sources (page title, then section / equation):
 *   [KA]  "MoE：条件计算与路由" (llm-knowledge-atlas, notes 04-04):
 *         core formula y = sum_{e in TopK(g(x))} g_e(x) E_e(x); the router
 *         g(x) = softmax(W_r x); §7 Eq.(1) S = TopK(g(x)), Eq.(2) renormalised
 *         gate g~_e = g_e / sum_{j in S} g_j, Eq.(3) y = sum_{e in S} g~_e E_e(x);
 *         the ALF-LB bias b_e added to the routing scores before Top-k; the
 *         balance loss L = lambda * E * sum_e f_e P_e; §1 the load
 *         n_e = sum_i 1[e in E(x_i)]; §3 the capacity C = ceil(c B k / E).
 *   [DU]  "深入理解 MoE (混合专家模型)：稀疏激活与高效扩展" (aiattnstudio):
 *         §2.2 the sparse gate Softmax(TopK(W_g x, k)); §4.2.1 the balance loss
 *         with P_i the mean routing probability; §10.2 the SwiGLU expert
 *         E(x) = W2 (SiLU(W1 x) * W3 x); §4.2.2 the capacity-bounded router
 *         (an over-full expert keeps its highest-probability tokens); §9.2
 *         expert-choice MoE (each expert picks its own top tokens).
 *   [MO]  "MoE" (t4mako.github.io): training instability, subtracting the
 *         maximum before the softmax exponentials.
 *   [CS]  CSDN note on MoE (adg.csdn.net): the toy MoE demo (capacity keeps the
 *         first C tokens of each expert in token order; dropped tokens add
 *         nothing) and the DeepseekV3MoE excerpt (shared experts fused into one
 *         MLP of width n_shared * moe_intermediate_size and added to the routed
 *         output; moe_infer's histogram and argsort permutation).
 *   [JN]  "MOE大模型对比篇" (llm.jiangnianmeng.cn): §2.1 balance loss with
 *         P_i = (1/T) sum_x p_i(x); §2.2 router z-loss
 *         L_z = (1/B) sum_i (log sum_j exp(x_j^(i)))^2.
 *
 * Readings where the pages are silent or disagree are fixed here and listed in
 * the design notes:  Top-k over key_e = p_e + b_e, ties to the lower expert
 * index, found by a full sort; gates from the unbiased p; f_e = n_e / (k T)
 * counted before capacity; capacity C = ceil(c k T / E) computed in double, with
 * pairs kept in token-major (t, then slot) order; rows of one expert ordered by
 * (t, slot) ascending.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Exact widening of a bf16 bit pattern: the 16 bits are the top half of an fp32. */
static double bf16_val(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z))   [DU §10.2]. */
static double silu(double z) { return z / (1.0 + exp(-z)); }

/* ------------------------------------------------------------------------- */
/* Router logits  l[t][e] = sum_i W_r[e][i] x[t][i]  (+ o_e)   [KA router]    */
/* W_r is the E x d router projection, x is T x d; o is an optional           */
/* per-expert logit offset (the bias of an nn.Linear router, [CS] toy gate).  */
/* ------------------------------------------------------------------------- */
void oracle_router_logits(int T, int d, int E, const uint16_t *x, const uint16_t *wr,
                          const float *offset, double *logits)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i)
                acc += bf16_val(wr[(size_t)e * d + i]) * bf16_val(x[(size_t)t * d + i]);
            if (offset) acc += (double)offset[e];
            logits[(size_t)t * E + e] = acc;
        }
    }
}

/* Order used for Top-k: larger key first; equal keys -> lower expert index.   */
typedef struct { double key; int e; } keyed_t;

static int keyed_cmp(const void *pa, const void *pb)
{
    const keyed_t *a = (const keyed_t *)pa, *b = (const keyed_t *)pb;
    if (a->key > b->key) return -1;
    if (a->key < b->key) return 1;
    return (a->e < b->e) ? -1 : (a->e > b->e);
}

/* ------------------------------------------------------------------------- */
/* Routing for every token, from its logits.                                   */
/*  m      = max_e l_e                                                         */
/*  p_e    = exp(l_e - m) / sum_j exp(l_j - m)        (softmax, [MO] max       */
/*                                                     subtraction)            */
/*  lse    = m + log sum_j exp(l_j - m)               ([JN] §2.2 inner term)   */
/*  key_e  = p_e + b_e                                 ([KA] ALF-LB)           */
/*  S      = the k largest keys, descending            ([KA] §7 Eq.(1))        */
/*  g~_s   = p_{S_s} / sum_{j in S} p_j                ([KA] §7 Eq.(2))        */
/*  gap    = key of the k-th minus key of the (k+1)-th (+inf when k == E, or  */
/*           k == 0)                                                           */
/* When force_mask[t] != 0 the selection S of token t is taken from            */
/* force_ids[t][0..k) instead (used only for near-tie tokens, whose order a    */
/* lower-precision implementation may legitimately flip); the gates are then   */
/* computed for that set by the same Eq.(2).                                   */
/* ------------------------------------------------------------------------- */
/* Variants (flags):                                                            */
/*  ORACLE_SIGMOID   scores s_e = 1 / (1 + exp(-l_e)), each expert on its own,  */
/*                   instead of the softmax (the CSDN note, §9: DeepSeek-V3     */
/*                   moved the gate from softmax to sigmoid); p below then     */
/*                   holds s                                                    */
/*  ORACLE_NO_RENORM gates are the selected scores themselves, not divided by  */
/*                   their sum ("MoE：条件计算与路由" §7: without the renormal-  */
/*                   isation the output scale follows the dropped mass)         */
/* entropy[t] (optional) = -sum_e q_e log q_e of the router distribution q     */
/* ("MoE：条件计算与路由" §9), q = p for the softmax, q = s / sum s for sigmoid.  */
#define ORACLE_SIGMOID 1
#define ORACLE_NO_RENORM 2

void oracle_route(int T, int E, int k, int flags, const double *logits, const float *sel_bias,
                  const int32_t *force_ids, const uint8_t *force_mask,
                  double *p, double *lse, int32_t *ids, double *gates, double *gap,
                  double *entropy)
{
#pragma omp parallel
    {
        keyed_t *ord = (keyed_t *)malloc(sizeof(keyed_t) * (size_t)(E > 0 ? E : 1));
#pragma omp for schedule(static)
        for (int t = 0; t < T; ++t) {
            const double *l = logits + (size_t)t * E;
            double *pt = p + (size_t)t * E;
            double m = l[0];
            for (int e = 1; e < E; ++e)
                if (l[e] > m) m = l[e];
            double s = 0.0;
            for (int e = 0; e < E; ++e) s += exp(l[e] - m);
            for (int e = 0; e < E; ++e) pt[e] = exp(l[e] - m) / s;
            lse[t] = m + log(s);
            if (flags & ORACLE_SIGMOID)
                for (int e = 0; e < E; ++e) pt[e] = 1.0 / (1.0 + exp(-l[e]));
            if (entropy) {
                double qs = 0.0, h = 0.0;
                for (int e = 0; e < E; ++e) qs += pt[e];
                for (int e = 0; e < E; ++e) {
                    double q = pt[e] / qs;
                    if (q > 0.0) h -= q * log(q);
                }
                entropy[t] = h;
            }

            for (int e = 0; e < E; ++e) {
                ord[e].key = pt[e] + (sel_bias ? (double)sel_bias[e] : 0.0);
                ord[e].e = e;
            }
            qsort(ord, (size_t)E, sizeof(keyed_t), keyed_cmp);
            gap[t] = (k > 0 && k < E) ? ord[k - 1].key - ord[k].key : INFINITY;

            int32_t *it = ids + (size_t)t * k;
            if (force_mask && force_mask[t]) {
                for (int s2 = 0; s2 < k; ++s2) it[s2] = force_ids[(size_t)t * k + s2];
            } else {
                for (int s2 = 0; s2 < k; ++s2) it[s2] = ord[s2].e;
            }
            double denom = 0.0;
            for (int s2 = 0; s2 < k; ++s2) denom += pt[it[s2]];
            if (flags & ORACLE_NO_RENORM) denom = 1.0;
            for (int s2 = 0; s2 < k; ++s2) gates[(size_t)t * k + s2] = pt[it[s2]] / denom;
        }
        free(ord);
    }
}

/* ------------------------------------------------------------------------- */
/* Expert capacity C = ceil(c * k * T / E)   ([KA] §3, B = T tokens).         */
/* Returns -1 (no limit) when c <= 0.                                          */
/* ------------------------------------------------------------------------- */
int64_t oracle_capacity(double c, int k, int T, int E)
{
    if (!(c > 0.0)) return -1;
    return (int64_t)ceil(c * (double)k * (double)T / (double)E);
}

/* ------------------------------------------------------------------------- */
/* Dispatch: loads, capacity cut and the expert-contiguous permutation.        */
/*  counts[e]   = n_e = #{(t,s): ids[t][s] = e}              ([KA] §1)         */
/*  walking (t,s) in token-major order, a pair is kept iff fewer than C pairs  */
/*  of its expert were kept before it ([CS] toy demo: the first C tokens of    */
/*  each expert in token order); kept_counts[e] = pairs kept for e             */
/*  offsets[e]  = sum_{j<e} kept_counts[j]; offsets[E] = R                     */
/*  slot_row[t][s] = offsets[e] + (rank of (t,s) among e's kept pairs), or -1  */
/*  row_token[r]   = t of the pair placed at row r                              */
/* This is a stable sort by expert of the token-major flattening ([CS]         */
/* moe_infer's argsort, with ties in token order).                             */
/* ------------------------------------------------------------------------- */
void oracle_dispatch(int T, int E, int k, const int32_t *ids, int64_t C,
                     int32_t *counts, int32_t *kept_counts, int32_t *offsets,
                     int32_t *slot_row, int32_t *row_token, uint8_t *dropped)
{
    int32_t *rank = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T * (int64_t)k + 1));
    for (int e = 0; e < E; ++e) { counts[e] = 0; kept_counts[e] = 0; }
    for (int t = 0; t < T; ++t) {
        for (int s = 0; s < k; ++s) {
            int e = ids[(size_t)t * k + s];
            size_t q = (size_t)t * k + s;
            counts[e] += 1;
            if (C < 0 || kept_counts[e] < C) {
                rank[q] = kept_counts[e];
                kept_counts[e] += 1;
                dropped[q] = 0;
            } else {
                rank[q] = -1;
                dropped[q] = 1;
            }
        }
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + kept_counts[e];
    for (int t = 0; t < T; ++t) {
        for (int s = 0; s < k; ++s) {
            size_t q = (size_t)t * k + s;
            if (dropped[q]) { slot_row[q] = -1; continue; }
            int e = ids[q];
            int r = offsets[e] + rank[q];
            slot_row[q] = r;
            row_token[r] = t;
        }
    }
    free(rank);
}

/* ------------------------------------------------------------------------- */
/* Dispatch with probability-priority capacity ([DU] §4.2.2, the capacity-   */
/* bounded router: when more pairs reach an expert than its capacity, the    */
/* ones with the highest routing probability are kept).                      */
/* Reading: the priority of pair (t,s) is the token's unbiased score of its   */
/* expert, p[t][ids[t][s]] (softmax probability, or the sigmoid score); one   */
/* capacity C = ceil(c k T / E) per expert over all its pairs; equal scores   */
/* are taken in token-major (t, s) order.  Kept rows keep the stable layout   */
/* of oracle_dispatch: within an expert they are ordered by (t, s).           */
/* p: [T][E].  Outputs as oracle_dispatch.                                     */
/* force (optional, [T][k]): +1 / -1 put a pair above / below every score;    */
/* used only for pairs whose score sits within rounding of an expert's cut,   */
/* where a lower-precision implementation may legitimately decide otherwise.  */
/* ------------------------------------------------------------------------- */
typedef struct { double key; int64_t q; } prio_t;

static int prio_cmp(const void *pa, const void *pb)
{
    const prio_t *a = (const prio_t *)pa, *b = (const prio_t *)pb;
    if (a->key > b->key) return -1;
    if (a->key < b->key) return 1;
    return (a->q < b->q) ? -1 : (a->q > b->q);
}

void oracle_dispatch_priority(int T, int E, int k, const int32_t *ids, const double *p,
                              const int8_t *force, int64_t C, int32_t *counts,
                              int32_t *kept_counts,
                              int32_t *offsets, int32_t *slot_row, int32_t *row_token,
                              uint8_t *dropped)
{
    const int64_t n = (int64_t)T * k;
    prio_t *list = (prio_t *)malloc(sizeof(prio_t) * (size_t)(n > 0 ? n : 1));
    for (int e = 0; e < E; ++e) { counts[e] = 0; kept_counts[e] = 0; }
    for (int64_t q = 0; q < n; ++q) dropped[q] = 0;
    /* the cut, one expert at a time: sort its pairs by (score desc, q asc) */
    for (int e = 0; e < E; ++e) {
        int64_t m = 0;
        for (int64_t q = 0; q < n; ++q) {
            if (ids[q] != e) continue;
            list[m].key = p[(q / k) * (int64_t)E + e];
            if (force && force[q]) list[m].key = (force[q] > 0) ? INFINITY : -INFINITY;
            list[m].q = q;
            ++m;
        }
        counts[e] = (int32_t)m;
        if (C >= 0 && m > C) {
            qsort(list, (size_t)m, sizeof(prio_t), prio_cmp);
            for (int64_t j = C; j < m; ++j) dropped[list[j].q] = 1;
        }
        kept_counts[e] = (int32_t)((C >= 0 && m > C) ? C : m);
    }
    /* the permutation: kept pairs of each expert in (t, s) order */
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = kept_counts[e] + offsets[e];
    int32_t *next = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int e = 0; e < E; ++e) next[e] = offsets[e];
    for (int64_t q = 0; q < n; ++q) {
        if (dropped[q]) { slot_row[q] = -1; continue; }
        int r = next[ids[q]]++;
        slot_row[q] = r;
        row_token[r] = (int32_t)(q / k);
    }
    free(next);
    free(list);
}

/* ------------------------------------------------------------------------- */
/* Expert-choice routing ([DU] §9.2 Expert Choice MoE: every expert picks the */
/* tokens that matter most to it; "MoE：条件计算与路由", routing table: each    */
/* expert takes its top-r_e tokens, naturally balanced, a token may be picked */
/* by several experts or none).                                               */
/* Readings: the score of token t for expert e is the router score p[t][e]    */
/* (softmax over experts, or the sigmoid score), which is also the gate; every */
/* expert takes r tokens, r = min(T, ceil(c k T / E)) with c = 1 when c <= 0,  */
/* so that at c = 1 the rows computed equal those of token-choice top-k;      */
/* equal scores go to the lower token index.  Expert e's rows are            */
/* e*r .. e*r + r - 1, its chosen tokens in ascending order.                 */
/* p: [T][E]; row_token, row_gate: [E*r].  force (optional, [E][T]): +1 / -1 */
/* put (e, t) above / below every score for the pick (never for the gate);    */
/* used only near an expert's cut, as for oracle_dispatch_priority.           */
/* ------------------------------------------------------------------------- */
int64_t oracle_ec_capacity(double c, int k, int T, int E)
{
    double cc = (c > 0.0) ? c : 1.0;
    int64_t r = (int64_t)ceil(cc * (double)k * (double)T / (double)E);
    return r < T ? r : T;
}

static int i32_cmp(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a < b) ? -1 : (a > b);
}

void oracle_expert_choice(int T, int E, int64_t r, const double *p, const int8_t *force,
                          int32_t *row_token, double *row_gate)
{
    prio_t *list = (prio_t *)malloc(sizeof(prio_t) * (size_t)(T > 0 ? T : 1));
    for (int e = 0; e < E; ++e) {
        for (int t = 0; t < T; ++t) {
            list[t].key = p[(size_t)t * E + e];
            if (force && force[(size_t)e * T + t])
                list[t].key = (force[(size_t)e * T + t] > 0) ? INFINITY : -INFINITY;
            list[t].q = t;
        }
        qsort(list, (size_t)T, sizeof(prio_t), prio_cmp);
        int32_t *rt = row_token + (size_t)e * r;
        for (int64_t j = 0; j < r; ++j) rt[j] = (int32_t)list[j].q;
        qsort(rt, (size_t)r, sizeof(int32_t), i32_cmp);
        for (int64_t j = 0; j < r; ++j) row_gate[(size_t)e * r + j] = p[(size_t)rt[j] * E + e];
    }
    free(list);
}

/* ------------------------------------------------------------------------- */
/* One SwiGLU expert on one input row   ([DU] §10.2):                          */
/*   out[o] = sum_j W2[o][j] * SiLU(sum_i W1[j][i] x_i) * (sum_i W3[j][i] x_i) */
/* W1, W3: [Mw][d] (nn.Linear(d -> Mw).weight), W2: [d][Mw]                     */
/* (nn.Linear(Mw -> d).weight).                                                 */
/* ------------------------------------------------------------------------- */
void oracle_swiglu_row(int d, int Mw, const uint16_t *xrow, const uint16_t *w1,
                       const uint16_t *w3, const uint16_t *w2, double *out)
{
    double *xv = (double *)malloc(sizeof(double) * (size_t)d);
    double *h = (double *)malloc(sizeof(double) * (size_t)Mw);
    for (int i = 0; i < d; ++i) xv[i] = bf16_val(xrow[i]);
    for (int j = 0; j < Mw; ++j) {
        double a = 0.0, b = 0.0;
        for (int i = 0; i < d; ++i) {
            a += bf16_val(w1[(size_t)j * d + i]) * xv[i];
            b += bf16_val(w3[(size_t)j * d + i]) * xv[i];
        }
        h[j] = silu(a) * b;
    }
    for (int o = 0; o < d; ++o) {
        double acc = 0.0;
        for (int j = 0; j < Mw; ++j) acc += bf16_val(w2[(size_t)o * Mw + j]) * h[j];
        out[o] = acc;
    }
    free(h);
    free(xv);
}

/* ------------------------------------------------------------------------- */
/* Expert outputs for a list of (row, expert) pairs: out[r] = E_e(x_rows[r]).  */
/* W1, W3: [E][M][d]; W2: [E][d][M].                                            */
/* ------------------------------------------------------------------------- */
void oracle_expert_rows(int n, int d, int M, const uint16_t *x_rows, const int32_t *expert,
                        const uint16_t *w1, const uint16_t *w3, const uint16_t *w2,
                        double *out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < n; ++r) {
        size_t e = (size_t)expert[r];
        oracle_swiglu_row(d, M, x_rows + (size_t)r * d, w1 + e * M * d, w3 + e * M * d,
                          w2 + e * d * M, out + (size_t)r * d);
    }
}

/* ------------------------------------------------------------------------- */
/* Layer output for the tokens listed in sel[0..n_sel):                         */
/*   y[t] = sum_{kept s} g~[t][s] * E_{ids[t][s]}(x_t)  +  Ys(x_t)              */
/* ([KA] §7 Eq.(3); dropped pairs contribute nothing and the remaining gates   */
/* are not renormalised, [CS] toy demo; the shared experts of width            */
/* Ms = n_shared * M act as one SwiGLU MLP with gate 1, added to the routed    */
/* sum, [CS] DeepseekV3MoE forward).  ws1/ws3: [Ms][d], ws2: [d][Ms], or NULL. */
/* ------------------------------------------------------------------------- */
void oracle_layer_tokens(int T, int d, int M, int E, int k, int Ms,
                         const uint16_t *x, const int32_t *ids, const double *gates,
                         const uint8_t *dropped,
                         const uint16_t *w1, const uint16_t *w3, const uint16_t *w2,
                         const uint16_t *ws1, const uint16_t *ws3, const uint16_t *ws2,
                         int n_sel, const int32_t *sel, double *y_sel)
{
    (void)T; (void)E;
#pragma omp parallel
    {
        double *tmp = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int q = 0; q < n_sel; ++q) {
            size_t t = (size_t)sel[q];
            double *yt = y_sel + (size_t)q * d;
            for (int o = 0; o < d; ++o) yt[o] = 0.0;
            for (int s = 0; s < k; ++s) {
                size_t pq = t * k + s;
                if (dropped[pq]) continue;
                size_t e = (size_t)ids[pq];
                oracle_swiglu_row(d, M, x + t * d, w1 + e * M * d, w3 + e * M * d,
                                  w2 + e * d * M, tmp);
                for (int o = 0; o < d; ++o) yt[o] += gates[pq] * tmp[o];
            }
            if (Ms > 0 && ws1) {
                oracle_swiglu_row(d, Ms, x + t * d, ws1, ws3, ws2, tmp);
                for (int o = 0; o < d; ++o) yt[o] += tmp[o];
            }
        }
        free(tmp);
    }
}

/* ------------------------------------------------------------------------- */
/* Expert-choice layer output for the tokens listed in sel[0..n_sel):          */
/*   y[t] = sum over experts e that picked t (e ascending) of                  */
/*          row_gate[row] * E_e(x_t)  +  Ys(x_t)                               */
/* ([KA] §7 Eq.(3) with the selection made by the experts; the shared experts */
/* as in oracle_layer_tokens).  A token no expert picked gets only Ys.        */
/* ------------------------------------------------------------------------- */
void oracle_ec_layer_tokens(int T, int d, int M, int E, int64_t r, int Ms,
                            const uint16_t *x, const int32_t *row_token, const double *row_gate,
                            const uint16_t *w1, const uint16_t *w3, const uint16_t *w2,
                            const uint16_t *ws1, const uint16_t *ws3, const uint16_t *ws2,
                            int n_sel, const int32_t *sel, double *y_sel)
{
    (void)T;
#pragma omp parallel
    {
        double *tmp = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int q = 0; q < n_sel; ++q) {
            const int32_t t = sel[q];
            double *yt = y_sel + (size_t)q * d;
            for (int o = 0; o < d; ++o) yt[o] = 0.0;
            for (int e = 0; e < E; ++e) {
                for (int64_t j = 0; j < r; ++j) {
                    size_t row = (size_t)e * r + j;
                    if (row_token[row] != t) continue;
                    oracle_swiglu_row(d, M, x + (size_t)t * d, w1 + (size_t)e * M * d,
                                      w3 + (size_t)e * M * d, w2 + (size_t)e * d * M, tmp);
                    for (int o = 0; o < d; ++o) yt[o] += row_gate[row] * tmp[o];
                }
            }
            if (Ms > 0 && ws1) {
                oracle_swiglu_row(d, Ms, x + (size_t)t * d, ws1, ws3, ws2, tmp);
                for (int o = 0; o < d; ++o) yt[o] += tmp[o];
            }
        }
        free(tmp);
    }
}

/* ------------------------------------------------------------------------- */
/* Side outputs.                                                                */
/*   f_e  = n_e / N                   (fraction of routed pairs, before any    */
/*                                     capacity cut; sums to 1; N = k T for    */
/*                                     token choice, E r for expert choice)    */
/*   P_e  = (1/T) sum_t p_e(t)        ([JN] §2.1, [DU] §4.2.1)                 */
/*   L_bal = lambda * E * sum_e f_e P_e   ([KA] balance loss)                   */
/*   L_z  = (1/T) sum_t lse_t^2       ([JN] §2.2)                               */
/* With T == 0 or k == 0 the undefined ratios are reported as 0.               */
/* ------------------------------------------------------------------------- */
void oracle_losses_n(int T, int E, double N, const int32_t *counts, const double *p,
                     const double *lse, double lambda, double *f, double *P,
                     double *L_bal, double *L_z)
{
    double sfp = 0.0, sz = 0.0;
    for (int e = 0; e < E; ++e) {
        f[e] = (T > 0 && N > 0.0) ? (double)counts[e] / N : 0.0;
        double acc = 0.0;
        for (int t = 0; t < T; ++t) acc += p[(size_t)t * E + e];
        P[e] = (T > 0) ? acc / (double)T : 0.0;
        sfp += f[e] * P[e];
    }
    for (int t = 0; t < T; ++t) sz += lse[t] * lse[t];
    *L_bal = lambda * (double)E * sfp;
    *L_z = (T > 0) ? sz / (double)T : 0.0;
}

void oracle_losses(int T, int E, int k, const int32_t *counts, const double *p,
                   const double *lse, double lambda, double *f, double *P,
                   double *L_bal, double *L_z)
{
    oracle_losses_n(T, E, (double)k * (double)T, counts, p, lse, lambda, f, P, L_bal, L_z);
}

/* ------------------------------------------------------------------------- */
/* Combine alone, from expert-order rows   ([KA] §7 Eq.(3); [CS] moe_infer's  */
/* un-permute new_x[idxs] = outs, then the fp32 gate-weighted sum over k, and */
/* DeepseekV3MoE's y + shared_experts(identity)):                             */
/*   y[t] = sum_{s: slot_row[t][s] >= 0} gates[t][s] * y_perm[slot_row[t][s]] */
/*          + y_shared[t]                                                     */
/* y_perm: [R][d] bf16, y_shared: [T][d] bf16 or NULL.                         */
/* ------------------------------------------------------------------------- */
void oracle_combine(int T, int d, int k, const uint16_t *y_perm, const int32_t *slot_row,
                    const double *gates, const uint16_t *y_shared, double *y)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        double *yt = y + (size_t)t * d;
        for (int o = 0; o < d; ++o) yt[o] = 0.0;
        for (int s = 0; s < k; ++s) {
            int r = slot_row[(size_t)t * k + s];
            if (r < 0) continue;
            double g = gates[(size_t)t * k + s];
            for (int o = 0; o < d; ++o) yt[o] += g * bf16_val(y_perm[(size_t)r * d + o]);
        }
        if (y_shared)
            for (int o = 0; o < d; ++o) yt[o] += bf16_val(y_shared[(size_t)t * d + o]);
    }
}

/* ------------------------------------------------------------------------- */
/* Importance of each expert over the batch and its squared coefficient of    */
/* variation (the CSDN note, "Balancing Expert Utilization": Importance(X) =  */
/* sum_x G(x), L_importance = w * CV(Importance)^2).  G(x) is the sparse gate */
/* vector: the token's gates on its selected experts, zero elsewhere (before  */
/* any capacity cut).  CV = population standard deviation / mean over the E   */
/* experts; reported as 0 when the mean is 0.                                */
/* ------------------------------------------------------------------------- */
void oracle_importance(int T, int E, int k, const int32_t *ids, const double *gates,
                       double *importance, double *cv2)
{
    for (int e = 0; e < E; ++e) importance[e] = 0.0;
    for (int t = 0; t < T; ++t)
        for (int s = 0; s < k; ++s)
            importance[ids[(size_t)t * k + s]] += gates[(size_t)t * k + s];
    double mean = 0.0;
    for (int e = 0; e < E; ++e) mean += importance[e];
    mean /= (double)E;
    double var = 0.0;
    for (int e = 0; e < E; ++e) var += (importance[e] - mean) * (importance[e] - mean);
    var /= (double)E;
    *cv2 = (mean != 0.0) ? var / (mean * mean) : 0.0;
}

/* ------------------------------------------------------------------------- */
/* ALF-LB bias update ("MoE：条件计算与路由", ALF-LB section: the bias of an    */
/* overloaded expert decreases, that of an underloaded expert increases, at  */
/* rate gamma, outside the backward graph).  Reading of the unstated rule:   */
/*   b_e <- b_e + gamma * sign(nbar - n_e),  nbar = k T / E,  sign(0) = 0,   */
/* with b and gamma in fp32 and the sum rounded once to fp32.                */
/* ------------------------------------------------------------------------- */
void oracle_alf_bias_update(int E, int T, int k, const int32_t *counts, float gamma,
                            const float *bias_in, float *bias_out)
{
    const double nbar = (double)k * (double)T / (double)E;
    for (int e = 0; e < E; ++e) {
        const double diff = nbar - (double)counts[e];
        const double sgn = (diff > 0.0) ? 1.0 : ((diff < 0.0) ? -1.0 : 0.0);
        bias_out[e] = (float)((double)bias_in[e] + (double)gamma * sgn);
    }
}
