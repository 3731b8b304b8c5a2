/*
 * moe_oracle.c -- plain, slow CPU oracle of the fused MoE layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this library.  The CUDA product
 * path never calls it and shares no code, header or constant with it.
 *
 * Source of every definition: the page "用Ascend C写一个MoE融合算子" (Writing
 * a fused MoE operator in Ascend C), section "MoE的计算流程" (the five-step
 * compute flow: Routing, Gating, Dispatch, Expert, Combine), its code
 * listings for the router kernel (section "1. Routing + Gating 合并") and the
 * expert kernel (section "2. Dispatch + Expert + Combine 流水线"); the page
 * "CANN ops-transformer：MoE 路由算子的负载均衡策略" (token dropping, section
 * "负载不均衡的根源"); and the page "CANN ops-transformer MoE" article, section
 * 4.3 (capacity_factor = 1.2).  Where the pages are silent the readings are:
 *   - TopK ties go to the lower expert index; the k columns are ordered by
 *     descending logit (then ascending index).
 *   - Gate softmax runs over the k selected logits only.
 *   - GELU is the exact erf form 0.5 z (1 + erf(z / sqrt 2)).
 *   - capacity C = ceil(cf * T * k / E - 1e-9); cf <= 0 means no limit.
 *   - Overflow is dropped in ascending (token, slot) order; survivors keep
 *     their softmax weight (no renormalisation); a token whose every slot is
 *     dropped gets y = 0.
 *   - Router logits are fp32 (the article's mixed-precision advice, section
 *     4.2, keeps the router in FP32): the dot product is accumulated in fp64
 *     and rounded once to fp32, then the optional fp32 bias is added in fp32.
 *
 * Arithmetic: inputs are bf16 bit patterns, decoded exactly; every dot
 * product accumulates in double in ascending index order; the FFN, the
 * softmax and the combine stay in double.  No blocking, fusion or reordering.
 *
 * Layouts (row-major, contiguous):
 *   x[T][H], w_router[H][E], bias[E] (optional), W1[E][H][F] (SwiGLU:
 *   [E][H][2F] = [gate | up]), W2[E][F][H],
 *   logits[T][E], ids[T][k], top_logits[T][k], w[T][k], counts[E],
 *   offsets[E+1], perm[T*k] (entries t*k+j), slot[T][k] (-1 = dropped).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact widening of a bf16 bit pattern: bf16 is the top half of an fp32. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Step 1, routing: scores = x * W_router  (compute-flow step 1; the router
 * kernel's "Step 1: x × W_router" with x [batch, hidden_dim] and W_router
 * [hidden_dim, num_experts]).
 *   logits[t][e] = fp32( sum_h x[t][h] * w_router[h][e] )  (+ bias[e] in fp32)
 */
int oracle_router_logits(int T, int H, int E, const uint16_t *x,
                         const uint16_t *w_router, const float *bias,
                         float *logits, int nthreads)
{
    if (T < 0 || H < 1 || E < 1 || !x || !w_router || !logits) return 1;
    set_threads(nthreads);
    int bad = 0;
#pragma omp parallel
    {
        double *acc = (double *)malloc(sizeof(double) * (size_t)E);
        if (!acc) {
#pragma omp atomic write
            bad = 2;
        }
#pragma omp for schedule(static)
        for (int t = 0; t < T; t++) {
            if (!acc) continue;
            /* acc[e] accumulates over h in ascending order for every e */
            for (int e = 0; e < E; e++) acc[e] = 0.0;
            for (int h = 0; h < H; h++) {
                double xv = bf16_value(x[(size_t)t * H + h]);
                for (int e = 0; e < E; e++)
                    acc[e] += xv * bf16_value(w_router[(size_t)h * E + e]);
            }
            for (int e = 0; e < E; e++) {
                float l = (float)acc[e];
                if (bias) l = l + bias[e];
                logits[(size_t)t * E + e] = l;
            }
        }
        free(acc);
    }
    return bad;
}

/*
 * Step 1 continued, TopK (the router kernel's "Step 2: TopK选择", one
 * independent top-k per sample): sort the E experts of token t by descending
 * logit with a stable insertion sort, so equal logits keep ascending index
 * order, and keep the first k.
 */
int oracle_topk(int T, int E, int k, const float *logits, int32_t *ids,
                float *top_logits)
{
    if (T < 0 || E < 1 || k < 1 || k > E || !logits || !ids || !top_logits) return 1;
    int *order = (int *)malloc(sizeof(int) * (size_t)E);
    if (!order) return 2;
    for (int t = 0; t < T; t++) {
        const float *l = logits + (size_t)t * E;
        for (int e = 0; e < E; e++) {
            /* insert e behind every earlier index whose logit is >= l[e] */
            int pos = e;
            while (pos > 0 && l[order[pos - 1]] < l[e]) {
                order[pos] = order[pos - 1];
                pos--;
            }
            order[pos] = e;
        }
        for (int j = 0; j < k; j++) {
            ids[(size_t)t * k + j] = order[j];
            top_logits[(size_t)t * k + j] = l[order[j]];
        }
    }
    free(order);
    return 0;
}

/*
 * Step 2, gating: weights = Softmax(scores) over the k selected scores only
 * (the router kernel's "Step 3: Softmax归一化（只对top-k个分数做）").
 *   w[t][j] = exp(s_j - max_i s_i) / sum_i exp(s_i - max_i s_i), in double.
 */
int oracle_gate_softmax(int T, int k, const float *top_logits, float *w)
{
    if (T < 0 || k < 1 || !top_logits || !w) return 1;
    for (int t = 0; t < T; t++) {
        const float *s = top_logits + (size_t)t * k;
        double m = (double)s[0];
        for (int j = 1; j < k; j++)
            if ((double)s[j] > m) m = (double)s[j];
        double z = 0.0;
        for (int j = 0; j < k; j++) z += exp((double)s[j] - m);
        for (int j = 0; j < k; j++)
            w[(size_t)t * k + j] = (float)(exp((double)s[j] - m) / z);
    }
    return 0;
}

/*
 * Step 2 variant, the Softmax -> Top-k order of the CANN MoE article's
 * section 2.1: the softmax runs over all E logits of the token and the k
 * selected experts keep their probabilities,
 *   p_e = exp(l_e - max_i l_i) / sum_i exp(l_i - max_i l_i),   w[t][j] = p_{ids[t][j]},
 * (mode 1), or those k probabilities divided by their sum (mode 2).  In
 * double, stored as fp32.  Selection is unchanged (softmax is monotonic).
 */
int oracle_gate_softmax_all(int T, int E, int k, const float *logits, const int32_t *ids,
                            int mode, float *w)
{
    if (T < 0 || E < 1 || k < 1 || k > E || !logits || !ids || !w) return 1;
    if (mode != 1 && mode != 2) return 1;
    for (int t = 0; t < T; t++) {
        const float *l = logits + (size_t)t * E;
        double m = (double)l[0];
        for (int e = 1; e < E; e++)
            if ((double)l[e] > m) m = (double)l[e];
        double z = 0.0;
        for (int e = 0; e < E; e++) z += exp((double)l[e] - m);
        double sel = 0.0;
        for (int j = 0; j < k; j++) sel += exp((double)l[ids[(size_t)t * k + j]] - m) / z;
        for (int j = 0; j < k; j++) {
            double p = exp((double)l[ids[(size_t)t * k + j]] - m) / z;
            w[(size_t)t * k + j] = (float)(mode == 1 ? p : p / sel);
        }
    }
    return 0;
}

/*
 * Expert capacity from the capacity factor (article section 4.3,
 * capacity_factor = 1.2; the blocked dispatch buffer of the compute flow is
 * [num_experts, expert_capacity]).  Reading: C = ceil(cf*T*k/E - 1e-9); the
 * 1e-9 guard keeps an exact integer quotient from rounding up.  Returns -1
 * (no limit) for cf <= 0 or NaN.
 */
long oracle_capacity(int T, int k, int E, double cf)
{
    if (!(cf > 0.0)) return -1;
    double c = ceil(cf * (double)T * (double)k / (double)E - 1e-9);
    if (c < 0.0) c = 0.0;
    if (c > (double)T * (double)k) c = (double)T * (double)k;
    return (long)c;
}

/*
 * Step 3, dispatch: x_i = x[assigned_to_expert_i].  Follows the expert
 * kernel's GatherTokensByExpert literally: for each expert e, scan tokens b
 * ascending and slots j ascending; every match is the next row of expert e.
 * With a capacity C the first C matches are kept and later ones dropped
 * (token dropping of overloaded experts).
 *   counts[e]   kept rows of e
 *   offsets     exclusive prefix sum of counts, offsets[E] = total kept
 *   perm[r]     t*k + j of the r-th kept row (rows grouped by expert)
 *   slot[t][j]  row r holding assignment (t, j), or -1 if dropped
 * Ids outside [0, E) are an error (return 3).
 */
int oracle_dispatch(int T, int k, int E, long capacity, const int32_t *ids,
                    int32_t *counts, int32_t *offsets, int32_t *perm,
                    int32_t *slot)
{
    if (T < 0 || k < 1 || E < 1 || !ids || !counts || !offsets || !perm || !slot) return 1;
    for (long i = 0; i < (long)T * k; i++) {
        if (ids[i] < 0 || ids[i] >= E) return 3;
        slot[i] = -1;
    }
    int32_t row = 0;
    for (int e = 0; e < E; e++) {
        offsets[e] = row;
        int32_t count = 0;
        for (int b = 0; b < T; b++) {
            for (int j = 0; j < k; j++) {
                if (ids[(size_t)b * k + j] != e) continue;
                if (capacity >= 0 && count >= capacity) continue; /* dropped */
                perm[row] = b * k + j;
                slot[(size_t)b * k + j] = row;
                row++;
                count++;
            }
        }
        counts[e] = count;
    }
    offsets[E] = row;
    return 0;
}

/*
 * Step 4, one expert on one row: y = activation(x × W1) × W2 with GELU
 * (the expert kernel's "Step 3: Expert计算": Mmad with M = tokens,
 * N = ffn_hidden_dim, K = hidden_dim; GELU; Mmad with N = hidden_dim,
 * K = ffn_hidden_dim).  u and g are kept in double; no bf16 rounding of the
 * hidden activation is emulated.
 */
static void expert_ffn_row(int H, int F, const uint16_t *xrow,
                           const uint16_t *w1e, const uint16_t *w2e,
                           double *g, double *out)
{
    /* u[f] = sum_h x[h] * W1[h][f], accumulated over h in ascending order
     * (the loops run h-outer only so that W1 is read row by row) */
    for (int f = 0; f < F; f++) g[f] = 0.0;
    for (int h = 0; h < H; h++) {
        double xv = bf16_value(xrow[h]);
        const uint16_t *w1row = w1e + (size_t)h * F;
        for (int f = 0; f < F; f++) g[f] += xv * bf16_value(w1row[f]);
    }
    for (int f = 0; f < F; f++) {
        double u = g[f];
        g[f] = 0.5 * u * (1.0 + erf(u / sqrt(2.0)));
    }
    /* out[h] = sum_f g[f] * W2[f][h], accumulated over f in ascending order */
    for (int h = 0; h < H; h++) out[h] = 0.0;
    for (int f = 0; f < F; f++) {
        double gv = g[f];
        const uint16_t *w2row = w2e + (size_t)f * H;
        for (int h = 0; h < H; h++) out[h] += gv * bf16_value(w2row[h]);
    }
}

/*
 * Step 4 with a gated expert (the SwiGLU FFN of the Llama 3 / Mixtral /
 * DeepSeek models the compute-flow page names): with W1 = [W_gate | W_up]
 * of shape [H][2F] and W2 = W_down [F][H],
 *   g = x W_gate,  u = x W_up,  a_f = SiLU(g_f) u_f = g_f / (1 + exp(-g_f)) u_f,
 *   out = a W_down,
 * all in double, dot products accumulated in ascending index order.
 */
static void expert_swiglu_row(int H, int F, const uint16_t *xrow,
                              const uint16_t *w1e, const uint16_t *w2e,
                              double *g, double *out)
{
    /* g[0..F) = gate, g[F..2F) = up, both accumulated over h ascending */
    for (int f = 0; f < 2 * F; f++) g[f] = 0.0;
    for (int h = 0; h < H; h++) {
        double xv = bf16_value(xrow[h]);
        const uint16_t *w1row = w1e + (size_t)h * 2 * F;
        for (int f = 0; f < 2 * F; f++) g[f] += xv * bf16_value(w1row[f]);
    }
    for (int f = 0; f < F; f++) {
        double gate = g[f];
        g[f] = gate / (1.0 + exp(-gate)) * g[F + f];
    }
    for (int h = 0; h < H; h++) out[h] = 0.0;
    for (int f = 0; f < F; f++) {
        double av = g[f];
        const uint16_t *w2row = w2e + (size_t)f * H;
        for (int h = 0; h < H; h++) out[h] += av * bf16_value(w2row[h]);
    }
}

int oracle_expert_swiglu(int H, int F, const uint16_t *xrow, const uint16_t *w1e,
                         const uint16_t *w2e, double *out)
{
    if (H < 1 || F < 1 || !xrow || !w1e || !w2e || !out) return 1;
    double *g = (double *)malloc(sizeof(double) * 2 * (size_t)F);
    if (!g) return 2;
    expert_swiglu_row(H, F, xrow, w1e, w2e, g, out);
    free(g);
    return 0;
}

/* Exported single-row expert FFN (for the oracle's own pins). */
int oracle_expert_ffn(int H, int F, const uint16_t *xrow, const uint16_t *w1e,
                      const uint16_t *w2e, double *out)
{
    if (H < 1 || F < 1 || !xrow || !w1e || !w2e || !out) return 1;
    double *g = (double *)malloc(sizeof(double) * (size_t)F);
    if (!g) return 2;
    expert_ffn_row(H, F, xrow, w1e, w2e, g, out);
    free(g);
    return 0;
}

/*
 * Step 5, combine: y = Σ weights_i × y_i, written back to the token's
 * original position and accumulated over its top-k slots (the expert
 * kernel's ScatterWithWeights: output(orig_pos, d) += weight * expert_out).
 * Here written per token: y[t] = sum over kept j (ascending) of
 * w[t][j] * Expert_{ids[t][j]}(x[t]).  A token with no kept slot gets 0.
 * Computed for the n_rows tokens listed in rows[]; y is [n_rows][H].
 */
int oracle_combine_rows_act(int T, int H, int F, int E, int k, int act, const uint16_t *x,
                            const uint16_t *w1, const uint16_t *w2,
                            const int32_t *ids, const float *w, const int32_t *slot,
                            int n_rows, const int32_t *rows, double *y, int nthreads);

int oracle_combine_rows(int T, int H, int F, int E, int k, const uint16_t *x,
                        const uint16_t *w1, const uint16_t *w2,
                        const int32_t *ids, const float *w, const int32_t *slot,
                        int n_rows, const int32_t *rows, double *y, int nthreads)
{
    return oracle_combine_rows_act(T, H, F, E, k, 0, x, w1, w2, ids, w, slot, n_rows, rows, y,
                                   nthreads);
}

/*
 * As oracle_combine_rows with the expert chosen by `act`: 0 = GELU FFN
 * (W1 [E][H][F]), 1 = SwiGLU (W1 [E][H][2F] = [gate | up]); W2 [E][F][H].
 */
int oracle_combine_rows_act(int T, int H, int F, int E, int k, int act, const uint16_t *x,
                            const uint16_t *w1, const uint16_t *w2,
                            const int32_t *ids, const float *w, const int32_t *slot,
                            int n_rows, const int32_t *rows, double *y, int nthreads)
{
    if (act != 0 && act != 1) return 1;
    const size_t w1_cols = (size_t)(act == 1 ? 2 : 1) * (size_t)F;
    if (T < 0 || H < 1 || F < 1 || E < 1 || k < 1 || n_rows < 0) return 1;
    if (!x || !w1 || !w2 || !ids || !w || !slot || (n_rows && (!rows || !y))) return 1;
    for (int i = 0; i < n_rows; i++)
        if (rows[i] < 0 || rows[i] >= T) return 3;
    int bad = 0;
    set_threads(nthreads);
#pragma omp parallel
    {
        double *g = (double *)malloc(sizeof(double) * w1_cols);
        double *v = (double *)malloc(sizeof(double) * (size_t)H);
        if (!g || !v) {
#pragma omp atomic write
            bad = 2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int i = 0; i < n_rows; i++) {
            if (!g || !v) continue;
            int t = rows[i];
            double *yt = y + (size_t)i * H;
            for (int h = 0; h < H; h++) yt[h] = 0.0;
            for (int j = 0; j < k; j++) {
                if (slot[(size_t)t * k + j] < 0) continue; /* dropped */
                int e = ids[(size_t)t * k + j];
                if (e < 0 || e >= E) continue;
                if (act == 1)
                    expert_swiglu_row(H, F, x + (size_t)t * H, w1 + (size_t)e * H * w1_cols,
                                      w2 + (size_t)e * F * H, g, v);
                else
                    expert_ffn_row(H, F, x + (size_t)t * H,
                                   w1 + (size_t)e * H * F, w2 + (size_t)e * F * H, g, v);
                double wt = (double)w[(size_t)t * k + j];
                for (int h = 0; h < H; h++) yt[h] += wt * v[h];
            }
        }
        free(g);
        free(v);
    }
    return bad;
}

/*
 * Step 5 on expert outputs that are given rather than computed: the expert
 * kernel's ScatterWithWeights (output(orig_pos, d) += weight * expert_out)
 * for every token t, over its kept slots j in ascending order:
 *   y[t] = sum_{j: slot[t][j] >= 0} w[t][j] * Y[slot[t][j]]
 * Y [n_Y][H] holds the expert outputs in dispatch order (bf16 bit patterns,
 * decoded exactly); the sum is in double; a token with no kept slot gets 0.
 * A slot outside [-1, n_Y) is an error (return 3).
 */
int oracle_combine_given(int T, int H, int k, int n_Y, const uint16_t *Y, const float *w,
                         const int32_t *slot, double *y)
{
    if (T < 0 || H < 1 || k < 1 || n_Y < 0 || !w || !slot || (T && !y)) return 1;
    if (n_Y && !Y) return 1;
    for (long i = 0; i < (long)T * k; i++)
        if (slot[i] < -1 || slot[i] >= n_Y) return 3;
    for (int t = 0; t < T; t++) {
        double *yt = y + (size_t)t * H;
        for (int h = 0; h < H; h++) yt[h] = 0.0;
        for (int j = 0; j < k; j++) {
            int32_t r = slot[(size_t)t * k + j];
            if (r < 0) continue; /* dropped */
            double wt = (double)w[(size_t)t * k + j];
            const uint16_t *Yr = Y + (size_t)r * H;
            for (int h = 0; h < H; h++) yt[h] += wt * bf16_value(Yr[h]);
        }
    }
    return 0;
}
