/*
 * moe_oracle.c -- plain, slow CPU oracle of one Mixture-of-Experts layer.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path never
 * calls it, and it shares no code, header or table with the CUDA library.
 *
 * What it computes.  The pages (CUCo: An Agentic Framework for Compute and
 * Communication Co-design; abstract, and Table 4 row "MoE Dispatch/Combine")
 * name a DeepSeek-V3 MoE layer whose dispatch/combine surrounds local expert
 * compute, but never write the layer's arithmetic down.  This file takes the
 * plainest reading of a DeepSeek-V3 / Mixtral MoE layer:
 *
 *   scores   logits[t,e] = sum_i x[t,i] * Wr[e,i]; softmax configs compare
 *            the logits, sigmoid configs compare s = 1/(1+exp(-logit)).
 *   select   top-k per token, ties to the lower index; sigmoid configs add a
 *            per-expert bias for selection only and may restrict the choice
 *            to the best `topk_group` of `n_group` contiguous expert groups
 *            (group score = sum of the group's two largest biased scores).
 *   gates    softmax: p = softmax over all experts, w_j = p_j / sum_sel p;
 *            sigmoid: w_j = s_j / sum_sel s; both times `routed_scale`.
 *   dispatch stable counting sort of the T*k (token, slot) pairs by expert.
 *   experts  y = W2 (silu(W1 x) * (W3 x)), SwiGLU; W13 holds W1 rows then
 *            W3 rows; h is rounded to bf16 when activations are bf16.
 *   combine  out[t] = sum_j w[t,j] * y_{e_j}(x_t)  (+ shared expert y_sh).
 *
 * Precision: every sum runs in double, in natural index order.  Decisions that
 * choose an integer (which experts win) compare fp32 values, as the kernels
 * do: the biased score s + b and the group score a + b are fp32 additions.
 * Each function below names the step it follows.  The code is written to be
 * read against that description, not to be fast: one OpenMP thread per token.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_BF16 = 1 };
enum { OR_SOFTMAX = 0, OR_SIGMOID = 1 };

/* ---- element access ---------------------------------------------------- */

static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* element i of an array that is either fp32 or bf16 (stored as raw bits) */
static double load_elem(const void* p, int dtype, size_t i) {
    if (dtype == OR_BF16) return bf16_bits_to_double(((const uint16_t*)p)[i]);
    return (double)((const float*)p)[i];
}

/* Round a double to the nearest bf16 value, ties to even, in one step (no
 * intermediate fp32 rounding).  bf16 keeps 8 significant bits and the fp32
 * exponent range; below 2^-126 its spacing is the fixed 2^-133. */
double oracle_round_bf16(double v) {
    if (!isfinite(v) || v == 0.0) return v;
    int ex;
    (void)frexp(v, &ex);               /* |v| = m * 2^ex, m in [0.5, 1) */
    int qexp = ex - 8;                 /* spacing of 8-significant-bit values */
    if (qexp < -133) qexp = -133;
    double q = ldexp(1.0, qexp);
    double r = nearbyint(v / q) * q;   /* default rounding mode: to nearest even */
    if (fabs(r) > 3.3895313892515355e38) r = copysign(INFINITY, v);
    return r;
}

static double silu(double a) { return a / (1.0 + exp(-a)); }

/* ---- step 1: scores ---------------------------------------------------- */

/* logits[t,e] = sum_i x[t,i] * Wr[e,i], summed in double, rounded to fp32.
 * Sigmoid configs store s = 1/(1+exp(-logit)) (computed in double from the
 * rounded logit) instead. */
void oracle_router_scores(const void* x, int xdtype, const float* w_router,
                          int T, int d, int E, int score_fn, float* scores) {
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i)
                acc += load_elem(x, xdtype, (size_t)t * d + i) * (double)w_router[(size_t)e * d + i];
            float logit = (float)acc;
            if (score_fn == OR_SIGMOID)
                scores[(size_t)t * E + e] = (float)(1.0 / (1.0 + exp(-(double)logit)));
            else
                scores[(size_t)t * E + e] = logit;
        }
    }
}

/* ---- step 2: selection ------------------------------------------------- */

/* Index of the largest key among candidates allowed[e] != 0, ties to the
 * lowest index (only a strictly larger key replaces the current best). */
static int argmax_lowest(const float* key, const unsigned char* allowed, int n) {
    int best = -1;
    for (int e = 0; e < n; ++e) {
        if (!allowed[e]) continue;
        if (best < 0 || key[e] > key[best]) best = e;
    }
    return best;
}

/* Experts chosen for one token, written in selection order: descending key,
 * equal keys by ascending index.  key = score (softmax, or sigmoid without
 * bias) or fp32(score + bias).  With n_group > 1 the experts are split into
 * n_group contiguous groups; each group's score is the fp32 sum of its two
 * largest keys; only the best topk_group groups (ties to the lower group)
 * stay eligible.  Returns 0, or -1 if fewer than k experts are eligible. */
static int select_one(const float* score, const float* bias, int E, int k,
                      int n_group, int topk_group, int32_t* idx_out) {
    float* key = (float*)malloc(sizeof(float) * E);
    unsigned char* allowed = (unsigned char*)malloc(E);
    int rc = 0;
    for (int e = 0; e < E; ++e) {
        key[e] = bias ? (float)(score[e] + bias[e]) : score[e];
        allowed[e] = 1;
    }
    if (n_group > 1) {
        int gs = E / n_group;
        if (gs < 2 || topk_group < 1 || topk_group > n_group || gs * n_group != E) {
            free(allowed); free(key);
            return -1;
        }
        float* gscore = (float*)malloc(sizeof(float) * n_group);
        unsigned char* gallowed = (unsigned char*)malloc(n_group);
        unsigned char* in_group = (unsigned char*)malloc(gs);
        for (int g = 0; g < n_group; ++g) {
            memset(in_group, 1, gs);
            int a = argmax_lowest(key + g * gs, in_group, gs);
            in_group[a] = 0;
            int b = argmax_lowest(key + g * gs, in_group, gs);
            gscore[g] = key[g * gs + a] + key[g * gs + b];
            gallowed[g] = 1;
        }
        unsigned char* keep = (unsigned char*)calloc(n_group, 1);
        for (int r = 0; r < topk_group; ++r) {
            int g = argmax_lowest(gscore, gallowed, n_group);
            keep[g] = 1;
            gallowed[g] = 0;
        }
        for (int e = 0; e < E; ++e) allowed[e] = keep[e / gs];
        free(keep); free(in_group); free(gallowed); free(gscore);
    }
    for (int j = 0; j < k; ++j) {
        int e = argmax_lowest(key, allowed, E);
        if (e < 0) { rc = -1; break; }
        idx_out[j] = e;
        allowed[e] = 0;
    }
    free(allowed);
    free(key);
    return rc;
}

int oracle_select(const float* scores, const float* bias, int T, int E, int k,
                  int n_group, int topk_group, int32_t* idx) {
    int bad = 0;
    #pragma omp parallel for schedule(static) reduction(|:bad)
    for (int t = 0; t < T; ++t)
        bad |= select_one(scores + (size_t)t * E, bias, E, k, n_group, topk_group,
                          idx + (size_t)t * k) != 0;
    return bad ? -1 : 0;
}

/* ---- step 3: gate weights ---------------------------------------------- */

/* softmax: p_e = exp(l_e - max) / sum_e' exp(l_e' - max) over all experts,
 *          w_j = p_{e_j} / sum_j' p_{e_j'};
 * sigmoid: w_j = s_{e_j} / sum_j' s_{e_j'}  (the bias never enters);
 * both then multiplied by routed_scale.  All in double. */
void oracle_gates(const float* scores, const int32_t* idx, int T, int E, int k,
                  int score_fn, double routed_scale, double* w) {
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        const float* s = scores + (size_t)t * E;
        const int32_t* sel = idx + (size_t)t * k;
        double* wt = w + (size_t)t * k;
        if (score_fn == OR_SOFTMAX) {
            double m = s[0];
            for (int e = 1; e < E; ++e) if (s[e] > m) m = s[e];
            double z = 0.0;
            for (int e = 0; e < E; ++e) z += exp((double)s[e] - m);
            double psum = 0.0;
            for (int j = 0; j < k; ++j) { wt[j] = exp((double)s[sel[j]] - m) / z; psum += wt[j]; }
            for (int j = 0; j < k; ++j) wt[j] = wt[j] / psum * routed_scale;
        } else {
            double ssum = 0.0;
            for (int j = 0; j < k; ++j) ssum += (double)s[sel[j]];
            for (int j = 0; j < k; ++j) wt[j] = (double)s[sel[j]] / ssum * routed_scale;
        }
    }
}

/* ---- step 4: dispatch -------------------------------------------------- */

/* Stable counting sort of slots s = t*k + j by expert idx[s]:
 *   counts[e]   = number of slots routed to e
 *   offsets[e]  = sum_{e' < e} counts[e'], offsets[E] = T*k
 *   slot_to_row[s] = offsets[e] + (number of earlier slots s' < s with e)
 *   row_to_token[slot_to_row[s]] = s / k
 * Returns -1 if an index lies outside [0, E). */
int oracle_dispatch(const int32_t* idx, int T, int k, int E, int32_t* counts,
                    int32_t* offsets, int32_t* slot_to_row, int32_t* row_to_token) {
    long S = (long)T * k;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (long s = 0; s < S; ++s) {
        if (idx[s] < 0 || idx[s] >= E) return -1;
        counts[idx[s]]++;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* next = (int32_t*)malloc(sizeof(int32_t) * (E > 0 ? E : 1));
    for (int e = 0; e < E; ++e) next[e] = offsets[e];
    for (long s = 0; s < S; ++s) {
        int32_t row = next[idx[s]]++;
        slot_to_row[s] = row;
        row_to_token[row] = (int32_t)(s / k);
    }
    free(next);
    return 0;
}

/* ---- step 5: one SwiGLU expert on one row ------------------------------ */

/* y[n] = sum_i h_i * W2[n,i],  h_i = silu(g_i) * u_i,
 * g_i = sum_c x_c * W13[i,c] (gate rows 0..I-1), u_i = sum_c x_c * W13[I+i,c]
 * (up rows I..2I-1).  h is rounded to bf16 when round_h is set. */
static void swiglu_row(const void* x, int xdtype, size_t xoff, const void* w13,
                       const void* w2, int wdtype, size_t w13off, size_t w2off,
                       int d, int I, int round_h, double* h, double* y) {
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int c = 0; c < d; ++c) {
            double xc = load_elem(x, xdtype, xoff + c);
            g += xc * load_elem(w13, wdtype, w13off + (size_t)i * d + c);
            u += xc * load_elem(w13, wdtype, w13off + (size_t)(I + i) * d + c);
        }
        double hi = silu(g) * u;
        h[i] = round_h ? oracle_round_bf16(hi) : hi;
    }
    for (int n = 0; n < d; ++n) {
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += h[i] * load_elem(w2, wdtype, w2off + (size_t)n * I + i);
        y[n] = acc;
    }
}

/* y[r] = SwiGLU_{row_expert[r]}(x[r]) for each row r; W13 [E,2I,d], W2 [E,d,I].
 * This is the per-segment expert FFN applied to already permuted rows. */
void oracle_expert_rows(const void* x, int xdtype, int n_rows, const int32_t* row_expert,
                        const void* w13, const void* w2, int wdtype, int d, int I,
                        int round_h, double* y) {
    #pragma omp parallel
    {
        double* h = (double*)malloc(sizeof(double) * (I > 0 ? I : 1));
        #pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < n_rows; ++r) {
            size_t e = (size_t)row_expert[r];
            swiglu_row(x, xdtype, (size_t)r * d, w13, w2, wdtype, e * 2 * I * d, e * d * I,
                       d, I, round_h, h, y + (size_t)r * d);
        }
        free(h);
    }
}

/* ---- step 6: combine --------------------------------------------------- */

/* out[t,:] = sum_j w[t,j] * y[slot_to_row[t*k+j], :]  (+ shared[t,:]),
 * summed in slot order in double. */
void oracle_combine(const float* y, const int32_t* slot_to_row, const float* w,
                    const float* shared, int T, int k, int d, double* out) {
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) {
                size_t row = (size_t)slot_to_row[(size_t)t * k + j];
                acc += (double)w[(size_t)t * k + j] * (double)y[row * d + c];
            }
            if (shared) acc += (double)shared[(size_t)t * d + c];
            out[(size_t)t * d + c] = acc;
        }
    }
}

/* ---- the whole layer, token by token ------------------------------------ */

/* For each of n_tok tokens independently (x rows [n_tok,d]):
 *   scores   = scores_in[t] if given, else step 1 on x[t]
 *   experts  = step 2, gates = step 3,
 *   out[t]   = sum_j w_j * SwiGLU_{e_j}(x[t]) + SwiGLU_shared(x[t]).
 * Tokens never interact, so any subset of a batch can be evaluated alone.
 * Returns 0, or -1 if some token had fewer than k eligible experts. */
int oracle_moe_tokens(const void* x, int xdtype, int n_tok, int d,
                      const float* scores_in, const float* w_router, const float* bias,
                      int E, int k, int n_group, int topk_group, int score_fn,
                      double routed_scale, const void* w13, const void* w2, int wdtype, int I,
                      const void* w13_sh, const void* w2_sh, int I_sh, int round_h,
                      int32_t* idx_out, double* w_out, double* out) {
    int bad = 0;
    int Imax = I > I_sh ? I : I_sh;
    #pragma omp parallel reduction(|:bad)
    {
        float* sc = (float*)malloc(sizeof(float) * E);
        double* h = (double*)malloc(sizeof(double) * (Imax > 0 ? Imax : 1));
        double* y = (double*)malloc(sizeof(double) * d);
        #pragma omp for schedule(dynamic, 1)
        for (int t = 0; t < n_tok; ++t) {
            size_t xoff = (size_t)t * d;
            if (scores_in) {
                memcpy(sc, scores_in + (size_t)t * E, sizeof(float) * E);
            } else {
                for (int e = 0; e < E; ++e) {
                    double acc = 0.0;
                    for (int i = 0; i < d; ++i)
                        acc += load_elem(x, xdtype, xoff + i) * (double)w_router[(size_t)e * d + i];
                    float logit = (float)acc;
                    sc[e] = score_fn == OR_SIGMOID ? (float)(1.0 / (1.0 + exp(-(double)logit))) : logit;
                }
            }
            int32_t* sel = idx_out + (size_t)t * k;
            double* wt = w_out + (size_t)t * k;
            if (select_one(sc, score_fn == OR_SIGMOID ? bias : NULL, E, k, n_group, topk_group, sel) != 0) {
                bad = 1;
                continue;
            }
            oracle_gates(sc, sel, 1, E, k, score_fn, routed_scale, wt);
            double* o = out + (size_t)t * d;
            for (int c = 0; c < d; ++c) o[c] = 0.0;
            for (int j = 0; j < k; ++j) {
                size_t e = (size_t)sel[j];
                swiglu_row(x, xdtype, xoff, w13, w2, wdtype, e * 2 * I * d, e * d * I, d, I,
                           round_h, h, y);
                for (int c = 0; c < d; ++c) o[c] += wt[j] * y[c];
            }
            if (w13_sh && w2_sh && I_sh > 0) {
                swiglu_row(x, xdtype, xoff, w13_sh, w2_sh, wdtype, 0, 0, d, I_sh, round_h, h, y);
                for (int c = 0; c < d; ++c) o[c] += y[c];
            }
        }
        free(y); free(h); free(sc);
    }
    return bad ? -1 : 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
