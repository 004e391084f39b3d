/*
 * smc_oracle.c -- plain float64 CPU oracle for the speculative-decoding verify step,
 * the SMC-SD reweight / ESS / systematic-resample / page-table steps and the PACER
 * blockwise stop rule.
 *
 * TEST INFRASTRUCTURE. Only the test-suite, the smoke check and the benchmark's CPU
 * baseline leg load this library. The CUDA library never calls it, and the two share
 * no code, header, table or constant.
 *
 * Every function below is written as the definition it follows: double arithmetic,
 * the host C library's exp/log, loops in index order, no blocking and no reordering.
 * Inputs are the same bytes the GPU reads: bf16 logits are widened exactly to double,
 * float32 uniforms and parameters are widened exactly.
 *
 * Sources (gist.science summary pages):
 *  [SMC]   "Faster LLM Inference via Sequential Monte Carlo"
 *          sec. 1 (SD verifies by rejection sampling and discards the block after the
 *          first rejection), sec. 2 steps 1-4 (N particles, K draft tokens each, one
 *          target scoring pass, importance reweighting by the target/draft probability
 *          ratio, resampling when the effective sample size drops below a threshold,
 *          exactly K+1 tokens per particle and step), sec. 3 (page-based KV cache:
 *          resampling is a metadata update only; power sampling as a modified target).
 *  [PACER] "PACER: Blockwise Pre-verification for Speculative Decoding with Adaptive
 *          Length", Methodik 1-3 (blocks of b draft tokens, mean estimated acceptance of
 *          the block against a threshold t, stop and verify the accumulated tokens,
 *          t grows by a factor rho after every successful block).
 *  [UAG]   "Cross-Family Speculative Decoding for Polish Language Models on Apple
 *          Silicon", sec. 1 (verification of k candidates in one target pass).
 * The pages print no formulas. Where they name a step without its rule, the textbook
 * rule is used, and the comment at that step says which.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_EINVAL (-1)
#define OR_EDTYPE (-2)
#define OR_ENONFINITE (-5)
#define OR_ERANGE (-6)

/* ------------------------------------------------------------------------------------ */
/* input decoding                                                                        */
/* ------------------------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE float32: widen by shifting into the high 16 bits. */
static double bf16_bits_to_double(uint16_t bits) {
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* Logit `i` of a [rows, V] row-major buffer; dtype 0 = float32, 1 = bf16. */
static double logit_at(const void* base, int dtype, long long i) {
    if (dtype == 0) return (double)((const float*)base)[i];
    return bf16_bits_to_double(((const uint16_t*)base)[i]);
}

/* ------------------------------------------------------------------------------------ */
/* step 1: scaled log-softmax normaliser                                                 */
/* ------------------------------------------------------------------------------------ */

/*
 * [SMC] sec. 2 step 3 weighs particles by target versus draft *probabilities*, so both
 * rows are turned into normalised distributions.  Row scores are s_i = scale * z_i with
 * scale = alpha / T (alpha = 1 except for the power target of sec. 3, T the sampling
 * temperature), and
 *     L = m + log( sum_i exp(s_i - m) ),   m = max_i s_i,
 * summed in index order.  -inf logits are masked tokens (exp gives 0).  NaN or +inf in
 * a row, or a row of nothing but -inf, is reported as OR_ENONFINITE.
 */
int oracle_row_lse(const void* logits, int dtype, long long row, int V, double scale,
                   double* L_out) {
    if (!logits || !L_out || V <= 0 || !(scale > 0.0) || isinf(scale)) return OR_EINVAL;
    if (dtype != 0 && dtype != 1) return OR_EDTYPE;
    const long long base = row * (long long)V;
    double m = -INFINITY;
    for (int i = 0; i < V; ++i) {
        double s = scale * logit_at(logits, dtype, base + i);
        if (isnan(s) || s == INFINITY) return OR_ENONFINITE;
        if (s > m) m = s;
    }
    if (m == -INFINITY) return OR_ENONFINITE;
    double sum = 0.0;
    for (int i = 0; i < V; ++i) {
        double s = scale * logit_at(logits, dtype, base + i);
        sum += exp(s - m);
    }
    *L_out = m + log(sum);
    return OR_OK;
}

/* log-probability of token x in a row with normaliser L */
static double row_logprob(const void* logits, int dtype, long long row, int V, double scale,
                          double L, int x) {
    return scale * logit_at(logits, dtype, row * (long long)V + x) - L;
}

/* ------------------------------------------------------------------------------------ */
/* inverse-CDF draw                                                                      */
/* ------------------------------------------------------------------------------------ */

/*
 * Draw from unnormalised non-negative weights r[0..V) with one uniform u in [0,1):
 *     R = sum_i r_i,   token = min{ i : sum_{j<=i} r_j > u * R }     (strict ">")
 * If rounding leaves no such i, the last index with r_i > 0 is taken.  The margin is the
 * distance of u*R to the nearer end of the chosen token's interval, divided by R.
 * Returns OR_EINVAL if R is not positive.
 */
int oracle_sample_inverse_cdf(const double* r, int V, double u, int* token_out,
                              double* margin_out) {
    if (!r || !token_out || V <= 0) return OR_EINVAL;
    double R = 0.0;
    for (int i = 0; i < V; ++i) R += r[i];
    if (!(R > 0.0)) return OR_EINVAL;
    const double target = u * R;
    double C = 0.0, C_prev = 0.0;
    int tok = -1;
    for (int i = 0; i < V; ++i) {
        C_prev = C;
        C += r[i];
        if (C > target) { tok = i; break; }
    }
    if (tok < 0) {
        /* rounding fallback: last index with positive weight, interval [C - r, C] */
        for (int i = V - 1; i >= 0; --i)
            if (r[i] > 0.0) { tok = i; break; }
        C = R;
        C_prev = R - r[tok];
    }
    *token_out = tok;
    if (margin_out) {
        double a = target - C_prev, b = C - target;
        *margin_out = (a < b ? a : b) / R;
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------------------ */
/* speculative-decoding verify                                                           */
/* ------------------------------------------------------------------------------------ */

/*
 * SD verify for S sequences ([SMC] sec. 1; [UAG] sec. 1; ragged lengths from [PACER]
 * Methodik 2).
 *
 * Rows: target logits hold K_s+1 rows per sequence, draft logits K_s rows.  Fixed
 * layout (offsets NULL): K_s = K, target rows s*(K+1)+k, draft rows s*K+k, draft token
 * draft_tokens[s*K+k].  Ragged layout: target rows tgt_offsets[s]..tgt_offsets[s+1]-1,
 * draft rows (and draft tokens) drf_offsets[s]..drf_offsets[s+1]-1, with
 * K_s = drf_offsets[s+1]-drf_offsets[s] = tgt_offsets[s+1]-tgt_offsets[s]-1 <= K.
 * Both models use the same temperature T: p = softmax(z_t/T), q = softmax(z_d/T).
 *
 * The pages only say "rejection sampling" and that the block is discarded at the first
 * rejection.  The rule applied is the textbook one:
 *   accept draft x_k iff u[s*(K+1)+k] < min(1, p_k(x_k)/q_k(x_k)), tested in k order;
 *   acc = first rejected k, or K_s if none is rejected;
 *   acc < K_s : out_token ~ normalise(max(0, p_acc - q_acc)) with u[s*(K+1)+K];
 *   acc = K_s : out_token ~ p_{K_s} (bonus token) with u[s*(K+1)+K].
 * If the residual has zero mass (only possible through rounding), the draw falls back to
 * p at the same row.
 *
 * Outputs: accept_len[S], out_token[S]; optional (NULL allowed): lse_tgt / lse_drf per
 * row (double, natural log, scaled logits), accept_margin[S*K] (|u - ratio| for every
 * test that was made, -1 for tests not made), token_margin[S].
 */
int oracle_sd_verify(const void* tgt, const void* drf, int dtype, const int32_t* draft_tokens,
                     const int32_t* tgt_offsets, const int32_t* drf_offsets, int S, int K, int V,
                     float temperature, const float* uniforms, int32_t* accept_len,
                     int32_t* out_token, double* lse_tgt, double* lse_drf,
                     double* accept_margin, double* token_margin) {
    if (!tgt || !drf || !draft_tokens || !uniforms || !accept_len || !out_token) return OR_EINVAL;
    if (S <= 0 || K < 0 || V <= 0) return OR_EINVAL;
    if (!(temperature > 0.0f) || isinf(temperature)) return OR_EINVAL;
    if ((tgt_offsets == NULL) != (drf_offsets == NULL)) return OR_EINVAL;
    if (dtype != 0 && dtype != 1) return OR_EDTYPE;
    const int ragged = tgt_offsets != NULL;
    const double scale = 1.0 / (double)temperature;

    /* validate the ragged layout before touching any row */
    if (ragged) {
        for (int s = 0; s < S; ++s) {
            int nt = tgt_offsets[s + 1] - tgt_offsets[s];
            int nd = drf_offsets[s + 1] - drf_offsets[s];
            if (tgt_offsets[s] < 0 || drf_offsets[s] < 0 || nd < 0 || nd > K || nt != nd + 1)
                return OR_ERANGE;
        }
    }

    double* r = (double*)malloc(sizeof(double) * (size_t)V);
    if (!r) return OR_EINVAL;
    int rc = OR_OK;

    for (int s = 0; s < S && rc == OR_OK; ++s) {
        const int Ks = ragged ? drf_offsets[s + 1] - drf_offsets[s] : K;
        const long long trow0 = ragged ? tgt_offsets[s] : (long long)s * (K + 1);
        const long long drow0 = ragged ? drf_offsets[s] : (long long)s * K;
        const float* u = uniforms + (long long)s * (K + 1);

        /* normalisers of every row of this sequence */
        double Lt_row[64 + 1], Ld_row[64];
        double *Lt = Lt_row, *Ld = Ld_row;
        double* heap = NULL;
        if (Ks > 64) {
            heap = (double*)malloc(sizeof(double) * (size_t)(2 * Ks + 1));
            if (!heap) { rc = OR_EINVAL; break; }
            Lt = heap;
            Ld = heap + Ks + 1;
        }
        for (int k = 0; k <= Ks && rc == OR_OK; ++k) {
            rc = oracle_row_lse(tgt, dtype, trow0 + k, V, scale, &Lt[k]);
            if (rc == OR_OK && lse_tgt) lse_tgt[trow0 + k] = Lt[k];
        }
        for (int k = 0; k < Ks && rc == OR_OK; ++k) {
            rc = oracle_row_lse(drf, dtype, drow0 + k, V, scale, &Ld[k]);
            if (rc == OR_OK && lse_drf) lse_drf[drow0 + k] = Ld[k];
        }
        if (rc != OR_OK) { free(heap); break; }

        /* accept tests in position order, stop at the first rejection */
        int acc = Ks;
        for (int k = 0; k < Ks; ++k) {
            if (accept_margin) accept_margin[(long long)s * K + k] = -1.0;
        }
        for (int k = 0; k < Ks; ++k) {
            const int x = draft_tokens[drow0 + k];
            if (x < 0 || x >= V) { rc = OR_ERANGE; break; }
            double lp = row_logprob(tgt, dtype, trow0 + k, V, scale, Lt[k], x);
            double lq = row_logprob(drf, dtype, drow0 + k, V, scale, Ld[k], x);
            double ell = lp - lq;
            double a = exp(ell < 0.0 ? ell : 0.0); /* min(1, p/q) */
            double uk = (double)u[k];
            if (accept_margin) accept_margin[(long long)s * K + k] = fabs(uk - a);
            if (!(uk < a)) { acc = k; break; }
        }
        if (rc != OR_OK) { free(heap); break; }
        accept_len[s] = acc;

        /* final draw: residual at the rejected position, or bonus from the last row */
        const double uf = (double)u[K];
        int tok = 0;
        double marg = 0.0;
        int drawn = 0;
        if (acc < Ks) {
            const long long tr = trow0 + acc, dr = drow0 + acc;
            for (int i = 0; i < V; ++i) {
                double p = exp(scale * logit_at(tgt, dtype, tr * V + i) - Lt[acc]);
                double q = exp(scale * logit_at(drf, dtype, dr * V + i) - Ld[acc]);
                double d = p - q;
                r[i] = d > 0.0 ? d : 0.0;
            }
            if (oracle_sample_inverse_cdf(r, V, uf, &tok, &marg) == OR_OK) drawn = 1;
        }
        if (!drawn) {
            const int row = acc; /* acc == Ks: bonus row; else zero-mass residual fallback */
            const long long tr = trow0 + row;
            for (int i = 0; i < V; ++i)
                r[i] = exp(scale * logit_at(tgt, dtype, tr * V + i) - Lt[row]);
            if (oracle_sample_inverse_cdf(r, V, uf, &tok, &marg) != OR_OK) rc = OR_ENONFINITE;
        }
        out_token[s] = tok;
        if (token_margin) token_margin[s] = marg;
        free(heap);
    }
    free(r);
    return rc;
}

/* ------------------------------------------------------------------------------------ */
/* SMC-SD reweight and bonus token                                                       */
/* ------------------------------------------------------------------------------------ */

/*
 * [SMC] sec. 2 step 3: each particle's weight is updated by the ratio of target to draft
 * probability of its K draft tokens, in log space.  [SMC] sec. 3 ("flexibility") names
 * modified targets, power sampling and reward-weighted decoding, and sec. 5
 * ("extensibility") reward optimisation and hard constraints through the same importance
 * weights; two readings of a power target are offered (target_mode):
 *
 *  0 (per position): pi = softmax(alpha * z_t / T) at every position (alpha = 1 is the
 *    plain target p; alpha != 1 is p^alpha renormalised per position), q = softmax(z_d/T):
 *        logw_s += sum_{k<K} ( log pi_k(x_k) - log q_k(x_k) );
 *    the (K+1)-th token ([SMC] sec. 2 "exactly K+1 tokens per particle") is drawn from pi
 *    at target row K with uniforms[s]; its weight factor pi/pi is 1, so it adds nothing.
 *
 *  1 (whole sequence): the target is the unnormalised power of the sequence probability,
 *    gamma(x) = prod_t p_t(x_t)^alpha with p = softmax(z_t / T).  Importance sampling of
 *    gamma under the proposals used (q for the draft tokens, p for the (K+1)-th token)
 *    gives
 *        logw_s += sum_{k<K} ( alpha * log p_k(x_k) - log q_k(x_k) )
 *                  + (alpha - 1) * log p_K(b_s),
 *    where b_s is drawn from p at target row K with uniforms[s].  alpha = 1 gives the same
 *    result as mode 0.
 *
 * In both modes, when log_reward is given, logw_s += reward_scale * log_reward[s] (an
 * additive log-potential per particle; a NaN or infinite reward is OR_ENONFINITE).
 *
 * Layout: target rows s*(K+1)+k, draft rows s*K+k, draft_tokens[s*K+k].
 * logw is float32 in/out: the update is done in double and rounded once on store.
 * Optional outputs: lse_tgt[S*(K+1)] (normalisers at the target's scale: alpha/T in mode 0,
 * 1/T in mode 1), lse_drf[S*K], bonus_margin[S], dlogw[S] (the double increment before
 * rounding).
 */
int oracle_smc_reweight_tilted(const void* tgt, const void* drf, int dtype,
                               const int32_t* draft_tokens, int S, int K, int V,
                               float temperature, float alpha, int target_mode,
                               const float* log_reward, float reward_scale,
                               const float* uniforms, float* logw, int32_t* bonus_token,
                               double* lse_tgt, double* lse_drf, double* bonus_margin,
                               double* dlogw) {
    if (!tgt || !drf || !uniforms || !logw || !bonus_token) return OR_EINVAL;
    if (K > 0 && !draft_tokens) return OR_EINVAL;
    if (S <= 0 || K < 0 || V <= 0) return OR_EINVAL;
    if (!(temperature > 0.0f) || isinf(temperature)) return OR_EINVAL;
    if (!(alpha > 0.0f) || isinf(alpha)) return OR_EINVAL;
    if (target_mode != 0 && target_mode != 1) return OR_EINVAL;
    if (log_reward && (isnan(reward_scale) || isinf(reward_scale))) return OR_EINVAL;
    if (dtype != 0 && dtype != 1) return OR_EDTYPE;
    const double a = (double)alpha;
    const double scale_t = target_mode == 0 ? a / (double)temperature : 1.0 / (double)temperature;
    const double scale_d = 1.0 / (double)temperature;
    const double w_t = target_mode == 0 ? 1.0 : a; /* factor on log p of a draft token */

    double* r = (double*)malloc(sizeof(double) * (size_t)V);
    if (!r) return OR_EINVAL;
    int rc = OR_OK;
    for (int s = 0; s < S && rc == OR_OK; ++s) {
        double inc = 0.0;
        for (int k = 0; k < K && rc == OR_OK; ++k) {
            const long long tr = (long long)s * (K + 1) + k, dr = (long long)s * K + k;
            double Lt, Ld;
            rc = oracle_row_lse(tgt, dtype, tr, V, scale_t, &Lt);
            if (rc == OR_OK) rc = oracle_row_lse(drf, dtype, dr, V, scale_d, &Ld);
            if (rc != OR_OK) break;
            if (lse_tgt) lse_tgt[tr] = Lt;
            if (lse_drf) lse_drf[dr] = Ld;
            const int x = draft_tokens[dr];
            if (x < 0 || x >= V) { rc = OR_ERANGE; break; }
            const double lp = row_logprob(tgt, dtype, tr, V, scale_t, Lt, x);
            const double lq = row_logprob(drf, dtype, dr, V, scale_d, Ld, x);
            inc += target_mode == 0 ? lp - lq : w_t * lp - lq;
        }
        if (rc != OR_OK) break;

        /* (K+1)-th token from the target's row K at its scale */
        const long long tr = (long long)s * (K + 1) + K;
        double LK;
        rc = oracle_row_lse(tgt, dtype, tr, V, scale_t, &LK);
        if (rc != OR_OK) break;
        if (lse_tgt) lse_tgt[tr] = LK;
        for (int i = 0; i < V; ++i) r[i] = exp(scale_t * logit_at(tgt, dtype, tr * V + i) - LK);
        int tok;
        double marg;
        if (oracle_sample_inverse_cdf(r, V, (double)uniforms[s], &tok, &marg) != OR_OK) {
            rc = OR_ENONFINITE;
            break;
        }
        bonus_token[s] = tok;
        if (bonus_margin) bonus_margin[s] = marg;
        if (target_mode == 1)
            inc += (a - 1.0) * row_logprob(tgt, dtype, tr, V, scale_t, LK, tok);

        if (log_reward) {
            const double rw = (double)log_reward[s];
            if (isnan(rw) || isinf(rw)) { rc = OR_ENONFINITE; break; }
            inc += (double)reward_scale * rw;
        }
        if (dlogw) dlogw[s] = inc;
        logw[s] = (float)((double)logw[s] + inc);
    }
    free(r);
    return rc;
}

/* The per-position target of mode 0 above, without a reward term. */
int oracle_smc_reweight(const void* tgt, const void* drf, int dtype, const int32_t* draft_tokens,
                        int S, int K, int V, float temperature, float alpha,
                        const float* uniforms, float* logw, int32_t* bonus_token,
                        double* lse_tgt, double* lse_drf, double* bonus_margin,
                        double* dlogw) {
    return oracle_smc_reweight_tilted(tgt, drf, dtype, draft_tokens, S, K, V, temperature, alpha,
                                      0, NULL, 0.0f, uniforms, logw, bonus_token, lse_tgt,
                                      lse_drf, bonus_margin, dlogw);
}

/* ------------------------------------------------------------------------------------ */
/* draft-token sampling                                                                  */
/* ------------------------------------------------------------------------------------ */

/*
 * [SMC] sec. 2 step 1: the draft model proposes K tokens per particle; each is drawn from
 * the draft's tempered distribution q = softmax(z_d / T) at its position.  For R draft
 * rows (row r of a [R, V] buffer) with one uniform each:
 *     L_r = log sum_i exp(z_{r,i} / T),   q_r(i) = exp(z_{r,i} / T - L_r),
 *     token[r] = min{ i : sum_{j<=i} q_r(j) > u_r }      (the inverse-CDF draw above),
 *     logq[r]  = z_{r,token} / T - L_r   (what the verify needs from the draft side).
 * Optional outputs: logq[R], lse[R], margin[R] (as oracle_sample_inverse_cdf).
 */
int oracle_draft_sample(const void* logits, int dtype, int R, int V, float temperature,
                        const float* uniforms, int32_t* tokens, double* logq, double* lse,
                        double* margin) {
    if (!logits || !uniforms || !tokens || R <= 0 || V <= 0) return OR_EINVAL;
    if (!(temperature > 0.0f) || isinf(temperature)) return OR_EINVAL;
    if (dtype != 0 && dtype != 1) return OR_EDTYPE;
    const double scale = 1.0 / (double)temperature;
    double* r = (double*)malloc(sizeof(double) * (size_t)V);
    if (!r) return OR_EINVAL;
    int rc = OR_OK;
    for (int row = 0; row < R && rc == OR_OK; ++row) {
        double L;
        rc = oracle_row_lse(logits, dtype, row, V, scale, &L);
        if (rc != OR_OK) break;
        for (int i = 0; i < V; ++i)
            r[i] = exp(scale * logit_at(logits, dtype, (long long)row * V + i) - L);
        int tok;
        double marg;
        if (oracle_sample_inverse_cdf(r, V, (double)uniforms[row], &tok, &marg) != OR_OK) {
            rc = OR_ENONFINITE;
            break;
        }
        tokens[row] = tok;
        if (logq) logq[row] = row_logprob(logits, dtype, row, V, scale, L, tok);
        if (lse) lse[row] = L;
        if (margin) margin[row] = marg;
    }
    free(r);
    return rc;
}

/* ------------------------------------------------------------------------------------ */
/* effective sample size and systematic resampling                                       */
/* ------------------------------------------------------------------------------------ */

/*
 * [SMC] sec. 2 step 4: when the effective sample size of a prompt's N particles falls
 * below a threshold, low-weight particles are dropped and high-weight ones duplicated.
 * The pages name neither the ESS formula nor the scheme; the textbook forms are used:
 *   per group g:  M = max_i logw_i,  w_i = exp(logw_i - M),  ESS = (sum w)^2 / sum w^2;
 *   resample iff ESS < threshold (strict: "falls below");
 *   systematic resampling:  C_i = (sum_{j<=i} w_j) / W,  C_{N-1} := 1,
 *                           v_j = (j + U_g) / N,  a_j = min{ i : C_i > v_j },
 *   after which the group's log-weights are reset to 0.
 *   Without resampling a_j = j and logw is unchanged.
 * Ancestors are group-local indices in [0, N).
 * Optional outputs: ess_margin[G] = |ESS - thr| / N; anc_margin[G*N] = min_i |C_i - v_j|
 * (-1 where no resampling happened).
 */
int oracle_ess_resample(float* logw, int G, int N, float ess_threshold, const float* uniforms,
                        int32_t* ancestors, float* ess_out, int32_t* resampled,
                        double* ess_margin, double* anc_margin) {
    if (!logw || !uniforms || !ancestors || G <= 0 || N <= 0) return OR_EINVAL;
    if (isnan(ess_threshold)) return OR_EINVAL;
    double* w = (double*)malloc(sizeof(double) * (size_t)N);
    double* C = (double*)malloc(sizeof(double) * (size_t)N);
    if (!w || !C) { free(w); free(C); return OR_EINVAL; }
    int rc = OR_OK;
    for (int g = 0; g < G; ++g) {
        float* lw = logw + (long long)g * N;
        double M = -INFINITY;
        for (int i = 0; i < N; ++i) {
            double v = (double)lw[i];
            if (isnan(v) || v == INFINITY) { rc = OR_ENONFINITE; break; }
            if (v > M) M = v;
        }
        if (rc == OR_OK && M == -INFINITY) rc = OR_ENONFINITE;
        if (rc != OR_OK) break;
        double W = 0.0, W2 = 0.0;
        for (int i = 0; i < N; ++i) {
            w[i] = exp((double)lw[i] - M);
            W += w[i];
            W2 += w[i] * w[i];
        }
        const double ess = W * W / W2;
        if (ess_out) ess_out[g] = (float)ess;
        if (ess_margin) ess_margin[g] = fabs(ess - (double)ess_threshold) / N;
        const int do_resample = ess < (double)ess_threshold;
        if (resampled) resampled[g] = do_resample;
        if (!do_resample) {
            for (int j = 0; j < N; ++j) {
                ancestors[(long long)g * N + j] = j;
                if (anc_margin) anc_margin[(long long)g * N + j] = -1.0;
            }
            continue;
        }
        double acc = 0.0;
        for (int i = 0; i < N; ++i) {
            acc += w[i];
            C[i] = acc / W;
        }
        C[N - 1] = 1.0;
        const double U = (double)uniforms[g];
        for (int j = 0; j < N; ++j) {
            const double v = ((double)j + U) / (double)N;
            int a = N - 1;
            for (int i = 0; i < N; ++i)
                if (C[i] > v) { a = i; break; }
            ancestors[(long long)g * N + j] = a;
            if (anc_margin) {
                double mm = INFINITY;
                for (int i = 0; i < N; ++i) {
                    double d = fabs(C[i] - v);
                    if (d < mm) mm = d;
                }
                anc_margin[(long long)g * N + j] = mm;
            }
        }
        for (int i = 0; i < N; ++i) lw[i] = 0.0f;
    }
    free(w);
    free(C);
    return rc;
}

/* ------------------------------------------------------------------------------------ */
/* paged-KV page-table remap                                                             */
/* ------------------------------------------------------------------------------------ */

/*
 * [SMC] sec. 3: with page-based KV management, resampling moves no KV data; only
 * metadata changes.  Child j of group g takes its ancestor's page list:
 *     table_out[g*N+j][:] = table_in[g*N+a_j][:]   (identity where the group did not
 *                                                  resample; resampled may be NULL = all)
 * and, when refcount is given, refcount[p] = number of entries of table_out equal to p.
 * Entries equal to -1 are empty slots: copied, never counted.  Any other entry outside
 * [0, num_pages), or an ancestor outside [0, N), is OR_ERANGE.
 */
int oracle_pagetable_remap(const int32_t* ancestors, const int32_t* resampled, int G, int N,
                           const int32_t* table_in, int32_t* table_out, int pages_per_seq,
                           int32_t* refcount, int num_pages) {
    if (!ancestors || !table_in || !table_out || G <= 0 || N <= 0 || pages_per_seq <= 0)
        return OR_EINVAL;
    if (refcount && num_pages <= 0) return OR_EINVAL;
    for (int g = 0; g < G; ++g) {
        const int moved = resampled ? resampled[g] != 0 : 1;
        for (int j = 0; j < N; ++j) {
            int a = moved ? ancestors[(long long)g * N + j] : j;
            if (a < 0 || a >= N) return OR_ERANGE;
            const int32_t* src = table_in + ((long long)g * N + a) * pages_per_seq;
            int32_t* dst = table_out + ((long long)g * N + j) * pages_per_seq;
            for (int p = 0; p < pages_per_seq; ++p) dst[p] = src[p];
        }
    }
    if (refcount) {
        for (int p = 0; p < num_pages; ++p) refcount[p] = 0;
        const long long n = (long long)G * N * pages_per_seq;
        for (long long i = 0; i < n; ++i) {
            int32_t id = table_out[i];
            if (id == -1) continue;
            if (id < 0 || id >= num_pages) return OR_ERANGE;
            refcount[id] += 1;
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------------------ */
/* PACER blockwise stop                                                                  */
/* ------------------------------------------------------------------------------------ */

/*
 * [PACER] Methodik 1-3.  The draft produces blocks of b tokens; a pre-verification layer
 * estimates each token's acceptance from its hidden state; drafting stops when the mean
 * estimate of a block falls below a threshold t, and the accumulated tokens (the block
 * that stopped included) go to verification; after every block that passes, t is
 * multiplied by rho.  The pre-verification layer is modelled as a logistic head,
 *     score_j = 1 / (1 + exp(-(sum_d w_d h_{j,d} + c))).
 *   t = t0;  for block i = 0..max_blocks-1:
 *       m_i = (1/b) sum_{j in block i} score_j;
 *       if m_i < t: length = (i+1)*b, stop;  else t = t * rho;
 *   no stop: length = max_blocks * b.
 * The layer reads the block's hidden states together with position embeddings
 * (Methodik 1; the ablation in "Ergebnisse" finds them essential).  With a position
 * embedding table e (bf16 [max_blocks*b, d], row j for draft position j of every
 * sequence) the head's input is h_j + e_j:
 *     score_j = 1 / (1 + exp(-(sum_d w_d (h_{j,d} + e_{j,d}) + c))),
 * and without one (pos_emb NULL) it is h_j alone.
 * hidden: bf16 [S, max_blocks*b, d]; w: bf16 [d].  block_scores[S*max_blocks] (optional)
 * receives m_i for scored blocks and -1 for blocks after the stop; margin[S] (optional)
 * receives min_i |m_i - t_i| over the comparisons made that decide the length: the last
 * block's comparison is left out, since stopping there and passing there both give
 * max_blocks*b (INFINITY when no comparison decides it).
 */
int oracle_pacer_block_stop_pos(const uint16_t* hidden, const uint16_t* w,
                                const uint16_t* pos_emb, float c, int S, int b, int max_blocks,
                                int d, float t0, float rho, int32_t* lengths,
                                double* block_scores, double* margin) {
    if (!hidden || !w || !lengths || S <= 0 || b <= 0 || max_blocks <= 0 || d <= 0)
        return OR_EINVAL;
    if (isnan(c) || isinf(c) || isnan(t0) || isinf(t0) || !(rho > 0.0f) || isinf(rho))
        return OR_EINVAL;
    const int P = max_blocks * b;
    for (int s = 0; s < S; ++s) {
        double t = (double)t0;
        int len = max_blocks * b;
        double mm = INFINITY;
        int stopped = 0;
        for (int i = 0; i < max_blocks; ++i) {
            if (stopped) {
                if (block_scores) block_scores[(long long)s * max_blocks + i] = -1.0;
                continue;
            }
            double msum = 0.0;
            for (int j = i * b; j < (i + 1) * b; ++j) {
                const uint16_t* h = hidden + ((long long)s * P + j) * d;
                const uint16_t* e = pos_emb ? pos_emb + (long long)j * d : NULL;
                double dot = 0.0;
                for (int k = 0; k < d; ++k) {
                    /* h + e of two bf16 values is exact in double */
                    const double x = e ? bf16_bits_to_double(h[k]) + bf16_bits_to_double(e[k])
                                       : bf16_bits_to_double(h[k]);
                    dot += bf16_bits_to_double(w[k]) * x;
                }
                double a = dot + (double)c;
                if (isnan(a)) return OR_ENONFINITE;
                msum += 1.0 / (1.0 + exp(-a));
            }
            const double mi = msum / (double)b;
            if (block_scores) block_scores[(long long)s * max_blocks + i] = mi;
            double dm = fabs(mi - t);
            if (i < max_blocks - 1 && dm < mm) mm = dm;
            if (mi < t) {
                len = (i + 1) * b;
                stopped = 1;
            } else {
                t = t * (double)rho;
            }
        }
        lengths[s] = len;
        if (margin) margin[s] = mm;
    }
    return OR_OK;
}

/* The stop rule above without position embeddings. */
int oracle_pacer_block_stop(const uint16_t* hidden, const uint16_t* w, float c, int S, int b,
                            int max_blocks, int d, float t0, float rho, int32_t* lengths,
                            double* block_scores, double* margin) {
    return oracle_pacer_block_stop_pos(hidden, w, NULL, c, S, b, max_blocks, d, t0, rho, lengths,
                                       block_scores, margin);
}
