/*
 * svpa_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU restatement of the verification step of
 * speculative decoding over a paged KV cache.  It exists to check the CUDA
 * library; nothing in the product path may link or call it.  It shares no
 * code, header or constant with the CUDA sources.
 *
 * Precision: every attention quantity is fp64, computed from the stored bf16
 * or FP8-E4M3 bits.  The draft/target acceptance test is the one fp32 step (a
 * single rounded fp32 multiply u*Q compared with P); residual sums and CDFs
 * are fp64.  Compile with -ffp-contract=off so that no multiply-add is fused.
 *
 * Sources (page title, section / equation):
 *  - "The Sub-Millisecond Speculative Decoding Meltdown" (atozofsoftwareengineering
 *    blog), section "Speculative Decoding Mechanics & The K-Token Penalty",
 *    equation A_speculative = Softmax((Q K^T + M_tree)/sqrt(d_k)) V; section
 *    "Triton CUDA Fused Speculative Tree-Verification Kernel" (block-table
 *    lookup per page, K/V cache layout [blocks, heads, block_size, dim],
 *    per-block per-head K/V scales); section "Custom FP8 Quantized Memory
 *    Block Layout" (e4m3 pages with per-block scale factors).
 *  - "LOW-LATENCY INFERENCE: SPECULATIVE DECODING & PAGING" (innvotechnologies),
 *    section "Verification Acceptance Probabilities and Speedup Math"
 *    (alpha_i = min(1, P(x_i)/Q(x_i)), E[K], eta) and the architecture diagram
 *    (commit to block table on accept; discard KV blocks and resample on reject).
 *  - "Speculative Decoding & KV-Cache PagedAttention in Enterprise LLM Serving"
 *    (paurushmuley.com), PagedKVCacheManager: reference counts, release of a
 *    block to the free pool when its count reaches zero, block size 16.
 *  - "Speculative Decoding and KV-Cache Compression" (futurestack.online),
 *    section 2.2/2.3 (exact target distribution; the bundle's K/V is present
 *    before any acceptance decision).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  resample from normalise(max(0, P_k - Q_k)); bonus token from P at position
 *  gamma when every draft is accepted; inverse-CDF pick = first t whose
 *  cumulative mass exceeds u*S (strict); accept iff fp32(u*Q) <= P; a draw
 *  within 1e-6 of a CDF boundary is flagged; new committed length after the
 *  step = L + k + 1; tree acceptance by recursive residual rejection over a
 *  node's children in index order; the logits front-end takes one
 *  temperature for the target rows and one for the draft rows, and flags
 *  decisions within 5e-5 of their thresholds (the fp32 formation of P, Q).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_BAD_BLOCK 5
#define ORC_ERR_OUT_OF_BLOCKS 4

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t bits) {
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* OCP 8-bit floating point, E4M3 ("fn") variant: 1 sign bit, 4 exponent bits
 * with bias 7, 3 mantissa bits; exponent field 0 is subnormal
 * (m/8 * 2^(1-7)); there is no infinity; S.1111.111 is NaN; the largest
 * finite magnitude is S.1111.110 = 1.75 * 2^8 = 448. */
double oracle_e4m3_to_double(uint8_t byte) {
    int s = (byte >> 7) & 1;
    int e = (byte >> 3) & 15;
    int m = byte & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, 1 - 7);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

static int set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ */
/* paged verification attention                                        */
/* ------------------------------------------------------------------ */

/*
 * For every sequence b, query j (0..n_q-1) and query head h:
 *   the queries sit at positions L_b .. L_b+n_q-1 (their K/V are already in
 *   the pool); the positions present are p < T_b = L_b + n_q;
 *   K[p], V[p] come from physical block block_table[b][p / BS], slot p % BS;
 *   FP8 pools decode each byte and multiply by the (block, kv head) scale;
 *   query j sees every p < L_b, and a speculative slot p = L_b + i (i < n_q)
 *   when i is an ancestor of j or j itself (bit i of ancestor_mask[j]);
 *   with no mask, i <= j (causal);
 *   s_p = (q_j . K[p]) * sm_scale;  w = softmax over the visible p;
 *   out[b][j][h] = sum_p w_p V[p];  lse = log(sum_p exp(s_p)).
 * The kv head of query head h is h / (Hq / Hkv).
 * Inputs: q bf16 bits [B, n_q, Hq, D]; k_pool, v_pool [num_blocks, Hkv, BS, D]
 * of bf16 bits (kv_fp8 == 0) or E4M3 bytes (kv_fp8 != 0); k_scale, v_scale
 * fp32 (FP8 only): kv_fp8 == 1, one per (block, kv head), [num_blocks, Hkv];
 * kv_fp8 == 2, one per 64 consecutive elements of a token's row ("The
 * Sub-Millisecond Speculative Decoding Meltdown", implementation checklist:
 * block scales per 64-element tile), [num_blocks, Hkv, BS, D / 64];
 * block_table int32 [B, max_blocks];
 * context_lens int32 [B]; ancestor_mask uint64 [n_q] or NULL.
 * Outputs: out fp64 [B, n_q, Hq, D]; lse fp64 [B, n_q, Hq] (may be NULL).
 */
int oracle_paged_verify_attn(int B, int n_q, int Hq, int Hkv, int D, int BS,
                             int max_blocks, int num_blocks, int kv_fp8,
                             double sm_scale, const uint16_t *q,
                             const void *k_pool, const void *v_pool,
                             const float *k_scale, const float *v_scale,
                             const int32_t *block_table,
                             const int32_t *context_lens,
                             const uint64_t *ancestor_mask, double *out,
                             double *lse, int nthreads) {
    if (B < 0 || n_q < 1 || n_q > 64 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 ||
        D < 1 || BS < 1 || max_blocks < 1 || num_blocks < 1)
        return ORC_ERR_ARG;
    if (kv_fp8 && (!k_scale || !v_scale)) return ORC_ERR_ARG;
    if (kv_fp8 < 0 || kv_fp8 > 2 || (kv_fp8 == 2 && D % 64 != 0)) return ORC_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        long T = (long)context_lens[b] + n_q;
        if (context_lens[b] < 0 || (T + BS - 1) / BS > max_blocks) return ORC_ERR_ARG;
        for (long i = 0; i < (T + BS - 1) / BS; ++i) {
            int32_t blk = block_table[(long)b * max_blocks + i];
            if (blk < 0 || blk >= num_blocks) return ORC_ERR_BAD_BLOCK;
        }
    }
    const int G = Hq / Hkv;
    set_threads(nthreads);
    long units = (long)B * Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (long unit = 0; unit < units; ++unit) {
        int b = (int)(unit / Hkv), g = (int)(unit % Hkv);
        long L = context_lens[b];
        long T = L + n_q;
        /* 1. gather this (sequence, kv head)'s history into contiguous fp64 */
        double *K = (double *)malloc(sizeof(double) * (size_t)(T * D + 1));
        double *V = (double *)malloc(sizeof(double) * (size_t)(T * D + 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(T + 1));
        for (long p = 0; p < T; ++p) {
            int32_t blk = block_table[(long)b * max_blocks + p / BS];
            long slot = p % BS;
            long base = (((long)blk * Hkv + g) * BS + slot) * D;
            for (int d = 0; d < D; ++d) {
                if (kv_fp8) {
                    const uint8_t *kp = (const uint8_t *)k_pool;
                    const uint8_t *vp = (const uint8_t *)v_pool;
                    /* scale of this element: its (block, kv head), or its 64-element tile */
                    const long si = kv_fp8 == 1 ? (long)blk * Hkv + g
                                                : (((long)blk * Hkv + g) * BS + slot) * (D / 64) + d / 64;
                    K[p * D + d] = oracle_e4m3_to_double(kp[base + d]) * (double)k_scale[si];
                    V[p * D + d] = oracle_e4m3_to_double(vp[base + d]) * (double)v_scale[si];
                } else {
                    const uint16_t *kp = (const uint16_t *)k_pool;
                    const uint16_t *vp = (const uint16_t *)v_pool;
                    K[p * D + d] = oracle_bf16_to_double(kp[base + d]);
                    V[p * D + d] = oracle_bf16_to_double(vp[base + d]);
                }
            }
        }
        /* 2. textbook masked softmax(q K^T * scale) V for each query row */
        for (int gi = 0; gi < G; ++gi) {
            int h = g * G + gi;
            for (int j = 0; j < n_q; ++j) {
                const uint16_t *qv = q + (((long)b * n_q + j) * Hq + h) * D;
                double mx = -INFINITY;
                for (long p = 0; p < T; ++p) {
                    int visible;
                    if (p < L) {
                        visible = 1;
                    } else {
                        long i = p - L;
                        if (ancestor_mask)
                            visible = (int)((ancestor_mask[j] >> i) & 1ull);
                        else
                            visible = i <= j;
                    }
                    if (!visible) {
                        s[p] = -INFINITY;
                        continue;
                    }
                    double acc = 0.0;
                    for (int d = 0; d < D; ++d)
                        acc += oracle_bf16_to_double(qv[d]) * K[p * D + d];
                    s[p] = acc * sm_scale;
                    if (s[p] > mx) mx = s[p];
                }
                double sum = 0.0;
                for (long p = 0; p < T; ++p)
                    if (s[p] != -INFINITY) sum += exp(s[p] - mx);
                double *o = out + (((long)b * n_q + j) * Hq + h) * D;
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                for (long p = 0; p < T; ++p) {
                    if (s[p] == -INFINITY) continue;
                    double w = exp(s[p] - mx) / sum;
                    for (int d = 0; d < D; ++d) o[d] += w * V[p * D + d];
                }
                if (lse) lse[((long)b * n_q + j) * Hq + h] = mx + log(sum);
            }
        }
        free(K);
        free(V);
        free(s);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* rejection sampler                                                   */
/* ------------------------------------------------------------------ */

/*
 * Inverse-CDF draw from unnormalised non-negative weights r[0..V-1]:
 * S = sum r; the token is the first t whose running sum C_t exceeds u*S.
 * *near is set when some C_t/S lies within 1e-6 of u (a draw that fp32 and
 * fp64 arithmetic may resolve differently).  Returns -1 when S == 0.
 */
static int32_t draw_inverse_cdf(const double *r, int V, double u, uint8_t *near,
                                double *dist) {
    double S = 0.0;
    for (int t = 0; t < V; ++t) S += r[t];
    if (!(S > 0.0)) return -1;
    double target = u * S;
    double C = 0.0, best = INFINITY;
    int32_t tok = -1;
    for (int t = 0; t < V; ++t) {
        C += r[t];
        double dd = fabs(C / S - u);
        if (dd < best) best = dd;
        if (tok < 0 && C > target) tok = t;
    }
    if (tok < 0) {
        /* u*S >= S can only come from rounding: take the last token with mass */
        for (int t = V - 1; t >= 0; --t)
            if (r[t] > 0.0) { tok = t; break; }
    }
    if (near) *near = best < 1e-6;
    if (dist) *dist = best;
    return tok;
}

/* The draft/target acceptance test alpha_i = min(1, P/Q) realised with one
 * uniform: accept iff u*Q <= P, the product rounded once to fp32. */
static int accept_test(float u, float qx, float px) {
    volatile float a = u * qx; /* one rounded fp32 multiply, never fused */
    return a <= px;
}

/*
 * Linear speculative sampler, one row per sequence.
 * P fp32 [B, gamma+1, V] target distributions at the gamma+1 query positions;
 * Q fp32 [B, gamma, V] draft distributions; x int32 [B, gamma] draft tokens;
 * u_acc fp32 [B, gamma]; u_s fp32 [B].
 * Outputs accepted_len [B] (k), out_tokens [B, gamma+1] (x_0..x_{k-1}, then
 * the correction or bonus token, then -1), near [B] (1 when the final draw
 * was within 1e-6 of a CDF boundary), dist [B] (that distance; may be NULL).
 */
int oracle_spec_accept(int B, int gamma, int V, const float *P, const float *Q,
                       const int32_t *x, const float *u_acc, const float *u_s,
                       int32_t *accepted_len, int32_t *out_tokens, uint8_t *near,
                       double *dist, int nthreads) {
    if (B < 0 || gamma < 1 || V < 1) return ORC_ERR_ARG;
    for (long i = 0; i < (long)B * gamma; ++i)
        if (x[i] < 0 || x[i] >= V) return ORC_ERR_ARG;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 4)
    for (int b = 0; b < B; ++b) {
        const float *Pb = P + (long)b * (gamma + 1) * V;
        const float *Qb = Q + (long)b * gamma * V;
        int k = gamma;
        for (int i = 0; i < gamma; ++i) {
            int32_t xi = x[(long)b * gamma + i];
            if (!accept_test(u_acc[(long)b * gamma + i], Qb[(long)i * V + xi],
                             Pb[(long)i * V + xi])) {
                k = i;
                break;
            }
        }
        double *r = (double *)malloc(sizeof(double) * (size_t)V);
        int32_t tok;
        uint8_t nb = 0;
        double dd = INFINITY;
        if (k < gamma) {
            for (int t = 0; t < V; ++t) {
                double diff = (double)Pb[(long)k * V + t] - (double)Qb[(long)k * V + t];
                r[t] = diff > 0.0 ? diff : 0.0;
            }
            tok = draw_inverse_cdf(r, V, (double)u_s[b], &nb, &dd);
            if (tok < 0) { /* empty residual: fall back to the target row */
                for (int t = 0; t < V; ++t) r[t] = (double)Pb[(long)k * V + t];
                tok = draw_inverse_cdf(r, V, (double)u_s[b], &nb, &dd);
            }
        } else {
            for (int t = 0; t < V; ++t) r[t] = (double)Pb[(long)gamma * V + t];
            tok = draw_inverse_cdf(r, V, (double)u_s[b], &nb, &dd);
        }
        free(r);
        accepted_len[b] = k;
        int32_t *o = out_tokens + (long)b * (gamma + 1);
        for (int i = 0; i <= gamma; ++i)
            o[i] = i < k ? x[(long)b * gamma + i] : (i == k ? tok : -1);
        if (near) near[b] = nb;
        if (dist) dist[b] = dd;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* sampler front-end: probabilities formed from logits                 */
/* ------------------------------------------------------------------ */

/*
 * Max and normaliser of one row of logits at temperature T:
 * m = max_t l_t, S = sum_t exp((l_t - m) / T), so that
 * softmax(l / T)_t = exp((l_t - m) / T) / S.  -inf entries are masked tokens
 * (probability 0).  Returns -1 for a NaN or +inf entry or a row without a
 * finite entry.
 */
static int logit_row_stats(const float *l, int V, double T, double *m_out, double *S_out) {
    double m = -INFINITY;
    for (int t = 0; t < V; ++t) {
        if (isnan(l[t]) || (isinf(l[t]) && l[t] > 0.0f)) return -1;
        if ((double)l[t] > m) m = (double)l[t];
    }
    if (!isfinite(m)) return -1;
    double S = 0.0;
    for (int t = 0; t < V; ++t) S += exp(((double)l[t] - m) / T);
    *m_out = m;
    *S_out = S;
    return 0;
}

static double logit_prob(float l, double m, double S, double T) {
    return exp(((double)l - m) / T) / S;
}

/*
 * Inverse-CDF draw over unnormalised weights r (mass Z = sum r), the first
 * token whose running sum exceeds u*Z, with the near flag in absolute units:
 * set when u*Z lies within `band` of a running sum (0 before the first token
 * counts as one), or when u*Z reached Z by rounding.  Returns -1 when Z == 0.
 */
static int32_t draw_abs_band(const double *r, int V, double u, double band, uint8_t *near) {
    double Z = 0.0;
    for (int t = 0; t < V; ++t) Z += r[t];
    if (!(Z > 0.0)) return -1;
    const double target = u * Z;
    double C = 0.0, best = fabs(target);
    int32_t tok = -1;
    for (int t = 0; t < V; ++t) {
        C += r[t];
        if (fabs(C - target) < best) best = fabs(C - target);
        if (tok < 0 && C > target) tok = t;
    }
    if (tok < 0) {
        for (int t = V - 1; t >= 0; --t)
            if (r[t] > 0.0) { tok = t; break; }
        *near = 1;
    }
    if (best < band) *near = 1;
    return tok;
}

/*
 * Linear speculative sampler fed by logits.  The target pass yields logits,
 * the acceptance ratio takes softmax(logits)[x] for each draft token, and the
 * draft probability is the draft model's own ("Speculative Decoding and
 * KV-Cache Compression", section 2.3; "LOW-LATENCY INFERENCE: SPECULATIVE
 * DECODING & PAGING", architecture: target logits P checked against draft
 * logits Q).  The sampling temperatures are separate knobs for the target
 * and the draft (the first page's alert table lowers the draft temperature
 * alone), so P_i = softmax(Lp_i / T_target) and Q_i = softmax(Lq_i / T_draft),
 * Q being the distribution the drafts were drawn from.
 *
 * Lp fp32 [B, gamma+1, V] target logits; Lq fp32 [B, gamma, V] draft logits;
 * x, u_acc, u_s, accepted_len, out_tokens as in oracle_spec_accept.  Every
 * probability is fp64 (exp of the fp64 difference), and so are the tests:
 * accept x_i iff u_i * Q_i(x_i) <= P_i(x_i); the residual max(0, P_k - Q_k)
 * (P_k when it has no mass) or, with every draft accepted, P_gamma; the token
 * is the first whose running mass exceeds u * (total mass).
 *
 * near[b] is set when a decision sits within `band` of its threshold, where
 * an fp32 formation of P and Q may take it the other way: an acceptance test
 * that ran with |u Q - P| <= band * max(P, u Q) or max(P, u Q) < 2^-100; a
 * residual with mass below band; a draw with u*Z within band of a running sum
 * (absolute, in probability units).
 *
 * test_accept / test_near (uint8 [B, gamma], may be NULL) receive every
 * test's decision and near flag, the tests after the first rejection
 * included, so that a sampler whose near-threshold decisions went the other
 * way can be checked test by test.
 *
 * Returns ORC_ERR_ARG for bad sizes or temperatures, a draft token out of
 * range, or a row that logit_row_stats rejects.
 */
int oracle_spec_accept_logits(int B, int gamma, int V, double T_target, double T_draft, double band,
                              const float *Lp, const float *Lq, const int32_t *x, const float *u_acc,
                              const float *u_s, int32_t *accepted_len, int32_t *out_tokens,
                              uint8_t *near, uint8_t *test_accept, uint8_t *test_near, int nthreads) {
    if (B < 0 || gamma < 1 || V < 1 || !(T_target > 0.0) || !(T_draft > 0.0) || !(band >= 0.0))
        return ORC_ERR_ARG;
    for (long i = 0; i < (long)B * gamma; ++i)
        if (x[i] < 0 || x[i] >= V) return ORC_ERR_ARG;
    const double tiny = ldexp(1.0, -100);
    int bad = 0;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int b = 0; b < B; ++b) {
        const float *Pb = Lp + (long)b * (gamma + 1) * V;
        const float *Qb = Lq + (long)b * gamma * V;
        double *mp = (double *)malloc(sizeof(double) * (size_t)(4 * gamma + 2));
        double *Sp = mp + (gamma + 1), *mq = Sp + (gamma + 1), *Sq = mq + gamma;
        double *r = (double *)malloc(sizeof(double) * (size_t)V);
        uint8_t nb = 0;
        int ok = 1;
        for (int i = 0; i <= gamma && ok; ++i)
            ok = logit_row_stats(Pb + (long)i * V, V, T_target, &mp[i], &Sp[i]) == 0;
        for (int i = 0; i < gamma && ok; ++i)
            ok = logit_row_stats(Qb + (long)i * V, V, T_draft, &mq[i], &Sq[i]) == 0;
        if (!ok) {
            bad = 1;
            free(mp);
            free(r);
            continue;
        }
        int k = gamma;
        for (int i = 0; i < gamma; ++i) {
            const int32_t xi = x[(long)b * gamma + i];
            const double P = logit_prob(Pb[(long)i * V + xi], mp[i], Sp[i], T_target);
            const double Q = logit_prob(Qb[(long)i * V + xi], mq[i], Sq[i], T_draft);
            const double uq = (double)u_acc[(long)b * gamma + i] * Q;
            const double hi = P > uq ? P : uq;
            const int close = fabs(uq - P) <= band * hi || hi < tiny;
            const int accept = uq <= P;
            if (test_accept) test_accept[(long)b * gamma + i] = (uint8_t)accept;
            if (test_near) test_near[(long)b * gamma + i] = (uint8_t)close;
            if (k == gamma) {  /* a test that ran */
                if (close) nb = 1;
                if (!accept) k = i;
            }
        }
        int32_t tok;
        if (k < gamma) {
            double Z = 0.0;
            for (int t = 0; t < V; ++t) {
                const double d = logit_prob(Pb[(long)k * V + t], mp[k], Sp[k], T_target) -
                                 logit_prob(Qb[(long)k * V + t], mq[k], Sq[k], T_draft);
                r[t] = d > 0.0 ? d : 0.0;
                Z += r[t];
            }
            if (Z < band) nb = 1;
            if (!(Z > 0.0))  /* empty residual: draw from the target row */
                for (int t = 0; t < V; ++t) r[t] = logit_prob(Pb[(long)k * V + t], mp[k], Sp[k], T_target);
        } else {
            for (int t = 0; t < V; ++t) r[t] = logit_prob(Pb[(long)gamma * V + t], mp[gamma], Sp[gamma], T_target);
        }
        tok = draw_abs_band(r, V, (double)u_s[b], band, &nb);
        free(mp);
        free(r);
        accepted_len[b] = k;
        int32_t *o = out_tokens + (long)b * (gamma + 1);
        for (int i = 0; i <= gamma; ++i)
            o[i] = i < k ? x[(long)b * gamma + i] : (i == k ? tok : -1);
        if (near) near[b] = nb;
    }
    return bad ? ORC_ERR_ARG : ORC_OK;
}

/*
 * The tokens an fp32 formation of P and Q may draw for a given accepted count:
 * with k[b] < gamma the residual max(0, P_k - Q_k) of mass Z, else P_gamma
 * (Z = 1), and target u*Z; every token whose running-sum interval
 * [C_{t-1}, C_t], widened by `band` on both sides, contains the target.  The
 * sums are monotone, so the tokens form the range [tok_lo, tok_hi].  When the
 * residual's mass is below band (it may be empty, so the draw may come from
 * P_k) the range is the whole vocabulary.
 */
int oracle_logits_draw_window(int B, int gamma, int V, double T_target, double T_draft, double band,
                              const float *Lp, const float *Lq, const int32_t *k_in, const float *u_s,
                              int32_t *tok_lo, int32_t *tok_hi, int nthreads) {
    if (B < 0 || gamma < 1 || V < 1 || !(T_target > 0.0) || !(T_draft > 0.0) || !(band >= 0.0))
        return ORC_ERR_ARG;
    for (int b = 0; b < B; ++b)
        if (k_in[b] < 0 || k_in[b] > gamma) return ORC_ERR_ARG;
    int bad = 0;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int b = 0; b < B; ++b) {
        const int k = k_in[b];
        const float *lp = Lp + ((long)b * (gamma + 1) + k) * V;
        const float *lq = k < gamma ? Lq + ((long)b * gamma + k) * V : NULL;
        double m_p, S_p, m_q = 0.0, S_q = 1.0;
        if (logit_row_stats(lp, V, T_target, &m_p, &S_p) != 0 ||
            (lq && logit_row_stats(lq, V, T_draft, &m_q, &S_q) != 0)) {
            bad = 1;
            continue;
        }
        double *r = (double *)malloc(sizeof(double) * (size_t)V);
        double Z = 0.0;
        for (int t = 0; t < V; ++t) {
            double w = logit_prob(lp[t], m_p, S_p, T_target);
            if (lq) {
                w -= logit_prob(lq[t], m_q, S_q, T_draft);
                if (w < 0.0) w = 0.0;
            }
            r[t] = w;
            Z += w;
        }
        int32_t lo = 0, hi = V - 1;
        if (!(lq && Z < band)) {
            const double target = (double)u_s[b] * Z;
            double C = 0.0;
            lo = -1;
            hi = -1;
            for (int t = 0; t < V; ++t) {
                C += r[t];
                if (lo < 0 && C >= target - band) lo = t;
                if (hi < 0 && C > target + band) hi = t;
            }
            if (lo < 0) lo = V - 1;
            if (hi < 0) hi = V - 1;
        }
        free(r);
        tok_lo[b] = lo;
        tok_hi[b] = hi;
    }
    return bad ? ORC_ERR_ARG : ORC_OK;
}

/* Tree helpers: a node is internal when some node names it as parent; its
 * draft row in Q is its rank among internal nodes in node order. */
static int tree_depth_of(const int32_t *parent, int node) {
    int d = 0;
    while (node > 0) { node = parent[node]; ++d; }
    return d;
}

/* Depth of the deepest node, or -1 when parent[] is not a tree in node order
 * (parent[0] = -1, 0 <= parent[i] < i). */
int oracle_tree_max_depth(const int32_t *parent, int n_nodes) {
    if (n_nodes < 1 || parent[0] != -1) return -1;
    for (int i = 1; i < n_nodes; ++i)
        if (parent[i] < 0 || parent[i] >= i) return -1;
    int md = 0;
    for (int i = 0; i < n_nodes; ++i) {
        int d = tree_depth_of(parent, i);
        if (d > md) md = d;
    }
    return md;
}

/*
 * Tree speculative sampler (recursive residual rejection over the children of
 * a node, children tested in index order; reduces to the linear sampler when
 * every node has one child).  Unnormalised residual R with mass Z:
 *   at a node: R = P[node], Z = 1;
 *   child c (token x_c): accept iff u_acc[c]*Q[node](x_c)*Z <= R(x_c)
 *     -- for the first child (Z = 1, R = P) this is the fp32 test u*Q <= P;
 *        later children use fp64;
 *   on reject: R <- max(0, R - Z*Q[node]), Z <- sum R;
 *   if a child is accepted: descend to it; if none: draw from R with u_s;
 *   at a leaf (all of its ancestors accepted): draw a bonus from P[leaf].
 * parent int32 [n_nodes] (parent[0] = -1, parent[i] < i); P fp32
 * [B, n_nodes, V]; Q fp32 [B, n_internal, V]; node_tokens int32 [B, n_nodes];
 * u_acc fp32 [B, n_nodes] (entry c is used for child c's test); u_s fp32 [B].
 * Outputs: accepted_len [B]; path_nodes [B, max_depth+1] (root, the accepted
 * nodes, then -1); out_tokens [B, max_depth+1]; near [B] set when any
 * fp64-vs-fp32 sensitive decision (a later-child test or the final draw) fell
 * within 1e-6 (in normalised units) of its threshold.
 */
int oracle_spec_accept_tree(int B, int n_nodes, int V, const int32_t *parent,
                            const float *P, const float *Q,
                            const int32_t *node_tokens, const float *u_acc,
                            const float *u_s, int32_t *accepted_len,
                            int32_t *path_nodes, int32_t *out_tokens,
                            uint8_t *near, int nthreads) {
    if (B < 0 || n_nodes < 1 || n_nodes > 64 || V < 1 || parent[0] != -1)
        return ORC_ERR_ARG;
    for (int i = 1; i < n_nodes; ++i)
        if (parent[i] < 0 || parent[i] >= i) return ORC_ERR_ARG;
    int *qrow = (int *)malloc(sizeof(int) * (size_t)n_nodes);
    int n_internal = 0;
    for (int i = 0; i < n_nodes; ++i) {
        int has_child = 0;
        for (int c = i + 1; c < n_nodes; ++c) has_child |= parent[c] == i;
        qrow[i] = has_child ? n_internal++ : -1;
    }
    const int W = oracle_tree_max_depth(parent, n_nodes) + 1;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        double *R = (double *)malloc(sizeof(double) * (size_t)V);
        int32_t *path = path_nodes + (long)b * W;
        int32_t *outt = out_tokens + (long)b * W;
        const int32_t *tok = node_tokens + (long)b * n_nodes;
        for (int i = 0; i < W; ++i) path[i] = outt[i] = -1;
        path[0] = 0;
        int node = 0, depth = 0;
        uint8_t nb = 0;
        int32_t final_tok = -1;
        for (;;) {
            const float *Pn = P + ((long)b * n_nodes + node) * V;
            if (qrow[node] < 0) { /* leaf reached: bonus from its target row */
                for (int t = 0; t < V; ++t) R[t] = (double)Pn[t];
                uint8_t nn = 0;
                final_tok = draw_inverse_cdf(R, V, (double)u_s[b], &nn, NULL);
                nb |= nn;
                break;
            }
            const float *Qn = Q + ((long)b * n_internal + qrow[node]) * V;
            for (int t = 0; t < V; ++t) R[t] = (double)Pn[t];
            double Z = 1.0;
            int accepted = -1, tested = 0;
            for (int c = node + 1; c < n_nodes; ++c) {
                if (parent[c] != node) continue;
                int32_t xc = tok[c];
                int ok;
                if (tested == 0) {
                    ok = accept_test(u_acc[(long)b * n_nodes + c], Qn[xc], Pn[xc]);
                } else {
                    double lhs = (double)u_acc[(long)b * n_nodes + c] * (double)Qn[xc] * Z;
                    ok = lhs <= R[xc];
                    if (Z > 0.0 && fabs(lhs - R[xc]) / Z < 1e-6) nb = 1;
                }
                ++tested;
                if (ok) { accepted = c; break; }
                double Znew = 0.0;
                for (int t = 0; t < V; ++t) {
                    double v = R[t] - Z * (double)Qn[t];
                    R[t] = v > 0.0 ? v : 0.0;
                    Znew += R[t];
                }
                Z = Znew;
            }
            if (accepted >= 0) {
                ++depth;
                path[depth] = accepted;
                outt[depth - 1] = tok[accepted];
                node = accepted;
                continue;
            }
            uint8_t nn = 0;
            final_tok = draw_inverse_cdf(R, V, (double)u_s[b], &nn, NULL);
            if (final_tok < 0) { /* empty residual: fall back to the target row */
                for (int t = 0; t < V; ++t) R[t] = (double)Pn[t];
                final_tok = draw_inverse_cdf(R, V, (double)u_s[b], &nn, NULL);
            }
            nb |= nn;
            break;
        }
        accepted_len[b] = depth;
        outt[depth] = final_tok;
        if (near) near[b] = nb;
        free(R);
    }
    free(qrow);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* draft-tree sampler fed by logits                                    */
/* ------------------------------------------------------------------ */

/*
 * Near-boundary scale after j rejected siblings at a node.  An fp32
 * formation of P and Q errs by at most eps ~ band/2 relative per
 * probability.  Carried through the recursion, the residual entry R_j(t)
 * then errs by at most eps (P(t) + a_j Q(t)) and its mass Z_j by eps (1 + a_j),
 * where a_0 = 0, a_1 = 1 and a_{j+1} = 2 a_j + 2.  A test after j
 * rejections, u Q(x) Z_j against R_j(x), is then off by at most
 * eps (P(x) + a_{j+1} Q(x)), which is <= 2^(j+1) band max(P(x), Q(x)).
 * A draw's running sums are off by at most eps (1 + a_j) <= 2^(j+1) band.
 */
static double tree_logit_scale(int j, double band) { return ldexp(band, j + 1); }

/* One node's children tests on fp64 P = P[node], Q = Q[qrow(node)]: for the
 * children c_1..c_m in index order, the exact decision of c_i given that
 * c_1..c_{i-1} were rejected (acc[i]) and whether it lies in the band
 * (close[i]); R ends as the residual after every child is rejected, with
 * mass *Z_out.  kids[] lists the children. */
static void tree_logit_node_tests(const double *Pn, const double *Qn, int V, const int32_t *kids, int m,
                                  const int32_t *tok, const float *ua, double band, double *R,
                                  uint8_t *acc, uint8_t *close, double *Z_out) {
    const double tiny = ldexp(1.0, -100);
    for (int t = 0; t < V; ++t) R[t] = Pn[t];
    double Z = 1.0;
    for (int i = 0; i < m; ++i) {
        const int c = kids[i];
        const int32_t x = tok[c];
        const double lhs = (double)ua[c] * Qn[x] * Z;
        const double hi = Pn[x] > Qn[x] ? Pn[x] : Qn[x];
        acc[i] = (uint8_t)(lhs <= R[x]);
        close[i] = (uint8_t)(fabs(lhs - R[x]) <= tree_logit_scale(i, band) * hi || hi < tiny);
        double Zn = 0.0;
        for (int t = 0; t < V; ++t) {
            const double v = R[t] - Z * Qn[t];
            R[t] = v > 0.0 ? v : 0.0;
            Zn += R[t];
        }
        Z = Zn;
    }
    *Z_out = Z;
}

/* fp64 softmax(l / T) of one row into out; -1 for a row logit_row_stats rejects. */
static int softmax_row(const float *l, int V, double T, double *out) {
    double m, S;
    if (logit_row_stats(l, V, T, &m, &S) != 0) return -1;
    for (int t = 0; t < V; ++t) out[t] = logit_prob(l[t], m, S, T);
    return 0;
}

/* The tree's shape: children of every node in index order, and each internal
 * node's row in the draft logits.  Returns the number of internal nodes, or
 * -1 for a parent array that is not a tree in node order. */
static int tree_shape(const int32_t *parent, int n_nodes, int32_t *kid_start, int32_t *kids, int32_t *qrow) {
    if (n_nodes < 1 || n_nodes > 64 || parent[0] != -1) return -1;
    for (int i = 1; i < n_nodes; ++i)
        if (parent[i] < 0 || parent[i] >= i) return -1;
    int n = 0, internal = 0;
    for (int i = 0; i < n_nodes; ++i) {
        kid_start[i] = n;
        for (int c = i + 1; c < n_nodes; ++c)
            if (parent[c] == i) kids[n++] = c;
        qrow[i] = n > kid_start[i] ? internal++ : -1;
    }
    kid_start[n_nodes] = n;
    return internal;
}

/*
 * Draft-tree sampler fed by logits: the tree recursion of
 * oracle_spec_accept_tree (children tested in index order, the residual
 * R <- max(0, R - Z Q) after each rejection, a draw from R when every child is
 * rejected -- from P when R is empty -- and a bonus from P at a leaf) on
 * P[node] = softmax(Lp[node] / T_target) and Q[node] = softmax(Lq[qrow(node)] /
 * T_draft), formed in fp64 ("Speculative Decoding and KV-Cache Compression",
 * section 2.3: the ratio takes softmax(logits)[x]; "The Sub-Millisecond
 * Speculative Decoding Meltdown", tree attention: the target scores every
 * node of the draft tree in one pass).  Every test is fp64: child c, after j
 * rejected siblings, is accepted iff u_acc[c] * Q(x_c) * Z <= R(x_c), where
 * R = P and Z = 1 for the first child.
 *
 * near[b] is set when a decision sits where an fp32 formation of P and Q may
 * take it the other way (tree_logit_scale): a test that ran with
 * |u Q Z - R(x)| <= 2^(j+1) band max(P(x), Q(x)), or max(P(x), Q(x)) < 2^-100;
 * a residual after j >= 1 rejections with mass below 2^(j+1) band; a draw
 * with u*Z within 2^(j+1) band (absolute) of a running sum, or within band
 * for a draw from P.
 *
 * Lp fp32 [B, n_nodes, V]; Lq fp32 [B, n_internal, V] (internal nodes in node
 * order); node_tokens, u_acc int32/fp32 [B, n_nodes]; u_s fp32 [B]; outputs
 * as oracle_spec_accept_tree.  Returns ORC_ERR_ARG for a bad tree, sizes or
 * temperatures, a node token out of range, or a row logit_row_stats rejects.
 */
int oracle_spec_accept_tree_logits(int B, int n_nodes, int V, const int32_t *parent, double T_target,
                                   double T_draft, double band, const float *Lp, const float *Lq,
                                   const int32_t *node_tokens, const float *u_acc, const float *u_s,
                                   int32_t *accepted_len, int32_t *path_nodes, int32_t *out_tokens,
                                   uint8_t *near, int nthreads) {
    int32_t kid_start[65], kids[64], qrow[64];
    const int n_internal = tree_shape(parent, n_nodes, kid_start, kids, qrow);
    if (n_internal < 0 || B < 0 || V < 1 || !(T_target > 0.0) || !(T_draft > 0.0) || !(band >= 0.0))
        return ORC_ERR_ARG;
    for (long i = 0; i < (long)B * n_nodes; ++i)
        if (i % n_nodes && (node_tokens[i] < 0 || node_tokens[i] >= V)) return ORC_ERR_ARG;
    const int W = oracle_tree_max_depth(parent, n_nodes) + 1;
    int bad = 0;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int b = 0; b < B; ++b) {
        double *P = (double *)malloc(sizeof(double) * (size_t)V * 3);
        double *Q = P + V, *R = Q + V;
        const int32_t *tok = node_tokens + (long)b * n_nodes;
        const float *ua = u_acc + (long)b * n_nodes;
        int32_t *path = path_nodes + (long)b * W;
        int32_t *outt = out_tokens + (long)b * W;
        for (int i = 0; i < W; ++i) path[i] = outt[i] = -1;
        path[0] = 0;
        int node = 0, depth = 0, ok = 1;
        uint8_t nb = 0;
        int32_t final_tok = -1;
        for (;;) {
            ok = softmax_row(Lp + ((long)b * n_nodes + node) * V, V, T_target, P) == 0;
            if (!ok) break;
            const int m = kid_start[node + 1] - kid_start[node];
            if (m == 0) { /* leaf: bonus from its own P, band as for any draw from P */
                final_tok = draw_abs_band(P, V, (double)u_s[b], band, &nb);
                break;
            }
            ok = softmax_row(Lq + ((long)b * n_internal + qrow[node]) * V, V, T_draft, Q) == 0;
            if (!ok) break;
            uint8_t acc[64], cl[64];
            double Z;
            tree_logit_node_tests(P, Q, V, kids + kid_start[node], m, tok, ua, band, R, acc, cl, &Z);
            int taken = -1;
            for (int i = 0; i < m && taken < 0; ++i) {
                if (cl[i]) nb = 1; /* a test that ran */
                if (acc[i]) taken = i;
            }
            if (taken >= 0) {
                node = kids[kid_start[node] + taken];
                ++depth;
                path[depth] = node;
                outt[depth - 1] = tok[node];
                continue;
            }
            /* every child rejected: R and Z are the residual after m rejections
             * (tree_logit_node_tests recomputed the residual past the accepted
             * child only when there was none) */
            const double s = tree_logit_scale(m, band);
            if (Z < s) nb = 1;
            if (Z > 0.0) {
                final_tok = draw_abs_band(R, V, (double)u_s[b], s, &nb);
            } else { /* empty residual: draw from the node's target row */
                final_tok = draw_abs_band(P, V, (double)u_s[b], band, &nb);
            }
            break;
        }
        free(P);
        if (!ok) {
            bad = 1;
            continue;
        }
        accepted_len[b] = depth;
        outt[depth] = final_tok;
        if (near) near[b] = nb;
    }
    return bad ? ORC_ERR_ARG : ORC_OK;
}

/*
 * Every outcome an fp32 formation of the tree sampler fed by logits may
 * produce, per sequence b and node n, from the inputs alone (the decisions
 * and bands of oracle_spec_accept_tree_logits):
 *   end_ok[b][n] = 1 when the walk may end at n: each test on the way from the
 *   root (the siblings before the path's child rejected, the path's child
 *   accepted) and, at an internal n, every child's rejection is the exact
 *   decision or lies in its band;
 *   [tok_lo, tok_hi][b][n] = the tokens the final draw at n may give: the
 *   tokens whose running-sum interval, widened by the draw's band, holds u*Z
 *   (from P[n] at a leaf; from the residual after all m children are
 *   rejected at an internal node, the whole vocabulary when its mass is below
 *   the band, as it may then be empty).
 */
int oracle_tree_logits_outcomes(int B, int n_nodes, int V, const int32_t *parent, double T_target,
                                double T_draft, double band, const float *Lp, const float *Lq,
                                const int32_t *node_tokens, const float *u_acc, const float *u_s,
                                uint8_t *end_ok, int32_t *tok_lo, int32_t *tok_hi, int nthreads) {
    int32_t kid_start[65], kids[64], qrow[64];
    const int n_internal = tree_shape(parent, n_nodes, kid_start, kids, qrow);
    if (n_internal < 0 || B < 0 || V < 1 || !(T_target > 0.0) || !(T_draft > 0.0) || !(band >= 0.0))
        return ORC_ERR_ARG;
    for (long i = 0; i < (long)B * n_nodes; ++i)
        if (i % n_nodes && (node_tokens[i] < 0 || node_tokens[i] >= V)) return ORC_ERR_ARG;
    int bad = 0;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int b = 0; b < B; ++b) {
        double *P = (double *)malloc(sizeof(double) * (size_t)V * 3);
        double *Q = P + V, *R = Q + V;
        const int32_t *tok = node_tokens + (long)b * n_nodes;
        const float *ua = u_acc + (long)b * n_nodes;
        uint8_t reach[64];
        uint8_t *eo = end_ok + (long)b * n_nodes;
        int32_t *lo = tok_lo + (long)b * n_nodes, *hi = tok_hi + (long)b * n_nodes;
        reach[0] = 1;
        for (int n = 0; n < n_nodes && !bad; ++n) { /* parents come before children */
            if (softmax_row(Lp + ((long)b * n_nodes + n) * V, V, T_target, P) != 0) {
                bad = 1;
                break;
            }
            const int m = kid_start[n + 1] - kid_start[n];
            double Z = 1.0, s = band;
            const double *W = P;
            int all_rejected_ok = 1;
            if (m > 0) {
                if (softmax_row(Lq + ((long)b * n_internal + qrow[n]) * V, V, T_draft, Q) != 0) {
                    bad = 1;
                    break;
                }
                uint8_t acc[64], cl[64];
                tree_logit_node_tests(P, Q, V, kids + kid_start[n], m, tok, ua, band, R, acc, cl, &Z);
                int before_ok = 1; /* the siblings before child i may all be rejected */
                for (int i = 0; i < m; ++i) {
                    const int c = kids[kid_start[n] + i];
                    reach[c] = (uint8_t)(reach[n] && before_ok && (acc[i] || cl[i]));
                    before_ok = before_ok && (!acc[i] || cl[i]);
                }
                all_rejected_ok = before_ok;
                s = tree_logit_scale(m, band);
                W = R;
            }
            eo[n] = (uint8_t)(reach[n] && all_rejected_ok);
            if (m > 0 && Z < s) { /* a residual that may be empty: any token */
                lo[n] = 0;
                hi[n] = V - 1;
                continue;
            }
            const double target = (double)u_s[b] * Z;
            double C = 0.0;
            int32_t l = -1, h = -1;
            for (int t = 0; t < V; ++t) {
                C += W[t];
                if (l < 0 && C >= target - s) l = t;
                if (h < 0 && C > target + s) h = t;
            }
            lo[n] = l < 0 ? V - 1 : l;
            hi[n] = h < 0 ? V - 1 : h;
        }
        free(P);
    }
    return bad ? ORC_ERR_ARG : ORC_OK;
}

/* ------------------------------------------------------------------ */
/* block-table commit / rollback                                       */
/* ------------------------------------------------------------------ */

/*
 * For each sequence b with committed length L and k = accepted_len[b]:
 *  - tree (path_nodes != NULL, row width path_w): for d = 1..k, in increasing
 *    d, copy the K and V rows (all kv heads) of speculative slot
 *    L + path_nodes[b][d] to slot L + d;
 *  - the new length is L + k + 1 (the last committed token and the k accepted
 *    drafts have K/V; the correction/bonus token gets its K/V next step);
 *  - logical blocks i with ceil(new/BS) <= i < ceil((L+n_q)/BS) are dropped:
 *    the table entry becomes -1 and the block's reference count falls by one;
 *    a block whose count reaches 0 is pushed on the free stack.
 * Sequences are processed in order b = 0..B-1 and blocks in increasing i, so
 * the free-stack order here is one valid order among many.
 * elem_bytes is 2 (bf16) or 1 (FP8); the pool layout is
 * [num_blocks, Hkv, BS, D].
 */
int oracle_block_table_commit(int B, int n_q, int BS, int max_blocks,
                              int num_blocks, int32_t *block_table,
                              int32_t *context_lens, const int32_t *accepted_len,
                              int32_t *refcount, int32_t *free_stack,
                              int32_t *free_top, const int32_t *path_nodes,
                              int path_w, void *k_pool, void *v_pool, int Hkv,
                              int D, int elem_bytes) {
    if (B < 0 || n_q < 1 || BS < 1 || max_blocks < 1 || num_blocks < 1)
        return ORC_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        long L = context_lens[b];
        int k = accepted_len[b];
        long T = L + n_q;
        if (L < 0 || k < 0 || k >= n_q || (T + BS - 1) / BS > max_blocks)
            return ORC_ERR_ARG;
        if (path_nodes) {
            if (path_w < k + 1) return ORC_ERR_ARG;
            size_t row = (size_t)D * (size_t)elem_bytes;
            for (int d = 1; d <= k; ++d) {
                long src = L + path_nodes[(long)b * path_w + d];
                long dst = L + d;
                if (src < dst || src >= T) return ORC_ERR_ARG;
                int32_t sb = block_table[(long)b * max_blocks + src / BS];
                int32_t db = block_table[(long)b * max_blocks + dst / BS];
                if (sb < 0 || sb >= num_blocks || db < 0 || db >= num_blocks)
                    return ORC_ERR_BAD_BLOCK;
                for (int g = 0; g < Hkv; ++g) {
                    size_t so = ((((size_t)sb * Hkv + g) * BS) + src % BS) * row;
                    size_t dof = ((((size_t)db * Hkv + g) * BS) + dst % BS) * row;
                    memmove((char *)k_pool + dof, (char *)k_pool + so, row);
                    memmove((char *)v_pool + dof, (char *)v_pool + so, row);
                }
            }
        }
        long new_len = L + k + 1;
        long keep = (new_len + BS - 1) / BS;
        long had = (T + BS - 1) / BS;
        for (long i = keep; i < had; ++i) {
            int32_t *e = &block_table[(long)b * max_blocks + i];
            int32_t blk = *e;
            if (blk < 0 || blk >= num_blocks) return ORC_ERR_BAD_BLOCK;
            *e = -1;
            refcount[blk] -= 1;
            if (refcount[blk] == 0) {
                if (*free_top >= num_blocks) return ORC_ERR_OUT_OF_BLOCKS;
                free_stack[(*free_top)++] = blk;
            }
        }
        context_lens[b] = (int32_t)new_len;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* paged K/V append (allocation, copy-on-write, FP8 quantise-on-write) */
/* ------------------------------------------------------------------ */

/* OCP E4M3 ("fn") code of a finite fp32 value: round to nearest, ties to
 * even, saturating at +-448 (the largest finite code, S.1111.110); written
 * from the format's definition: 4 exponent bits (bias 7), 3 mantissa bits,
 * subnormals at exponent field 0 with quantum 2^-9. */
uint8_t oracle_e4m3_encode(float xf) {
    double x = (double)xf;
    uint8_t sign = 0;
    if (signbit(x)) { sign = 0x80; x = -x; } /* E4M3 has a signed zero: -0 is 0x80 */
    if (!(x == x)) return 0x7F; /* NaN stays NaN (never produced here) */
    if (x >= 448.0) return sign | 0x7E;
    int e = -6; /* exponent of the quantum's binade; subnormals share e = -6 */
    if (x >= ldexp(1.0, -6)) e = (int)floor(log2(x));
    /* guard log2 rounding at exact powers of two */
    while (e > -6 && x < ldexp(1.0, e)) --e;
    while (x >= ldexp(1.0, e + 1)) ++e;
    double q = ldexp(1.0, e - 3); /* spacing of codes in this binade */
    double n = x / q;            /* exact: q is a power of two */
    double fl = floor(n), fr = n - fl;
    double r = fl;
    if (fr > 0.5 || (fr == 0.5 && fmod(fl, 2.0) != 0.0)) r = fl + 1.0;
    if (e == -6 && r < 8.0) return sign | (uint8_t)r; /* subnormal (or zero) */
    if (r >= 16.0) { r = 8.0; ++e; }
    int ef = e + 7;
    if (ef > 15 || (ef == 15 && r > 14.0)) return sign | 0x7E; /* saturate */
    return sign | (uint8_t)(ef << 3) | (uint8_t)((int)r - 8);
}

static float bf16_bits_to_float(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * Append n_new token rows to every sequence's paged K/V ("Speculative
 * Decoding & KV-Cache PagedAttention in Enterprise LLM Serving",
 * PagedKVCacheManager.EnsureCapacityAndAppendToken: a page past the table's
 * end is taken from the free pool with count 1; a page whose count is above 1
 * is cloned before it is written, the shared block losing one reference;
 * "The Sub-Millisecond Speculative Decoding Meltdown", "Custom FP8 Quantized
 * Memory Block Layout": e4m3 pages with per-block K and V scales).
 *
 * Sequence b's rows go to positions L_b .. L_b + n_new - 1 (L_b =
 * context_lens[b], which is not changed: the commit step sets the new
 * length).  Sequences are handled in index order; pages in increasing order.
 * A page holding history (index * BS < L_b) must already be mapped.
 * Free pops take free_stack[--free_top].
 *
 * FP8 pools (quantise-on-write): for every (written page, kv head) the scale
 * becomes amax / 448 (1 when amax = 0), amax being the largest magnitude of
 * the page's history values (stored code times the old scale, an fp32
 * product) and of the new rows (bf16 values); history codes are re-encoded
 * from their decoded value only when the scale changes; every code is
 * e4m3(value / scale) with one fp32 division; slots past the last row are 0.
 *
 * FP8 pools with one scale per 64-element tile (fp8 = 2; "The Sub-Millisecond
 * Speculative Decoding Meltdown", implementation checklist: block scales per
 * 64-element tile): each 64-value tile of a new row gets scale = amax / 448
 * of its own values (1 when amax = 0) and codes e4m3(value / scale); history
 * rows keep their codes and scales; codes past the last row are 0.
 *
 * new_k, new_v: bf16 bits [B, n_new, Hkv, D]; pools [num_blocks, Hkv, BS, D]
 * of bf16 bits (fp8 = 0) or E4M3 bytes (fp8 = 1, 2); scales [num_blocks, Hkv]
 * (fp8 = 1) or [num_blocks, Hkv, BS, D / 64] (fp8 = 2).
 */
int oracle_kv_append(int B, int n_new, int Hkv, int D, int BS, int max_blocks, int num_blocks,
                     int fp8, const uint16_t *new_k, const uint16_t *new_v, int32_t *block_table,
                     const int32_t *context_lens, int32_t *refcount, int32_t *free_stack,
                     int32_t *free_top, void *k_pool, void *v_pool, float *k_scale,
                     float *v_scale) {
    if (B < 0 || n_new < 1 || Hkv < 1 || D < 1 || BS < 1 || max_blocks < 1 || num_blocks < 1)
        return ORC_ERR_ARG;
    if (fp8 && (!k_scale || !v_scale)) return ORC_ERR_ARG;
    if (fp8 < 0 || fp8 > 2 || (fp8 == 2 && D % 64 != 0)) return ORC_ERR_ARG;
    const size_t eb = fp8 ? 1 : 2;
    const size_t page_bytes = (size_t)Hkv * BS * D * eb; /* one block, all heads */
    const long scales_per_block = fp8 == 2 ? (long)Hkv * BS * (D / 64) : Hkv;
    for (int b = 0; b < B; ++b) {
        const long L = context_lens[b], end = L + n_new;
        if (L < 0 || (end + BS - 1) / BS > max_blocks) return ORC_ERR_ARG;
        /* map, allocate or clone every page the rows touch */
        for (long i = L / BS; i <= (end - 1) / BS; ++i) {
            int32_t *ent = &block_table[(long)b * max_blocks + i];
            if (*ent < 0) {
                if (i * BS < L) return ORC_ERR_ARG; /* history without a page */
                if (*free_top <= 0) return ORC_ERR_OUT_OF_BLOCKS;
                int32_t blk = free_stack[--(*free_top)];
                if (blk < 0 || blk >= num_blocks) return ORC_ERR_BAD_BLOCK;
                refcount[blk] = 1;
                *ent = blk;
                continue;
            }
            if (*ent >= num_blocks) return ORC_ERR_BAD_BLOCK;
            if (refcount[*ent] > 1) { /* shared: copy-on-write */
                if (*free_top <= 0) return ORC_ERR_OUT_OF_BLOCKS;
                int32_t blk = free_stack[--(*free_top)];
                if (blk < 0 || blk >= num_blocks) return ORC_ERR_BAD_BLOCK;
                memcpy((char *)k_pool + (size_t)blk * page_bytes,
                       (char *)k_pool + (size_t)*ent * page_bytes, page_bytes);
                memcpy((char *)v_pool + (size_t)blk * page_bytes,
                       (char *)v_pool + (size_t)*ent * page_bytes, page_bytes);
                if (fp8)
                    for (long x = 0; x < scales_per_block; ++x) {
                        k_scale[(long)blk * scales_per_block + x] = k_scale[(long)*ent * scales_per_block + x];
                        v_scale[(long)blk * scales_per_block + x] = v_scale[(long)*ent * scales_per_block + x];
                    }
                refcount[*ent] -= 1;
                refcount[blk] = 1;
                *ent = blk;
            }
        }
        /* write the rows */
        for (long i = L / BS; i <= (end - 1) / BS; ++i) {
            const int32_t blk = block_table[(long)b * max_blocks + i];
            const long ps = i * BS;
            const long hist = L > ps ? (L - ps < BS ? L - ps : BS) : 0; /* history slots in the page */
            const long vend = end - ps < BS ? end - ps : BS;            /* slots in use after the write */
            for (int kv = 0; kv < 2; ++kv) {
                const uint16_t *src = kv ? new_v : new_k;
                char *pool = (char *)(kv ? v_pool : k_pool);
                float *scale = kv ? v_scale : k_scale;
                for (int h = 0; h < Hkv; ++h) {
                    const size_t tile = ((size_t)blk * Hkv + h) * BS * D; /* element offset of (blk, h) */
                    if (!fp8) {
                        uint16_t *t16 = (uint16_t *)pool + tile;
                        for (long s = hist; s < vend; ++s)
                            memcpy(t16 + s * D, src + (((size_t)b * n_new + (ps + s - L)) * Hkv + h) * D,
                                   (size_t)D * 2);
                        continue;
                    }
                    uint8_t *t8 = (uint8_t *)pool + tile;
                    if (fp8 == 2) {
                        for (long s = hist; s < vend; ++s)
                            for (int t0 = 0; t0 < D; t0 += 64) {
                                const uint16_t *row = src + (((size_t)b * n_new + (ps + s - L)) * Hkv + h) * D;
                                float amax = 0.f;
                                for (int d = t0; d < t0 + 64; ++d) {
                                    float v = bf16_bits_to_float(row[d]);
                                    float a = v < 0 ? -v : v;
                                    if (a > amax) amax = a;
                                }
                                volatile float sc = amax > 0.f ? amax / 448.0f : 1.0f;
                                for (int d = t0; d < t0 + 64; ++d) {
                                    volatile float q = bf16_bits_to_float(row[d]) / sc;
                                    t8[s * D + d] = oracle_e4m3_encode(q);
                                }
                                scale[(((long)blk * Hkv + h) * BS + s) * (D / 64) + t0 / 64] = sc;
                            }
                        for (long s = vend; s < BS; ++s) memset(t8 + s * D, 0, (size_t)D);
                        continue;
                    }
                    const float old_scale = scale[(long)blk * Hkv + h];
                    float amax = 0.f;
                    for (long s = 0; s < hist; ++s)
                        for (int d = 0; d < D; ++d) {
                            volatile float v = (float)oracle_e4m3_to_double(t8[s * D + d]) * old_scale;
                            float a = v < 0 ? -v : v;
                            if (a > amax) amax = a;
                        }
                    for (long s = hist; s < vend; ++s)
                        for (int d = 0; d < D; ++d) {
                            float v = bf16_bits_to_float(src[(((size_t)b * n_new + (ps + s - L)) * Hkv + h) * D + d]);
                            float a = v < 0 ? -v : v;
                            if (a > amax) amax = a;
                        }
                    volatile float new_scale = amax > 0.f ? amax / 448.0f : 1.0f;
                    if (hist > 0 && new_scale != old_scale)
                        for (long s = 0; s < hist; ++s)
                            for (int d = 0; d < D; ++d) {
                                volatile float v = (float)oracle_e4m3_to_double(t8[s * D + d]) * old_scale;
                                volatile float q = v / new_scale;
                                t8[s * D + d] = oracle_e4m3_encode(q);
                            }
                    for (long s = hist; s < vend; ++s)
                        for (int d = 0; d < D; ++d) {
                            float v = bf16_bits_to_float(src[(((size_t)b * n_new + (ps + s - L)) * Hkv + h) * D + d]);
                            volatile float q = v / new_scale;
                            t8[s * D + d] = oracle_e4m3_encode(q);
                        }
                    for (long s = vend; s < BS; ++s) memset(t8 + s * D, 0, (size_t)D);
                    scale[(long)blk * Hkv + h] = new_scale;
                }
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* speed-up model                                                      */
/* ------------------------------------------------------------------ */

/* E[K] = sum_{i=1}^{gamma} prod_{j=1}^{i} alpha_j */
double oracle_expected_accepted(const double *alpha, int gamma) {
    double total = 0.0, prod = 1.0;
    for (int i = 0; i < gamma; ++i) {
        prod *= alpha[i];
        total += prod;
    }
    return total;
}

/* eta = (E[K] + 1) / (gamma * r + 1), r = t_draft / t_target */
double oracle_speedup(double expected_accepted, int gamma, double r) {
    return (expected_accepted + 1.0) / ((double)gamma * r + 1.0);
}

/* ------------------------------------------------------------------ */
/*
 * Acceptance telemetry and the adaptive draft length.
 *
 * "Speculative Decoding & KV-Cache PagedAttention in Enterprise LLM
 * Serving": the lookahead follows a moving average of the acceptance rate
 * (above 0.85 -> 5 drafts, above 0.70 -> 4, above 0.50 -> 3, else 2);
 * "The Sub-Millisecond Speculative Decoding Meltdown", production failure
 * scenarios: when the exponential moving average of acceptance collapses
 * below 0.25, fall back to one token; "LOW-LATENCY INFERENCE: SPECULATIVE
 * DECODING & PAGING", acceptance math: E[K] = sum_{i=1..gamma} alpha^i for a
 * per-token rate alpha, speed-up (E[K] + 1) / (gamma * r + 1).
 *
 * One step with g drafts per sequence: a sequence that accepted k drafts ran
 * k + (k < g) acceptance tests (the k that passed and, if any, the one that
 * failed), so accepted / tests estimates the per-token rate.  Moving averages
 * in fp32, each product and sum rounded on its own (no fused multiply-add):
 *   A = decay * A + k,  N = decay * N + tests,  alpha = A / N.
 * Per sequence: state[b] = (A, N), gamma_next[b] from its alpha.  The batch
 * keeps its own (A, N) over the step's integer totals (sum k, sum tests), so
 * its gamma does not depend on the order of a sum.  Draft length from alpha:
 * > 0.85 -> 5, > 0.70 -> 4, > 0.50 -> 3, >= 0.25 -> 2, else 1.
 * telemetry: [0] batch alpha, [1] mean accepted per sequence this step,
 * [2] E[K] at (batch alpha, batch gamma), [3] speed-up at ratio r — fp32,
 * E[K] as the running product and sum in increasing i.
 */
int oracle_gamma_from_alpha(float alpha) {
    if (alpha > 0.85f) return 5;
    if (alpha > 0.70f) return 4;
    if (alpha > 0.50f) return 3;
    if (alpha >= 0.25f) return 2;
    return 1;
}

int oracle_gamma_update(int B, int gamma, const int32_t *accepted_len, float *seq_state,
                        int32_t *seq_gamma_next, float *batch_state, int32_t *batch_gamma_next,
                        float *telemetry, float decay, float r) {
    if (B < 1 || gamma < 1 || !accepted_len || !batch_state || !batch_gamma_next || !telemetry)
        return ORC_ERR_ARG;
    long long sum_k = 0, sum_t = 0;
    for (int b = 0; b < B; ++b) {
        const int k = accepted_len[b];
        if (k < 0 || k > gamma) return ORC_ERR_ARG;
        const int tests = k + (k < gamma ? 1 : 0);
        sum_k += k;
        sum_t += tests;
        if (seq_state) {
            volatile float a = decay * seq_state[2 * b];
            volatile float n = decay * seq_state[2 * b + 1];
            a = a + (float)k;
            n = n + (float)tests;
            seq_state[2 * b] = a;
            seq_state[2 * b + 1] = n;
            if (seq_gamma_next) {
                volatile float alpha = a / n;
                seq_gamma_next[b] = oracle_gamma_from_alpha(alpha);
            }
        }
    }
    volatile float a = decay * batch_state[0];
    volatile float n = decay * batch_state[1];
    a = a + (float)sum_k;
    n = n + (float)sum_t;
    batch_state[0] = a;
    batch_state[1] = n;
    volatile float alpha = a / n;
    const int g = oracle_gamma_from_alpha(alpha);
    *batch_gamma_next = g;
    volatile float ek = 0.f, prod = 1.f;
    for (int i = 0; i < g; ++i) {
        prod = prod * alpha;
        ek = ek + prod;
    }
    volatile float den = (float)g * r;
    den = den + 1.f;
    volatile float eta = ek + 1.f;
    eta = eta / den;
    telemetry[0] = alpha;
    telemetry[1] = (float)sum_k / (float)B;
    telemetry[2] = ek;
    telemetry[3] = eta;
    return ORC_OK;
}
