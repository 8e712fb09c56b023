/*
 * oracle.c -- plain, slow, obviously correct CPU oracle for the verify-and-accept
 * hot path of MTP speculative decoding.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The CUDA product path
 * never calls it and shares no code, header, table or constant with it.
 *
 * Every floating-point result is accumulated in double precision (float64);
 * inputs are the same fp32 / bf16 bit patterns the GPU path receives.  Build
 * with -ffp-contract=off so that no multiply-add is fused behind our back.
 *
 * Sources (web pages; cited by title and section):
 *  [MTPLX]  "MTPLX 2.24x faster TPS -- the native MTP inference engine"
 *           (molayo1419.me), sections "Architecture / Layer 0: MLX Runtime"
 *           (small-M verify qmv, innovation-tape GDN capture) and
 *           "Layer 2: Speculative cycle (the hot loop)" (fp32 Leviathan-Chen
 *           probability-ratio acceptance, (p-q)+ residual, bonus token,
 *           tape commit / rollback), and "QWEN 3.6 27B @ 63 TPS" (temperature
 *           0.6, top_p 0.95, top_k 20).
 *  [LLAMA]  "MTP in llama.cpp" (habr article, savepearlharbor.com copy),
 *           sections "How speculative decoding works" and "lossless": the
 *           greedy accept-until-mismatch loop with one extra token.
 *  [MLXCEL] "MTP와 DFlash" (mlxcel manual), section "Qwen3.8-Flash-Next
 *           (qwen4_exp) MTP": rollback replays the GatedDeltaNet recurrence
 *           over the accepted tokens.
 * Readings adopted where the pages are silent are stated at each function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* error-flag bits written per sequence by oracle_spec_accept */
#define OF_DRAFT_OUT_OF_RANGE 1 /* draft token not in [0, V)                    */
#define OF_DRAFT_ZERO_Q       2 /* q_k(d_k) == 0: the draft could not be drawn  */
#define OF_NONFINITE_LOGIT    4 /* NaN or +inf logit in a row that was used     */
#define OF_EMPTY_DIST         8 /* a distribution to sample from had no mass    */

static int g_threads = 1;

int oracle_abi_version(void) { return 1; }

void oracle_set_threads(int n) { g_threads = n < 1 ? 1 : n; }

int oracle_has_openmp(void) {
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_value(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* qmv: Y[M,N] = X[M,K] . W^T with a 4-bit affine group-64 weight.           */
/* ------------------------------------------------------------------------ */
/*
 * [MTPLX] "Layer 0": the verify step multiplies the M = K+1 verify rows by the
 * 4-bit quantised weights ("Qwen 3.6 27B 4-bit MLX").  The pages do not print
 * the bit layout; the reading adopted here:
 *   W[n,i] = s[n, i/gs] * q[n,i] + b[n, i/gs]          (gs = group_size = 64)
 *   q[n,i] = (w_packed[n, i/8] >> (4*(i%8))) & 15      (nibbles LSB-first)
 *   s, b   : bf16, row-major [N, K/gs];  X: fp32 or bf16 row-major [M, K].
 * The oracle is that definition written out, accumulated in float64 and
 * rounded to fp32 once at the end.
 */
int oracle_qmv(const uint32_t *w_packed, const uint16_t *scales, const uint16_t *biases,
               const void *x, int x_is_bf16, float *y, int M, int N, int K, int group_size) {
    if (M < 0 || N < 0 || K < 0 || group_size <= 0 || K % group_size != 0 || K % 8 != 0)
        return 1;
    const int groups = K / group_size;
    const int words = K / 8;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(g_threads)
#endif
    for (int n = 0; n < N; ++n) {
        for (int m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int i = 0; i < K; ++i) {
                uint32_t word = w_packed[(size_t)n * words + i / 8];
                int q = (int)((word >> (4 * (i % 8))) & 15u);
                double s = bf16_value(scales[(size_t)n * groups + i / group_size]);
                double b = bf16_value(biases[(size_t)n * groups + i / group_size]);
                double wv = s * (double)q + b;
                double xv = x_is_bf16 ? bf16_value(((const uint16_t *)x)[(size_t)m * K + i])
                                      : (double)((const float *)x)[(size_t)m * K + i];
                acc += xv * wv;
            }
            y[(size_t)m * N + n] = (float)acc;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Requantisation of a bf16 weight matrix to the 4-bit affine group format.  */
/* ------------------------------------------------------------------------ */
/*
 * [MTPLX] "Layer 0: MLX Runtime", the draft-only requantised LM head: the
 * target keeps its LM head at model precision and a separate 4-bit copy is
 * built in memory for the drafter.  The pages do not print the quantiser;
 * the reading adopted is the plain min/max affine one, in the qmv layout:
 *   per group of 64 inputs of a row:  lo = min w, hi = max w
 *   s = rn_bf16((hi - lo) / 15),  b = lo (a bf16 value already)
 *   q = 0 if s == 0, else clamp(rint((w - b) / s), 0, 15)
 * with every step an fp32 operation (subtraction, division, round half to
 * even): the code is an integer decided by floating point, so the oracle
 * takes the decision in the precision the product takes it in.  A zero
 * minimum or maximum is taken as +0 (which zero is smallest or largest is no
 * property of the group).  The weights are finite.
 */
static uint16_t bf16_rn_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u) return (uint16_t)(u >> 16); /* inf: no rounding */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb; /* round to nearest, ties to even */
    return (uint16_t)(u >> 16);
}

static float bf16_float(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

int oracle_requantize(const uint16_t *w, int N, int K, uint32_t *w_packed, uint16_t *scales,
                      uint16_t *biases) {
    if (N < 0 || K <= 0 || K % 64 != 0) return 1;
    const int groups = K / 64;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(g_threads)
#endif
    for (int n = 0; n < N; ++n) {
        for (int g = 0; g < groups; ++g) {
            const uint16_t *src = w + (size_t)n * K + (size_t)g * 64;
            float lo = bf16_float(src[0]), hi = lo;
            for (int i = 1; i < 64; ++i) {
                float v = bf16_float(src[i]);
                if (v < lo) lo = v;
                if (v > hi) hi = v;
            }
            if (lo == 0.0f) lo = 0.0f;              /* +0 */
            if (hi == 0.0f) hi = 0.0f;
            volatile float range = hi - lo;         /* fp32, one rounding */
            volatile float step = range / 15.0f;    /* fp32, one rounding */
            uint16_t s_bits = bf16_rn_bits(step);
            uint16_t b_bits = bf16_rn_bits(lo);     /* exact: lo is a bf16 value */
            float s = bf16_float(s_bits), b = bf16_float(b_bits);
            scales[(size_t)n * groups + g] = s_bits;
            biases[(size_t)n * groups + g] = b_bits;
            for (int word = 0; word < 8; ++word) {
                uint32_t packed = 0;
                for (int j = 0; j < 8; ++j) {
                    int q = 0;
                    if (s != 0.0f) {
                        volatile float diff = bf16_float(src[8 * word + j]) - b;
                        volatile float ratio = diff / s;
                        float r = rintf(ratio);
                        q = r < 0.0f ? 0 : (r > 15.0f ? 15 : (int)r);
                    }
                    packed |= (uint32_t)q << (4 * j);
                }
                w_packed[(size_t)n * (K / 8) + (size_t)g * 8 + word] = packed;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Sampling distribution of one logits row: temperature -> top-k -> top-p.   */
/* ------------------------------------------------------------------------ */
typedef struct {
    int idx;
    double key;
} cand_t;

/* order: larger key first; equal keys -> lower token id first */
static int cand_cmp(const void *a, const void *b) {
    const cand_t *x = (const cand_t *)a, *y = (const cand_t *)b;
    if (x->key > y->key) return -1;
    if (x->key < y->key) return 1;
    return (x->idx > y->idx) - (x->idx < y->idx);
}

/*
 * Fills p[0..V) with the filtered distribution of logits row z.
 * [MTPLX] "QWEN 3.6 27B @ 63 TPS" names the three settings (temperature, top_p,
 * top_k) but not their order.  Reading adopted (plainest, and the usual one):
 *   1. z' = z / T                          (T > 0)
 *   2. top-k: keep the k largest z'; equal values -> lower token id; exactly
 *      min(k, #finite) are kept.  k <= 0 or k >= V disables the filter.
 *   3. softmax over the kept set (float64).
 *   4. top-p: in descending probability (ties -> lower id) keep the shortest
 *      prefix whose cumulative probability is >= top_p, at least one token.
 *      top_p >= 1 disables the filter.
 *   5. renormalise over what is kept.
 * Non-finite logits: -inf is a legitimate mask value (never kept); NaN and
 * +inf are never kept and raise OF_NONFINITE_LOGIT.  A row with no finite
 * logit gives the all-zero vector (an empty distribution).
 * T == 0 gives the greedy one-hot on argmax z (lowest id on ties).
 * *topp_margin (if not NULL) receives min(top_p - cum_{c-1}, cum_c - top_p)
 * for the cut position c, or +inf when top-p did not apply.
 * Returns the number of tokens with nonzero probability.
 */
int oracle_filter_row(const float *z, int V, double temperature, int top_k, double top_p,
                      double *p, int *flags, double *topp_margin) {
    int nfinite = 0;
    if (topp_margin) *topp_margin = INFINITY;
    for (int x = 0; x < V; ++x) {
        p[x] = 0.0;
        if (isnan(z[x]) || (isinf(z[x]) && z[x] > 0)) {
            if (flags) *flags |= OF_NONFINITE_LOGIT;
        } else if (isfinite(z[x])) {
            ++nfinite;
        }
    }
    if (nfinite == 0) return 0;

    if (temperature == 0.0) { /* greedy */
        int best = -1;
        for (int x = 0; x < V; ++x)
            if (isfinite(z[x]) && (best < 0 || z[x] > z[best])) best = x;
        p[best] = 1.0;
        return 1;
    }

    cand_t *c = (cand_t *)malloc(sizeof(cand_t) * (size_t)nfinite);
    int n = 0;
    for (int x = 0; x < V; ++x)
        if (isfinite(z[x])) {
            c[n].idx = x;
            c[n].key = (double)z[x] / temperature;
            ++n;
        }
    qsort(c, (size_t)n, sizeof(cand_t), cand_cmp);
    int kept = n;
    if (top_k > 0 && top_k < V && top_k < kept) kept = top_k;

    /* softmax over the kept set; c[0] holds the largest z' */
    double zmax = c[0].key, sum = 0.0;
    for (int j = 0; j < kept; ++j) {
        c[j].key = exp(c[j].key - zmax);
        sum += c[j].key;
    }
    for (int j = 0; j < kept; ++j) c[j].key /= sum;

    if (top_p < 1.0) {
        /* re-sort by probability (descending, ties -> lower id) */
        qsort(c, (size_t)kept, sizeof(cand_t), cand_cmp);
        double cum = 0.0, prev = 0.0;
        int cut = kept;
        for (int j = 0; j < kept; ++j) {
            prev = cum;
            cum += c[j].key;
            if (cum >= top_p) {
                cut = j + 1;
                break;
            }
        }
        if (topp_margin) {
            double a = top_p - prev, b = cum - top_p;
            *topp_margin = fabs(a) < fabs(b) ? fabs(a) : fabs(b);
        }
        kept = cut;
        double s2 = 0.0;
        for (int j = 0; j < kept; ++j) s2 += c[j].key;
        for (int j = 0; j < kept; ++j) c[j].key /= s2;
    }
    for (int j = 0; j < kept; ++j) p[c[j].idx] = c[j].key;
    free(c);
    return kept;
}

/*
 * Inverse CDF in ascending token-id order: the smallest x with
 * sum_{y<=x} R(y) > u * Z, Z = sum R.  (Reading adopted: the pages fix no
 * sampling order or random-number generator; the uniform u is an input.)
 * If rounding leaves the running sum <= u*Z at the end, the last token with
 * R > 0 is returned.  Returns -1 when Z <= 0 (nothing to sample).
 * *margin receives the smallest |C_x - u Z| / Z over the tokens visited.
 */
static int inverse_cdf(const double *R, int V, double u, double *margin) {
    double Z = 0.0;
    for (int x = 0; x < V; ++x) Z += R[x];
    if (!(Z > 0.0)) return -1;
    double thr = u * Z, C = 0.0;
    int last = -1;
    for (int x = 0; x < V; ++x) {
        if (R[x] > 0.0) {
            C += R[x];
            last = x;
            double m = fabs(C - thr) / Z;
            if (margin && m < *margin) *margin = m;
            if (C > thr) return x;
        }
    }
    return last;
}

/*
 * Verify-and-accept for B sequences with K drafted tokens each.
 * [MTPLX] "Layer 2: Speculative cycle": per position, in fp32 (here float64),
 * accept the draft with probability min(1, p/q) (Leviathan et al. 2023;
 * Chen et al. 2023); on the first rejection emit a replacement drawn from
 * norm((p - q)+) and stop; when all K are accepted emit a bonus token from the
 * target distribution at position K+1.
 * [LLAMA] "How speculative decoding works": temperature 0 reduces to the greedy
 * loop -- accept while the draft equals the target's argmax, stop at the first
 * mismatch emitting the argmax, and take one more argmax token when all match.
 *
 * Layout: target_logits [B][K+1][V], draft_logits [B][K][V] (fp32),
 * draft_tokens [B][K], u_accept [B][K], u_sample [B].
 * Outputs: out_tokens [B][K+1] (-1 padded), n_accepted [B], err_flags [B]
 * (may be NULL), diag [B][3] (may be NULL): the smallest accept margin
 * |u_k - p/q|, top-p margin and inverse-CDF margin met on the path taken
 * (+inf where none).  Readings adopted:
 *  - u_k < p_k(d_k)/q_k(d_k) accepts;  q_k(d_k) == 0 rejects (OF_DRAFT_ZERO_Q);
 *    a draft token outside [0,V) rejects (OF_DRAFT_OUT_OF_RANGE).
 *  - if Z = sum (p-q)+ <= 0 the replacement is drawn from p instead.
 *  - one uniform u_sample per sequence: at most one token is ever drawn.
 *  - greedy (T == 0) never reads the draft logits.
 */
int oracle_spec_accept(const float *target_logits, const float *draft_logits,
                       const int32_t *draft_tokens, const float *u_accept, const float *u_sample,
                       int B, int K, int V, double temperature, int top_k, double top_p,
                       int32_t *out_tokens, int32_t *n_accepted, int32_t *err_flags, double *diag) {
    if (B < 0 || K < 1 || V < 1 || temperature < 0.0 || !(top_p > 0.0)) return 1;
    double *p = (double *)malloc(sizeof(double) * (size_t)V);
    double *q = (double *)malloc(sizeof(double) * (size_t)V);
    double *R = (double *)malloc(sizeof(double) * (size_t)V);
    for (int b = 0; b < B; ++b) {
        int flags = 0, nacc = 0;
        double m_acc = INFINITY, m_topp = INFINITY, m_cdf = INFINITY, mt;
        int32_t *tok = out_tokens + (size_t)b * (K + 1);
        for (int j = 0; j <= K; ++j) tok[j] = -1;
        int emitted = 0, stop = 0;
        for (int k = 0; k < K && !stop; ++k) {
            const float *zt = target_logits + ((size_t)b * (K + 1) + k) * V;
            const float *zd = draft_logits + ((size_t)b * K + k) * V;
            int d = draft_tokens[(size_t)b * K + k];
            oracle_filter_row(zt, V, temperature, top_k, top_p, p, &flags, &mt);
            if (mt < m_topp) m_topp = mt;
            int accept = 0;
            if (d < 0 || d >= V) {
                flags |= OF_DRAFT_OUT_OF_RANGE;
            } else if (temperature == 0.0) {
                accept = p[d] > 0.0; /* p is the one-hot argmax */
            } else {
                oracle_filter_row(zd, V, temperature, top_k, top_p, q, &flags, &mt);
                if (mt < m_topp) m_topp = mt;
                if (q[d] == 0.0) {
                    flags |= OF_DRAFT_ZERO_Q;
                } else {
                    double r = p[d] / q[d];
                    double u = (double)u_accept[(size_t)b * K + k];
                    double mg = fabs(u - r);
                    if (mg < m_acc) m_acc = mg;
                    accept = u < r;
                }
            }
            if (accept) {
                tok[k] = d;
                ++nacc;
                continue;
            }
            /* rejection at position k: draw the replacement */
            int x;
            if (temperature == 0.0) {
                /* greedy: the replacement is the argmax, the one token of p */
                x = -1;
                for (int y = 0; y < V; ++y)
                    if (p[y] > 0.0) x = y;
            } else {
                if (d < 0 || d >= V) { /* q was not evaluated above */
                    oracle_filter_row(zd, V, temperature, top_k, top_p, q, &flags, &mt);
                    if (mt < m_topp) m_topp = mt;
                }
                double Z = 0.0;
                for (int y = 0; y < V; ++y) {
                    double r = p[y] - q[y];
                    R[y] = r > 0.0 ? r : 0.0;
                    Z += R[y];
                }
                if (!(Z > 0.0)) memcpy(R, p, sizeof(double) * (size_t)V);
                x = inverse_cdf(R, V, (double)u_sample[b], &m_cdf);
            }
            if (x < 0) flags |= OF_EMPTY_DIST;
            tok[k] = x;
            emitted = 1;
            stop = 1;
        }
        if (!emitted) { /* all K accepted: bonus from position K+1 */
            const float *zt = target_logits + ((size_t)b * (K + 1) + K) * V;
            oracle_filter_row(zt, V, temperature, top_k, top_p, p, &flags, &mt);
            if (mt < m_topp) m_topp = mt;
            int x;
            if (temperature == 0.0) { /* greedy bonus: the argmax */
                x = -1;
                for (int y = 0; y < V; ++y)
                    if (p[y] > 0.0) x = y;
            } else {
                x = inverse_cdf(p, V, (double)u_sample[b], &m_cdf);
            }
            if (x < 0) flags |= OF_EMPTY_DIST;
            tok[K] = x;
        }
        n_accepted[b] = nacc;
        if (err_flags) err_flags[b] = flags;
        if (diag) {
            diag[(size_t)b * 3 + 0] = m_acc;
            diag[(size_t)b * 3 + 1] = m_topp;
            diag[(size_t)b * 3 + 2] = m_cdf;
        }
    }
    free(p);
    free(q);
    free(R);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* GatedDeltaNet recurrence and its innovation tape.                        */
/* ------------------------------------------------------------------------ */
/*
 * [MLXCEL] "Qwen3.8-Flash-Next (qwen4_exp) MTP" names the GatedDeltaNet
 * recurrence replayed over accepted tokens; [MTPLX] "Layer 0" records
 * (token, gate, state-delta) tuples so a rejection replays a small tape
 * instead of restoring a snapshot.  Neither page writes the update out.  The
 * reading adopted is the published gated delta rule (Yang, Kautz and
 * Hatamizadeh, "Gated Delta Networks", 2024), per (sequence b, head h), with
 * S in R^{dv x dk}:
 *     S'  = alpha_t * S                       (decay first)
 *     u   = S' k_t                            (ascending-j sum)
 *     e_t = beta_t * (v_t - u)                (the innovation)
 *     S_t = S' + e_t k_t^T                    (multiply, then add)
 *     o_t = S_t q_t
 * The tape record for (b,t,h) is (alpha_t, e_t, k_t): the gate and the rank-1
 * factors of the state delta.  Replaying L records applies
 *     S[i][j] <- alpha_t*S[i][j] + e_t[i]*k_t[j]
 * in order, which reproduces the sequential state after L tokens exactly.
 *
 * Layouts (all row-major): state [B][H][dv][dk]; q,k [B][T][H][dk];
 * v [B][T][H][dv]; alpha, beta [B][T][H]; out [B][T][H][dv];
 * oracle tape: alpha [B][T][H], e [B][T][H][dv], k [B][T][H][dk] (float64).
 */

/* One recurrence step on one head: S (dv x dk, float64) in place.  Writes e
 * (dv) and o (dv) when not NULL. */
static void gdn_step(double *S, int dk, int dv, const float *q, const float *k, const float *v,
                     double alpha, double beta, double *e, double *o) {
    for (int i = 0; i < dv * dk; ++i) S[i] = alpha * S[i];
    for (int i = 0; i < dv; ++i) {
        double u = 0.0;
        for (int j = 0; j < dk; ++j) u += S[(size_t)i * dk + j] * (double)k[j];
        double ei = beta * ((double)v[i] - u);
        if (e) e[i] = ei;
        for (int j = 0; j < dk; ++j) {
            double d = ei * (double)k[j];
            S[(size_t)i * dk + j] = S[(size_t)i * dk + j] + d;
        }
    }
    if (o) {
        for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * (double)q[j];
            o[i] = acc;
        }
    }
}

/* Runs n_steps[b] recurrence steps (0..T) on state (float64, in place) for
 * every (b,h).  out [B][T][H][dv] (may be NULL) receives o_t for the steps
 * taken. */
void oracle_gdn_sequential(double *state, const float *q, const float *k, const float *v,
                           const float *alpha, const float *beta, const int32_t *n_steps,
                           int B, int T, int H, int dk, int dv, double *out) {
#ifdef _OPENMP
#pragma omp parallel for collapse(2) schedule(static) num_threads(g_threads)
#endif
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            double *S = state + ((size_t)b * H + h) * dv * dk;
            int L = n_steps ? n_steps[b] : T;
            for (int t = 0; t < L; ++t) {
                size_t bth = ((size_t)b * T + t) * H + h;
                gdn_step(S, dk, dv, q + bth * dk, k + bth * dk, v + bth * dv,
                         (double)alpha[bth], (double)beta[bth], NULL,
                         out ? out + bth * dv : NULL);
            }
        }
}

/* Capture: runs all T steps from the fp32 snapshot state0 (never written) and
 * records the tape; out [B][T][H][dv] (may be NULL). */
void oracle_gdn_capture(const float *state0, const float *q, const float *k, const float *v,
                        const float *alpha, const float *beta, int B, int T, int H, int dk,
                        int dv, double *out, double *tape_alpha, double *tape_e,
                        double *tape_k) {
#ifdef _OPENMP
#pragma omp parallel for collapse(2) schedule(static) num_threads(g_threads)
#endif
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            size_t bh = (size_t)b * H + h;
            double *S = (double *)malloc(sizeof(double) * (size_t)dv * dk);
            for (int i = 0; i < dv * dk; ++i) S[i] = (double)state0[bh * dv * dk + i];
            for (int t = 0; t < T; ++t) {
                size_t bth = ((size_t)b * T + t) * H + h;
                gdn_step(S, dk, dv, q + bth * dk, k + bth * dk, v + bth * dv,
                         (double)alpha[bth], (double)beta[bth], tape_e + bth * dv,
                         out ? out + bth * dv : NULL);
                tape_alpha[bth] = (double)alpha[bth];
                for (int j = 0; j < dk; ++j) tape_k[bth * dk + j] = (double)k[bth * dk + j];
            }
            free(S);
        }
}

/* Replay: applies the first n_replay[b] tape records of every (b,h) to state
 * (float64, in place).  n_replay[b] == 0 leaves the state unchanged. */
void oracle_gdn_replay(double *state, const double *tape_alpha, const double *tape_e,
                       const double *tape_k, const int32_t *n_replay, int B, int T, int H,
                       int dk, int dv) {
#ifdef _OPENMP
#pragma omp parallel for collapse(2) schedule(static) num_threads(g_threads)
#endif
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            double *S = state + ((size_t)b * H + h) * dv * dk;
            for (int t = 0; t < n_replay[b]; ++t) {
                size_t bth = ((size_t)b * T + t) * H + h;
                double a = tape_alpha[bth];
                const double *e = tape_e + bth * dv;
                const double *kk = tape_k + bth * dk;
                for (int i = 0; i < dv; ++i)
                    for (int j = 0; j < dk; ++j) {
                        double decayed = a * S[(size_t)i * dk + j];
                        double delta = e[i] * kk[j];
                        S[(size_t)i * dk + j] = decayed + delta;
                    }
            }
        }
}

/* ------------------------------------------------------------------------
 * Short causal convolution windows of a GatedDeltaNet layer.
 * [MLXCEL] "MTP와 DFlash", section "Qwen3.8-Flash-Next (qwen4_exp) MTP": the
 * rollback replays the GatedDeltaNet recurrence and two convolution windows
 * over the accepted tokens; the batched DFlash paragraph of the same page:
 * linear-attention layers replay the convolution and recurrent state over
 * each row's accepted prefix.  The pages give no formula; the reading
 * adopted is the depthwise causal convolution of width W over a channel
 * stream, whose state is the W-1 most recent inputs of every channel:
 *   h(tau) = x[tau][c] for tau >= 0, window[W-1+tau][c] for -(W-1) <= tau < 0
 *   y[t][c] = sum_{j=0}^{W-1} weight[j][c] * h(t - (W-1) + j)
 * Layouts (time-major): window [B][W-1][C], x and y [B][T][C], weight [W][C].
 * ------------------------------------------------------------------------ */
static double conv_h(const double *win, const double *x, int W, int C, int c, int tau) {
    return tau >= 0 ? x[(size_t)tau * C + c] : win[(size_t)(W - 1 + tau) * C + c];
}

/* Capture: outputs of the T verify tokens from the committed window, which is
 * left unchanged.  Sum in ascending j. */
void oracle_conv_capture(const double *window, const double *x, const double *weight, int B,
                         int T, int C, int W, double *y) {
    for (int b = 0; b < B; ++b) {
        const double *win = window + (size_t)b * (W - 1) * C;
        const double *xb = x + (size_t)b * T * C;
        for (int t = 0; t < T; ++t)
            for (int c = 0; c < C; ++c) {
                double s = 0.0;
                for (int j = 0; j < W; ++j)
                    s += weight[(size_t)j * C + c] * conv_h(win, xb, W, C, c, t - (W - 1) + j);
                y[((size_t)b * T + t) * C + c] = s;
            }
    }
}

/* Replay (commit): the window after the first L_b = n_replay[b] verify tokens
 * is the last W-1 entries of (old window, x[0..L_b)); L_b = 0 leaves it as it
 * is.  Written as W-1 positions of h, not as a shift, so that a test can
 * compare it with shifting the window one token at a time. */
void oracle_conv_replay(double *window, const double *x, const int32_t *n_replay, int B, int T,
                        int C, int W) {
    double *tmp = (double *)malloc(sizeof(double) * (size_t)(W > 1 ? W - 1 : 1) * C);
    for (int b = 0; b < B; ++b) {
        double *win = window + (size_t)b * (W - 1) * C;
        const double *xb = x + (size_t)b * T * C;
        const int L = n_replay[b];
        for (int i = 0; i < W - 1; ++i)
            for (int c = 0; c < C; ++c)
                tmp[(size_t)i * C + c] = conv_h(win, xb, W, C, c, L - (W - 1) + i);
        memcpy(win, tmp, sizeof(double) * (size_t)(W - 1) * C);
    }
    free(tmp);
}
