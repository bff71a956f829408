/*
 * Plain fp64 CPU oracle of the memory-efficient ("linear") GRPO loss.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the CPU baseline
 * leg of the benchmark call this code to obtain expected values; the library
 * itself never links, loads or calls it, and the two share no code.
 *
 * What is computed, and where the pages fix it:
 *   - Group-relative advantages: responses of one prompt form a group; each
 *     reward is compared with the group mean and the better responses are
 *     reinforced ("Train your own R1 reasoning model with Unsloth", section 3,
 *     steps 3-5).  The spread normaliser (sample std + eps) is the reading the
 *     workload definitions take; the pages print no formula.
 *   - Token log-probabilities of the sampled tokens under the trained policy
 *     (q) and the frozen reference (p), computed from the lm_head logits with
 *     the logsumexp trick ("Long-context GRPO", section 4, last paragraph).
 *     The linear algorithm never stores the logits; it reaches exactly the
 *     same numbers as materialising them ("Long-context GRPO", section 2),
 *     so the oracle is that plain definition.
 *   - Per-token objective with the policy-gradient factor exp(q - sg(q)) * A,
 *     whose value is A and whose gradient w.r.t. q is A ("Long-context GRPO",
 *     section 4, the detach fragment), and the reverse-KL penalty with
 *     beta = 0.04 in its unbiased form exp(p-q) - (p-q) - 1 that needs no
 *     extra Q factor (same section).  KL is evaluated as expm1(x) - x.
 *   - Mean over completion tokens (mask), gradient to the hidden states and
 *     to the lm_head weight.
 *   - The variants of the four-way experiment of the same section and a
 *     per-completion mean; the pages give no formulas for these (their
 *     images are lost), so they follow the readings stated at each function.
 *     The three objective variants (no detach, reverse KL times Q, forward
 *     KL) are parity unpinned against the pages: the tests pin each one's
 *     gradient to its own value by finite differences, but nothing on the
 *     pages fixes the values themselves.
 *   - Exact decoders of the OCP FP8 formats E4M3 and E5M2 (the 8-bit forward
 *     reads its inputs as code * scale).
 *
 * Everything is fp64 on inputs widened exactly from their storage type
 * (bf16 / fp16 / double).  Sums run in ascending index order.  OpenMP only
 * splits independent rows (or independent vocabulary rows for dW) across
 * threads, so results do not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F64 = 0, OR_BF16 = 1, OR_F16 = 2 };

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- exact widening of the storage types -------------------------------- */

double oracle_bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

double oracle_f16_to_f64(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 10) & 31;
    int m = b & 1023;
    double v;
    if (e == 0) v = ldexp((double)m, -24);                 /* subnormal / zero */
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp((double)(1024 + m), e - 25);
    return sign ? -v : v;
}

/* OCP FP8 E4M3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; no
 * infinities; S.1111.111 is NaN; largest finite 448, smallest subnormal 2^-9. */
double oracle_e4m3_to_f64(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 15;
    int m = b & 7;
    double v;
    if (e == 15 && m == 7) v = NAN;
    else if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp((double)(8 + m), e - 10);
    return sign ? -v : v;
}

/* OCP FP8 E5M2: 1 sign, 5 exponent bits (bias 15), 2 mantissa bits; exponent
 * field 31 holds the infinities (mantissa 0) and NaNs; largest finite 57344,
 * smallest normal 2^-14, smallest subnormal 2^-16. */
double oracle_e5m2_to_f64(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 2) & 31;
    int m = b & 3;
    double v;
    if (e == 31) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m, -16);
    else v = ldexp((double)(4 + m), e - 17);
    return sign ? -v : v;
}

/* The value of every bf16 and fp16 bit pattern, filled by the decoders above
 * when the library loads: the same values, without a call per element in the
 * row loops below. */
static double bf16_value[65536];
static double f16_value[65536];

__attribute__((constructor)) static void fill_16bit_values(void) {
    for (uint32_t b = 0; b < 65536u; ++b) {
        bf16_value[b] = oracle_bf16_to_f64((uint16_t)b);
        f16_value[b] = oracle_f16_to_f64((uint16_t)b);
    }
}

static inline double ld(const void* p, int type, size_t i) {
    if (type == OR_BF16) return bf16_value[((const uint16_t*)p)[i]];
    if (type == OR_F16) return f16_value[((const uint16_t*)p)[i]];
    return ((const double*)p)[i];
}

/* ---- advantages ---------------------------------------------------------- */

/* rewards [n_groups*G] -> adv [n_groups*G]; fp64 with left-to-right sums,
 * rounded once to fp32.  sigma uses divisor G-1 (std_unbiased) or G; a group
 * whose divisor is 0 has sigma = 0. */
void oracle_group_advantages(const float* rewards, int n_groups, int G, float eps,
                             int std_unbiased, float* adv) {
    for (int gi = 0; gi < n_groups; ++gi) {
        const float* r = rewards + (size_t)gi * G;
        double sum = 0.0;
        for (int i = 0; i < G; ++i) sum = sum + (double)r[i];
        double mu = sum / (double)G;
        double ss = 0.0;
        for (int i = 0; i < G; ++i) {
            double dv = (double)r[i] - mu;
            ss = ss + dv * dv;
        }
        int div = std_unbiased ? G - 1 : G;
        double sigma = div > 0 ? sqrt(ss / (double)div) : 0.0;
        double den = sigma + (double)eps;
        for (int i = 0; i < G; ++i) adv[(size_t)gi * G + i] = (float)(((double)r[i] - mu) / den);
    }
}

/* ---- mask and valid-row index -------------------------------------------- */

/* completion i occupies positions j < len_i of its L-row block */
void oracle_build_mask(const int32_t* lengths, int n_seq, int L, uint8_t* mask) {
    for (int i = 0; i < n_seq; ++i)
        for (int j = 0; j < L; ++j) mask[(size_t)i * L + j] = (uint8_t)(j < lengths[i]);
}

int64_t oracle_valid_rows(const uint8_t* mask, int64_t N, int32_t* rows) {
    int64_t n = 0;
    for (int64_t t = 0; t < N; ++t)
        if (mask[t]) {
            if (rows) rows[n] = (int32_t)t;
            ++n;
        }
    return n;
}

/* counts of one shard of a batch: out[0] = masked-in rows, out[1] =
 * completions with at least one masked-in row */
void oracle_shard_counts(const uint8_t* mask, int n_seq, int L, int64_t* out) {
    out[0] = 0;
    out[1] = 0;
    for (int i = 0; i < n_seq; ++i) {
        int64_t c = 0;
        for (int j = 0; j < L; ++j) c += mask[(size_t)i * L + j] != 0;
        out[0] += c;
        out[1] += c > 0;
    }
}

/* ---- logits of one row and their logsumexp ------------------------------ */

/* widen row r of a [*, d] matrix into out[d] */
static void load_row(const void* M, int type, int64_t r, int d, double* out) {
    for (int k = 0; k < d; ++k) out[k] = ld(M, type, (size_t)r * d + k);
}

/* dot(h, W[v,:]) with h already widened; sum in ascending k */
static inline double dot_w(const double* h, const void* W, int type, int v, int d) {
    double acc = 0.0;
    if (type == OR_BF16) {
        const uint16_t* w = (const uint16_t*)W + (size_t)v * d;
        for (int k = 0; k < d; ++k) acc = acc + h[k] * bf16_value[w[k]];
    } else if (type == OR_F16) {
        const uint16_t* w = (const uint16_t*)W + (size_t)v * d;
        for (int k = 0; k < d; ++k) acc = acc + h[k] * f16_value[w[k]];
    } else {
        const double* w = (const double*)W + (size_t)v * d;
        for (int k = 0; k < d; ++k) acc = acc + h[k] * w[k];
    }
    return acc;
}

/* z[v] = sum_k h[t,k] * W[v,k] for all v (hrow: scratch of d doubles) */
static void row_logits(const void* H, const void* W, int type, int64_t t, int d, int V, double* z,
                       double* hrow) {
    load_row(H, type, t, d, hrow);
    for (int v = 0; v < V; ++v) z[v] = dot_w(hrow, W, type, v, d);
}

/* log sum_v exp(z_v), computed as m + log sum exp(z - m) */
double oracle_logsumexp(const double* z, int V) {
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) m = z[v] > m ? z[v] : m;
    double s = 0.0;
    for (int v = 0; v < V; ++v) s = s + exp(z[v] - m);
    return m + log(s);
}

/* ---- per-row forward terms ----------------------------------------------- */

/* Objectives of the four-way experiment ("Long-context GRPO", section 4), with
 * x = p - q (reference minus policy log-prob of the sampled token):
 *   0  GRPO as implemented: detached factor exp(q - sg q) * A and the
 *      reverse-KL estimator pen = exp(x) - x - 1
 *   1  the same without the detach: exp(q - q) is the constant 1, so the
 *      policy-gradient term carries no gradient
 *   2  the reverse-KL term multiplied by Q, the policy probability of the
 *      token: pen = exp(q) (exp(x) - x - 1)
 *   3  forward KL instead: pen = exp(-x) + x - 1
 * The per-token objective is ell = -A + beta * pen (the policy-gradient
 * factor has value 1 in every variant) and g = d ell / d q of the surrogate
 * in which sg(q) is a constant. */
static void objective_terms(int objective, double A, double q, double p, double beta, double* pen,
                            double* ell, double* g) {
    double x = p - q;
    double k_rev = expm1(x) - x;                  /* exp(x) - x - 1 without cancellation */
    switch (objective) {
        case 1:
            *pen = k_rev;
            *g = -beta * expm1(x);                /* d/dq beta (e^x - x - 1) */
            break;
        case 2:
            *pen = exp(q) * k_rev;
            *g = -A - beta * x * exp(q);          /* d/dq e^q (e^x - x - 1) = -x e^q */
            break;
        case 3:
            *pen = expm1(-x) + x;                 /* exp(q-p) - (q-p) - 1 */
            *g = -A + beta * expm1(-x);           /* d/dq: e^(q-p) - 1 */
            break;
        default:
            *pen = k_rev;
            *g = -A - beta * expm1(x);            /* -A + beta (1 - e^x) */
            break;
    }
    *ell = -A + beta * *pen;
}

/* out[i*9 + .] for row t = rows[i]:
 *   0 lse_pol  1 lse_ref  2 z_pol[tok]  3 z_ref[tok]  4 q  5 p  6 pen  7 ell  8 g
 * adv is per sequence; row t belongs to sequence t / L.
 * The reference logits use W_ref (NULL: the same W).  The frozen reference
 * is a constant of the objective: no gradient is taken through it. */
void oracle_row_terms(const void* h_pol, const void* h_ref, const void* W, const void* W_ref,
                      int type, const int32_t* tokens, const float* adv, int L, int d, int V,
                      double beta, int objective, const int32_t* rows, int64_t n_rows, double* out) {
    if (!W_ref) W_ref = W;
#pragma omp parallel
    {
        double* z = (double*)malloc(sizeof(double) * (size_t)V);
        double* hrow = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_rows; ++i) {
            int64_t t = rows[i];
            int tok = tokens[t];
            double A = (double)adv[t / L];
            row_logits(h_pol, W, type, t, d, V, z, hrow);
            double lse_pol = oracle_logsumexp(z, V);
            double zt_pol = z[tok];
            row_logits(h_ref, W_ref, type, t, d, V, z, hrow);
            double lse_ref = oracle_logsumexp(z, V);
            double zt_ref = z[tok];
            double q = zt_pol - lse_pol;
            double p = zt_ref - lse_ref;
            double pen, ell, g;
            objective_terms(objective, A, q, p, beta, &pen, &ell, &g);
            double* o = out + (size_t)i * 9;
            o[0] = lse_pol; o[1] = lse_ref; o[2] = zt_pol; o[3] = zt_ref;
            o[4] = q; o[5] = p; o[6] = pen; o[7] = ell; o[8] = g;
        }
        free(hrow);
        free(z);
    }
}

/* ---- the mean over completion tokens -------------------------------------- */

/* Per-row weight of the loss for the listed (masked-in, ascending) rows:
 *   loss_mode 0: 1 / N_v                       (mean over all completion tokens)
 *   loss_mode 1: 1 / (n_active * len_i)        (mean over completions of the
 *                token mean of each; len_i = masked-in rows of completion i,
 *                n_active = completions with len_i > 0) */
void oracle_row_weights(const int32_t* rows, int64_t n_rows, int L, int loss_mode, double* w) {
    if (loss_mode == 1) {
        int64_t i = 0, n_active = 0;
        while (i < n_rows) {                      /* rows are ascending: completions are contiguous runs */
            int64_t seq = rows[i] / L, j = i;
            while (j < n_rows && rows[j] / L == seq) ++j;
            ++n_active;
            i = j;
        }
        i = 0;
        while (i < n_rows) {
            int64_t seq = rows[i] / L, j = i;
            while (j < n_rows && rows[j] / L == seq) ++j;
            for (int64_t k = i; k < j; ++k) w[k] = 1.0 / ((double)n_active * (double)(j - i));
            i = j;
        }
    } else {
        for (int64_t i = 0; i < n_rows; ++i) w[i] = 1.0 / (double)n_rows;
    }
}

/* The same weights for one shard of a batch split by whole completions over
 * several devices: the divisors count the whole batch, so that the shards'
 * weighted sums add up to the batch's mean.
 *   loss_mode 0: 1 / n_valid_batch
 *   loss_mode 1: 1 / (n_active_batch * len_i), len_i counted in this shard's
 *                rows (a completion lies wholly in one shard) */
void oracle_row_weights_shard(const int32_t* rows, int64_t n_rows, int L, int loss_mode, int64_t n_valid_batch,
                              int64_t n_active_batch, double* w) {
    if (loss_mode == 1) {
        int64_t i = 0;
        while (i < n_rows) {
            int64_t seq = rows[i] / L, j = i;
            while (j < n_rows && rows[j] / L == seq) ++j;
            for (int64_t k = i; k < j; ++k) w[k] = 1.0 / ((double)n_active_batch * (double)(j - i));
            i = j;
        }
    } else {
        for (int64_t i = 0; i < n_rows; ++i) w[i] = 1.0 / (double)n_valid_batch;
    }
}

/* sum_i w_i * ell_i in ascending order: one shard's share of the batch loss */
double oracle_weighted_sum(const double* ell, const double* w, int64_t n) {
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) s = s + w[i] * ell[i];
    return s;
}

/* The loss from per-row objectives of all masked-in rows (ascending):
 * token mean, or the mean over completions of each completion's token mean. */
double oracle_reduce_loss(const double* ell, const int32_t* rows, int64_t n_rows, int L, int loss_mode) {
    if (n_rows == 0) return 0.0;
    if (loss_mode != 1) {
        double s = 0.0;
        for (int64_t i = 0; i < n_rows; ++i) s = s + ell[i];
        return s / (double)n_rows;
    }
    double total = 0.0;
    int64_t n_active = 0, i = 0;
    while (i < n_rows) {
        int64_t seq = rows[i] / L, j = i;
        double s = 0.0;
        while (j < n_rows && rows[j] / L == seq) s = s + ell[j++];
        total = total + s / (double)(j - i);
        ++n_active;
        i = j;
    }
    return total / (double)n_active;
}

/* loss over the masked rows for an objective and a mean; also returns N_v */
double oracle_loss(const void* h_pol, const void* h_ref, const void* W, int type,
                   const int32_t* tokens, const uint8_t* mask, const float* adv,
                   int64_t N, int L, int d, int V, double beta, int objective, int loss_mode,
                   int64_t* n_valid_out) {
    int32_t* rows = (int32_t*)malloc(sizeof(int32_t) * (size_t)(N > 0 ? N : 1));
    int64_t nv = oracle_valid_rows(mask, N, rows);
    double* terms = (double*)malloc(sizeof(double) * 9 * (size_t)(nv > 0 ? nv : 1));
    double* ell = (double*)malloc(sizeof(double) * (size_t)(nv > 0 ? nv : 1));
    oracle_row_terms(h_pol, h_ref, W, NULL, type, tokens, adv, L, d, V, beta, objective, rows, nv, terms);
    for (int64_t i = 0; i < nv; ++i) ell[i] = terms[(size_t)i * 9 + 7];
    double loss = oracle_reduce_loss(ell, rows, nv, L, loss_mode);
    free(ell);
    free(terms);
    free(rows);
    if (n_valid_out) *n_valid_out = nv;
    return loss;
}

/* Surrogate objective whose gradient is the gradient of the chosen objective:
 *   J = sum_i w_i [ -A exp(q_i - c_i) + beta pen_i ]
 * With c held at q's value this is the detached objective; passing
 * c == NULL re-evaluates c = q inside, i.e. the variant without the detach. */
double oracle_surrogate(const void* h_pol, const void* h_ref, const void* W, const void* W_ref,
                        int type, const int32_t* tokens, const float* adv, int L, int d, int V,
                        double beta, int objective, const int32_t* rows, int64_t n_rows, const double* c,
                        const double* w) {
    double* terms = (double*)malloc(sizeof(double) * 9 * (size_t)(n_rows > 0 ? n_rows : 1));
    oracle_row_terms(h_pol, h_ref, W, W_ref, type, tokens, adv, L, d, V, beta, objective, rows, n_rows, terms);
    double s = 0.0;
    for (int64_t i = 0; i < n_rows; ++i) {
        const double* o = terms + (size_t)i * 9;
        double A = (double)adv[rows[i] / L];
        double ci = c ? c[i] : o[4];
        s = s + w[i] * (-A * exp(o[4] - ci) + beta * o[6]);
    }
    free(terms);
    return s;
}

/* ---- backward ------------------------------------------------------------ */

/* dS[t,v] = w_t * g_t * (1[v == tok_t] - exp(z_tv - lse_t)) for the policy logits.
 *   dH[i,:] = sum_v dS[rows[i], v] * W[v,:]                 (if dH != NULL)
 *   dW[j,:] = sum_i dS[rows[i], vrows[j]] * h_pol[rows[i],:] (if dW != NULL;
 *             vrows == NULL means all V vocabulary rows in order)
 * lse, g and the loss weights w are per listed row. */
void oracle_grad(const void* h_pol, const void* W, int type, const int32_t* tokens,
                 int d, int V, const int32_t* rows, int64_t n_rows,
                 const double* lse, const double* g, const double* w,
                 double* dH, const int32_t* vrows, int64_t n_vrows, double* dW) {
    if (dH) {
#pragma omp parallel
        {
            double* z = (double*)malloc(sizeof(double) * (size_t)V);
            double* hrow = (double*)malloc(sizeof(double) * (size_t)d);
            double* wrow = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < n_rows; ++i) {
                int64_t t = rows[i];
                int tok = tokens[t];
                double* out = dH + (size_t)i * d;
                row_logits(h_pol, W, type, t, d, V, z, hrow);
                for (int k = 0; k < d; ++k) out[k] = 0.0;
                for (int v = 0; v < V; ++v) {
                    double dS = w[i] * g[i] * ((v == tok ? 1.0 : 0.0) - exp(z[v] - lse[i]));
                    load_row(W, type, v, d, wrow);
                    for (int k = 0; k < d; ++k) out[k] = out[k] + dS * wrow[k];
                }
            }
            free(wrow);
            free(hrow);
            free(z);
        }
    }
    if (dW) {
        int64_t nv = vrows ? n_vrows : V;
#pragma omp parallel
        {
            double* hrow = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 4)
            for (int64_t j = 0; j < nv; ++j) {
                int v = vrows ? vrows[j] : (int)j;
                double* out = dW + (size_t)j * d;
                for (int k = 0; k < d; ++k) out[k] = 0.0;
                for (int64_t i = 0; i < n_rows; ++i) {
                    int64_t t = rows[i];
                    load_row(h_pol, type, t, d, hrow);
                    double z = dot_w(hrow, W, type, v, d);
                    double dS = w[i] * g[i] * ((v == tokens[t] ? 1.0 : 0.0) - exp(z - lse[i]));
                    for (int k = 0; k < d; ++k) out[k] = out[k] + dS * hrow[k];
                }
            }
            free(hrow);
        }
    }
}
