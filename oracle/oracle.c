/*
 * oracle.c -- plain, slow, fp64 CPU decoder: the reference the CUDA path is
 * checked against.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load or call this library.  It shares no
 * code with the CUDA path; its inputs come from the seeded generator (gen/).
 *
 * What it computes.  The pages ("Execution", section "A constant-shape decode
 * graph") define the captured step as an exact re-organisation of an ordinary
 * causal decode step: K and V are written at `pos`, attention sweeps a fixed
 * capacity and a mask hides every position after `pos`.  Masked positions
 * contribute nothing, so the plain definition -- attention over positions
 * [0, pos] only, no capacity sweep, no splitting -- is the oracle.  The layer
 * structure is the pages' residual pair ("Models, Registry and the Driver",
 * section "Shared components", standard_stack / standard_layer):
 *     x = embed(token)
 *     per layer:  x += mixer(norm(x));  x += ffn(norm(x))
 *     logits = head(final_norm(x))
 * with mixer = QKV projection, RoPE, K/V write at pos, causal attention, output
 * projection, and ffn = SwiGLU ("Architecture Overview", section "Automatic
 * fusion": attention, RMSNorm, RoPE and SwiGLU as compositions).
 *
 * The pages give no formulas for the pieces; the plain Llama-style readings are
 * used (RMSNorm x / sqrt(mean(x^2) + eps) * g, half-split RoPE with
 * w_i = theta^(-2i/hd), scale 1/sqrt(hd), GQA head i -> kv head i / G,
 * silu(z) = z / (1 + e^-z)).  Stored K/V get the storage rounding of the KV
 * dtype (bf16 round-to-nearest-even, or none for fp32), because the step's
 * carried state is what is stored ("Execution", section "Verification",
 * tier 2: every output and carried state is compared).
 *
 * All arithmetic is IEEE fp64; weights are read exactly (bf16 or fp32 widen
 * exactly).  OpenMP is used only across independent output rows / heads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* element types of an array the oracle reads */
enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2 };

typedef struct orc_model {
    int n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_hidden, vocab;
    double rms_eps, rope_theta;
    int wdtype;   /* ORC_F32 or ORC_BF16: element type of every weight */
    int kvdtype;  /* ORC_F32 or ORC_BF16: storage type of K and V */
    const void *embed, *final_norm, *lm_head;
    /* n_layers * 9 pointers: attn_norm, wq, wk, wv, wo, ffn_norm, wg, wu, wd,
       each in nn.Linear layout [out, in], row-major */
    const void *const *layer;
} orc_model;

enum { L_ATTN_NORM = 0, L_WQ, L_WK, L_WV, L_WO, L_FFN_NORM, L_WG, L_WU, L_WD, L_NROLES };

/* ---------- exact element access and storage rounding ---------- */

double orc_bf16_value(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* fp64 -> bf16, one rounding to nearest, ties to even, from the IEEE-754
   binary64 encoding (8 significant bits kept, exponent range of binary32).
   NaN stays NaN; overflow goes to infinity. */
uint16_t orc_bf16_round(double v) {
    uint64_t u;
    memcpy(&u, &v, sizeof u);
    uint16_t sign = (uint16_t)((u >> 48) & 0x8000u);
    if (v != v) return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    int e;
    frexp(a, &e);                      /* a in [2^(e-1), 2^e) */
    int top = e - 1;
    /* spacing of bf16 numbers near a: 7 fraction bits, binary32 exponent range */
    int ulp_exp = (top < -126 ? -126 : top) - 7;
    double scaled = ldexp(a, -ulp_exp);                 /* exact power-of-two scaling */
    double fl = floor(scaled);
    double frac = scaled - fl;
    double r = fl;
    if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0)) r = fl + 1.0;
    double rounded = ldexp(r, ulp_exp);
    if (rounded > 3.3895313892515355e38)   /* above the largest finite bf16 */
        return (uint16_t)(sign | 0x7F80u);
    float f = (float)rounded;          /* exact: at most 8 significant bits */
    uint32_t fu;
    memcpy(&fu, &f, sizeof fu);
    return (uint16_t)(sign | ((fu >> 16) & 0x7FFFu));
}

static inline double rd(const void *p, int dt, int64_t i) {
    if (dt == ORC_BF16) return orc_bf16_value(((const uint16_t *)p)[i]);
    if (dt == ORC_F32) return (double)((const float *)p)[i];
    return ((const double *)p)[i];
}

static inline void wr_store(void *p, int dt, int64_t i, double v) {
    if (dt == ORC_BF16) ((uint16_t *)p)[i] = orc_bf16_round(v);
    else if (dt == ORC_F32) ((float *)p)[i] = (float)v;
    else ((double *)p)[i] = v;
}

/* ---------- the pieces ---------- */

/* RMSNorm: out_i = x_i / sqrt(mean(x^2) + eps) * g_i  (gain g, eps inside the root) */
void orc_rmsnorm(const double *x, int n, const void *g, int gdt, double eps, double *out) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss / (double)n + eps);
    for (int i = 0; i < n; ++i) out[i] = x[i] * inv * rd(g, gdt, i);
}

/* out[r] = sum_c W[r, c] * h[c]; W row-major [rows, cols] */
void orc_matvec(const void *W, int wdt, int rows, int cols, const double *h, double *out) {
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        double acc = 0.0;
        int64_t base = (int64_t)r * cols;
        for (int c = 0; c < cols; ++c) acc += rd(W, wdt, base + c) * h[c];
        out[r] = acc;
    }
}

/* Rotary embedding, half-split pairing: pair (i, i + hd/2), i in [0, hd/2),
   angle = pos * theta^(-2i/hd); (a, b) -> (a cos - b sin, a sin + b cos). */
void orc_rope(double *v, int hd, int pos, double theta) {
    int half = hd / 2;
    for (int i = 0; i < half; ++i) {
        double w = pow(theta, -2.0 * (double)i / (double)hd);
        double ang = (double)pos * w;
        double c = cos(ang), s = sin(ang);
        double a = v[i], b = v[i + half];
        v[i] = a * c - b * s;
        v[i + half] = a * s + b * c;
    }
}

double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/* softmax(s)_j = exp(s_j - max s) / sum_k exp(s_k - max s) */
void orc_softmax(const double *s, int n, double *a) {
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) if (s[j] > m) m = s[j];
    double z = 0.0;
    for (int j = 0; j < n; ++j) { a[j] = exp(s[j] - m); z += a[j]; }
    for (int j = 0; j < n; ++j) a[j] /= z;
}

/* One head of causal attention over the visible positions j in [0, npos):
   s_j = q . k_j / sqrt(hd), a = softmax(s), o = sum_j a_j v_j.
   k_j = K[j * stride .. + hd), v_j likewise; K and V in element type kvdt. */
void orc_attend(const double *q, const void *K, const void *V, int kvdt, int64_t stride,
                int npos, int hd, double *o) {
    double *s = (double *)malloc(sizeof(double) * (size_t)(npos > 0 ? npos : 1));
    double *a = (double *)malloc(sizeof(double) * (size_t)(npos > 0 ? npos : 1));
    double scale = 1.0 / sqrt((double)hd);
    for (int j = 0; j < npos; ++j) {
        double acc = 0.0;
        for (int d = 0; d < hd; ++d) acc += q[d] * rd(K, kvdt, (int64_t)j * stride + d);
        s[j] = acc * scale;
    }
    orc_softmax(s, npos, a);
    for (int d = 0; d < hd; ++d) o[d] = 0.0;
    for (int j = 0; j < npos; ++j)
        for (int d = 0; d < hd; ++d) o[d] += a[j] * rd(V, kvdt, (int64_t)j * stride + d);
    free(s);
    free(a);
}

/* threads of the parallel loops over output rows and heads (timing only: the
   results do not depend on it) */
extern void omp_set_num_threads(int);   /* OpenMP runtime API (linked with -fopenmp) */
extern int omp_get_max_threads(void);
void orc_set_threads(int n) { omp_set_num_threads(n > 0 ? n : 1); }
int orc_threads(void) { return omp_get_max_threads(); }

/* index of the largest value, lowest index on ties */
int orc_argmax(const double *v, int n) {
    int best = 0;
    for (int i = 1; i < n; ++i) if (v[i] > v[best]) best = i;
    return best;
}

static int check_model(const orc_model *m) {
    if (!m || m->n_layers <= 0 || m->d_model <= 0 || m->n_heads <= 0 || m->n_kv_heads <= 0 ||
        m->head_dim <= 0 || (m->head_dim & 1) || m->n_heads % m->n_kv_heads || m->vocab <= 0 ||
        m->ffn_hidden <= 0)
        return -1;
    return 0;
}

/* The feed-forward half of a layer: x += Wd (silu(Wg h) * (Wu h)), h = rmsnorm(x) g_ffn */
static void ffn_half(const orc_model *m, const void *const *w, double *x, double *h,
                     double *gt, double *up) {
    int d = m->d_model, F = m->ffn_hidden, wdt = m->wdtype;
    orc_rmsnorm(x, d, w[L_FFN_NORM], wdt, m->rms_eps, h);
    orc_matvec(w[L_WG], wdt, F, d, h, gt);
    orc_matvec(w[L_WU], wdt, F, d, h, up);
    for (int i = 0; i < F; ++i) gt[i] = orc_silu(gt[i]) * up[i];
    double *dx = (double *)malloc(sizeof(double) * (size_t)d);
    orc_matvec(w[L_WD], wdt, d, F, gt, dx);
    for (int i = 0; i < d; ++i) x[i] += dx[i];
    free(dx);
}

/* One decode step of one sequence ("Execution", sections "A constant-shape
   decode graph" and "Slot buffers"; "Models, Registry and the Driver",
   section "The Model": decode is a step of one token at an absolute position).
   K[l], V[l]: this sequence's stored keys/values of layer l, logical layout
   [cap, n_kv_heads, head_dim] in kvdtype; the step writes position `pos` and
   reads positions [0, pos].  logits: [vocab] fp64 out.  hidden_out (optional):
   the final residual x [d_model]. */
int orc_step(const orc_model *m, void *const *K, void *const *V, int cap, int token, int pos,
             double *logits, double *hidden_out) {
    if (check_model(m) || token < 0 || token >= m->vocab || pos < 0 || pos >= cap) return -1;
    int d = m->d_model, hd = m->head_dim, Hq = m->n_heads, Hkv = m->n_kv_heads;
    int G = Hq / Hkv, qd = Hq * hd, kvd = Hkv * hd, F = m->ffn_hidden, wdt = m->wdtype;
    double *x = (double *)malloc(sizeof(double) * (size_t)d);
    double *h = (double *)malloc(sizeof(double) * (size_t)d);
    double *q = (double *)malloc(sizeof(double) * (size_t)qd);
    double *k = (double *)malloc(sizeof(double) * (size_t)kvd);
    double *v = (double *)malloc(sizeof(double) * (size_t)kvd);
    double *o = (double *)malloc(sizeof(double) * (size_t)qd);
    double *dx = (double *)malloc(sizeof(double) * (size_t)d);
    double *gt = (double *)malloc(sizeof(double) * (size_t)F);
    double *up = (double *)malloc(sizeof(double) * (size_t)F);

    for (int i = 0; i < d; ++i) x[i] = rd(m->embed, wdt, (int64_t)token * d + i);
    for (int l = 0; l < m->n_layers; ++l) {
        const void *const *w = m->layer + (size_t)l * L_NROLES;
        /* mixer: norm, QKV, RoPE at pos, K/V write at pos, attention over [0, pos] */
        orc_rmsnorm(x, d, w[L_ATTN_NORM], wdt, m->rms_eps, h);
        orc_matvec(w[L_WQ], wdt, qd, d, h, q);
        orc_matvec(w[L_WK], wdt, kvd, d, h, k);
        orc_matvec(w[L_WV], wdt, kvd, d, h, v);
        for (int i = 0; i < Hq; ++i) orc_rope(q + (size_t)i * hd, hd, pos, m->rope_theta);
        for (int g = 0; g < Hkv; ++g) orc_rope(k + (size_t)g * hd, hd, pos, m->rope_theta);
        for (int c = 0; c < kvd; ++c) {
            wr_store(K[l], m->kvdtype, (int64_t)pos * kvd + c, k[c]);
            wr_store(V[l], m->kvdtype, (int64_t)pos * kvd + c, v[c]);
        }
#pragma omp parallel for schedule(static)
        for (int i = 0; i < Hq; ++i) {
            int g = i / G;
            const char *kb = (const char *)K[l], *vb = (const char *)V[l];
            size_t es = m->kvdtype == ORC_BF16 ? 2 : 4;
            orc_attend(q + (size_t)i * hd, kb + (size_t)g * hd * es, vb + (size_t)g * hd * es,
                       m->kvdtype, kvd, pos + 1, hd, o + (size_t)i * hd);
        }
        orc_matvec(w[L_WO], wdt, d, qd, o, dx);
        for (int i = 0; i < d; ++i) x[i] += dx[i];
        ffn_half(m, w, x, h, gt, up);
    }
    orc_rmsnorm(x, d, m->final_norm, wdt, m->rms_eps, h);
    orc_matvec(m->lm_head, wdt, m->vocab, d, h, logits);
    if (hidden_out) memcpy(hidden_out, x, sizeof(double) * (size_t)d);
    free(x); free(h); free(q); free(k); free(v); free(o); free(dx); free(gt); free(up);
    return 0;
}

/* Direct causal pass over a whole prompt, written independently of the
   per-step bookkeeping: every layer is evaluated for all n tokens at once,
   attention as a masked score matrix S[t, j] (j > t hidden) with a row-wise
   softmax.  K/V are rounded to the storage type exactly as a step stores them.
   Outputs the logits of every token [n, vocab] and the stored K/V of every
   position (Kout[l], Vout[l]: [n, n_kv_heads, head_dim] in kvdtype). */
int orc_full_causal(const orc_model *m, const int *tokens, int n, double *logits,
                    void *const *Kout, void *const *Vout) {
    if (check_model(m) || n <= 0) return -1;
    int d = m->d_model, hd = m->head_dim, Hq = m->n_heads, Hkv = m->n_kv_heads;
    int G = Hq / Hkv, qd = Hq * hd, kvd = Hkv * hd, F = m->ffn_hidden, wdt = m->wdtype;
    for (int t = 0; t < n; ++t) if (tokens[t] < 0 || tokens[t] >= m->vocab) return -1;
    double *X = (double *)malloc(sizeof(double) * (size_t)n * d);
    double *H = (double *)malloc(sizeof(double) * (size_t)n * d);
    double *Q = (double *)malloc(sizeof(double) * (size_t)n * qd);
    double *Kf = (double *)malloc(sizeof(double) * (size_t)n * kvd);
    double *Vf = (double *)malloc(sizeof(double) * (size_t)n * kvd);
    double *O = (double *)malloc(sizeof(double) * (size_t)n * qd);
    double *S = (double *)malloc(sizeof(double) * (size_t)n * n);
    double *dx = (double *)malloc(sizeof(double) * (size_t)d);
    double *gt = (double *)malloc(sizeof(double) * (size_t)F);
    double *up = (double *)malloc(sizeof(double) * (size_t)F);
    double scale = 1.0 / sqrt((double)hd);

    for (int t = 0; t < n; ++t)
        for (int i = 0; i < d; ++i) X[(size_t)t * d + i] = rd(m->embed, wdt, (int64_t)tokens[t] * d + i);
    for (int l = 0; l < m->n_layers; ++l) {
        const void *const *w = m->layer + (size_t)l * L_NROLES;
        for (int t = 0; t < n; ++t) {
            double *h = H + (size_t)t * d;
            orc_rmsnorm(X + (size_t)t * d, d, w[L_ATTN_NORM], wdt, m->rms_eps, h);
            orc_matvec(w[L_WQ], wdt, qd, d, h, Q + (size_t)t * qd);
            orc_matvec(w[L_WK], wdt, kvd, d, h, Kf + (size_t)t * kvd);
            orc_matvec(w[L_WV], wdt, kvd, d, h, Vf + (size_t)t * kvd);
            for (int i = 0; i < Hq; ++i) orc_rope(Q + (size_t)t * qd + (size_t)i * hd, hd, t, m->rope_theta);
            for (int g = 0; g < Hkv; ++g) orc_rope(Kf + (size_t)t * kvd + (size_t)g * hd, hd, t, m->rope_theta);
            for (int c = 0; c < kvd; ++c) {   /* storage rounding, then read back */
                wr_store(Kout[l], m->kvdtype, (int64_t)t * kvd + c, Kf[(size_t)t * kvd + c]);
                wr_store(Vout[l], m->kvdtype, (int64_t)t * kvd + c, Vf[(size_t)t * kvd + c]);
                Kf[(size_t)t * kvd + c] = rd(Kout[l], m->kvdtype, (int64_t)t * kvd + c);
                Vf[(size_t)t * kvd + c] = rd(Vout[l], m->kvdtype, (int64_t)t * kvd + c);
            }
        }
        for (int i = 0; i < Hq; ++i) {
            int g = i / G;
            for (int t = 0; t < n; ++t) {
                double mx = -INFINITY;
                for (int j = 0; j < n; ++j) {
                    double sv = -INFINITY;
                    if (j <= t) {
                        double acc = 0.0;
                        for (int dd = 0; dd < hd; ++dd)
                            acc += Q[(size_t)t * qd + (size_t)i * hd + dd] * Kf[(size_t)j * kvd + (size_t)g * hd + dd];
                        sv = acc * scale;
                    }
                    S[(size_t)t * n + j] = sv;
                    if (sv > mx) mx = sv;
                }
                double z = 0.0;
                for (int j = 0; j < n; ++j) {
                    double e = (j <= t) ? exp(S[(size_t)t * n + j] - mx) : 0.0;
                    S[(size_t)t * n + j] = e;
                    z += e;
                }
                double *o = O + (size_t)t * qd + (size_t)i * hd;
                for (int dd = 0; dd < hd; ++dd) {
                    double acc = 0.0;
                    for (int j = 0; j <= t; ++j) acc += (S[(size_t)t * n + j] / z) * Vf[(size_t)j * kvd + (size_t)g * hd + dd];
                    o[dd] = acc;
                }
            }
        }
        for (int t = 0; t < n; ++t) {
            double *x = X + (size_t)t * d;
            orc_matvec(w[L_WO], wdt, d, qd, O + (size_t)t * qd, dx);
            for (int i = 0; i < d; ++i) x[i] += dx[i];
            ffn_half(m, w, x, H + (size_t)t * d, gt, up);
        }
    }
    for (int t = 0; t < n; ++t) {
        orc_rmsnorm(X + (size_t)t * d, d, m->final_norm, wdt, m->rms_eps, H + (size_t)t * d);
        orc_matvec(m->lm_head, wdt, m->vocab, d, H + (size_t)t * d, logits + (size_t)t * m->vocab);
    }
    free(X); free(H); free(Q); free(Kf); free(Vf); free(O); free(S); free(dx); free(gt); free(up);
    return 0;
}
