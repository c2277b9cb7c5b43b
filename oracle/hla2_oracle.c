/*
 * Float64 serial recurrence for masked second-order Higher-order Linear Attention.
 *
 * TEST INFRASTRUCTURE ONLY: the independent CPU oracle that the CUDA library is
 * checked against, and the timed CPU baseline.  It shares no code with the CUDA
 * library.  Only the tests, the smoke check and the benchmark's CPU legs load it.
 *
 * What it computes, per head, token by token (page "Higher-order Linear Attention",
 * technical summary, item "1. Zweite Ordnung HLA"; section summary §3.1, §4.3):
 *   G_t = g^2 G_{t-1} + g k_t (k_t^T C_{t-1})      (cross summary, pre-update C)
 *   h_t = g^2 h_{t-1} + g k_t (k_t^T m_{t-1})      (cross summary, pre-update m)
 *   S_t = g S_{t-1} + k_t k_t^T                     (key second moment)
 *   C_t = g C_{t-1} + q_t v_t^T                     (query-value accumulator)
 *   m_t = g m_{t-1} + q_t                           (query mass)
 *   o_t = q_t^T (S_t C_t - G_t)  = (q_t^T S_t) C_t - q_t^T G_t
 *   den_t = q_t^T (S_t m_t - h_t);  normalised output o_t / (den_t + eps)
 * With masked = 0 the output is the unmasked product q_t^T S_t C_t (and the denominator
 * q_t^T S_t m_t): the "numerator-style bilinear form" of section summary §3, whose scan
 * is the unmasked monoid of §4.1.  The state evolves the same way in both cases.
 * The gradient routine is the reverse sweep of exactly this recurrence (section
 * summary §4.2: the reverse-mode scan must reproduce these gradients), with states
 * recomputed from checkpoints every `ck` tokens.
 *
 * Inputs are float32 arrays (bf16-rounded values are exact in float32); all
 * arithmetic and all outputs are float64.  Heads are independent and are spread
 * over OpenMP threads.  Packed state per head: [S d*d | C d*dv | G d*dv | m d | h d].
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int hla2_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

typedef struct {
    int d, dv;
    double *S, *C, *G, *m, *h; /* views into one buffer */
    double *kC, *u;            /* scratch */
} head_state;

static long state_floats(int d, int dv) { return (long)d * d + 2L * d * dv + 2L * d; }

static int hs_init(head_state* st, int d, int dv) {
    st->d = d;
    st->dv = dv;
    double* buf = (double*)calloc((size_t)(state_floats(d, dv) + dv + d), sizeof(double));
    if (!buf) return -1;
    st->S = buf;
    st->C = st->S + (long)d * d;
    st->G = st->C + (long)d * dv;
    st->m = st->G + (long)d * dv;
    st->h = st->m + d;
    st->kC = st->h + d;
    st->u = st->kC + dv;
    return 0;
}

static void hs_free(head_state* st) { free(st->S); }

/* One online update then the output (see file header). */
static void hs_step(head_state* st, const float* q, const float* k, const float* v,
                    double g, int normalize, double eps, int masked, double* o) {
    const int d = st->d, dv = st->dv;
    double *S = st->S, *C = st->C, *G = st->G, *m = st->m, *h = st->h;
    double *kC = st->kC, *u = st->u;
    /* k^T C_{t-1}, k^T m_{t-1} */
    for (int e = 0; e < dv; ++e) kC[e] = 0.0;
    double km = 0.0;
    for (int a = 0; a < d; ++a) {
        const double ka = k[a];
        const double* Ca = C + (long)a * dv;
        for (int e = 0; e < dv; ++e) kC[e] += ka * Ca[e];
        km += ka * m[a];
    }
    const double g2 = g * g;
    for (int a = 0; a < d; ++a) {
        const double ka = k[a], qa = q[a];
        double* Ga = G + (long)a * dv;
        double* Ca = C + (long)a * dv;
        double* Sa = S + (long)a * d;
        for (int e = 0; e < dv; ++e) Ga[e] = g2 * Ga[e] + g * ka * kC[e];
        h[a] = g2 * h[a] + g * ka * km;
        for (int c = 0; c < d; ++c) Sa[c] = g * Sa[c] + ka * (double)k[c];
        for (int e = 0; e < dv; ++e) Ca[e] = g * Ca[e] + qa * (double)v[e];
        m[a] = g * m[a] + qa;
    }
    /* u = q^T S_t */
    for (int c = 0; c < d; ++c) u[c] = 0.0;
    for (int a = 0; a < d; ++a) {
        const double qa = q[a];
        const double* Sa = S + (long)a * d;
        for (int c = 0; c < d; ++c) u[c] += qa * Sa[c];
    }
    /* o = u C_t - q^T G_t (unmasked: u C_t) */
    const double mk = masked ? 1.0 : 0.0;
    for (int e = 0; e < dv; ++e) o[e] = 0.0;
    for (int a = 0; a < d; ++a) {
        const double ua = u[a], qa = mk * q[a];
        const double* Ca = C + (long)a * dv;
        const double* Ga = G + (long)a * dv;
        for (int e = 0; e < dv; ++e) o[e] += ua * Ca[e] - qa * Ga[e];
    }
    if (normalize) {
        double den = 0.0;
        for (int a = 0; a < d; ++a) den += u[a] * m[a] - mk * (double)q[a] * h[a];
        const double inv = 1.0 / (den + eps);
        for (int e = 0; e < dv; ++e) o[e] *= inv;
    }
}

static double head_gamma(const double* gamma, long bh, long H) {
    return gamma ? gamma[bh % H] : 1.0;
}

int hla2_oracle_forward(const float* q, const float* k, const float* v, double* out,
                        long BH, long H, long n, int d, int dv, const double* gamma,
                        int normalize, double eps, const double* init_state,
                        double* final_state, int masked) {
    if (BH < 0 || n < 0 || d <= 0 || dv <= 0 || H <= 0) return -1;
    const long sf = state_floats(d, dv);
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < BH; ++bh) {
        head_state st;
        if (hs_init(&st, d, dv)) {
#pragma omp atomic write
            err = -2;
            continue;
        }
        if (init_state) memcpy(st.S, init_state + bh * sf, (size_t)sf * sizeof(double));
        const double g = head_gamma(gamma, bh, H);
        for (long t = 0; t < n; ++t) {
            const long row = bh * n + t;
            hs_step(&st, q + row * d, k + row * d, v + row * dv, g, normalize, eps, masked,
                    out + row * dv);
        }
        if (final_state) memcpy(final_state + bh * sf, st.S, (size_t)sf * sizeof(double));
        hs_free(&st);
    }
    return err;
}

/* One decode step for NH independent heads, state in place. */
int hla2_oracle_decode(double* state, const float* q, const float* k, const float* v,
                       double* out, long NH, long H, int d, int dv, const double* gamma,
                       int normalize, double eps, int masked) {
    if (NH < 0 || d <= 0 || dv <= 0 || H <= 0) return -1;
    const long sf = state_floats(d, dv);
    int err = 0;
#pragma omp parallel for schedule(static)
    for (long nh = 0; nh < NH; ++nh) {
        head_state st;
        if (hs_init(&st, d, dv)) {
#pragma omp atomic write
            err = -2;
            continue;
        }
        memcpy(st.S, state + nh * sf, (size_t)sf * sizeof(double));
        hs_step(&st, q + nh * d, k + nh * d, v + nh * dv, head_gamma(gamma, nh, H),
                normalize, eps, masked, out + nh * dv);
        memcpy(state + nh * sf, st.S, (size_t)sf * sizeof(double));
        hs_free(&st);
    }
    return err;
}

/* S, C, G after one token (G first: it reads the pre-update C). */
static void advance_SCG(double* S, double* C, double* G, double* kC, const float* qt,
                        const float* kt, const float* vt, int d, int dv, double g) {
    const double g2 = g * g;
    for (int e = 0; e < dv; ++e) kC[e] = 0.0;
    for (int a = 0; a < d; ++a)
        for (int e = 0; e < dv; ++e) kC[e] += (double)kt[a] * C[(long)a * dv + e];
    for (int a = 0; a < d; ++a) {
        for (int e = 0; e < dv; ++e)
            G[(long)a * dv + e] = g2 * G[(long)a * dv + e] + g * kt[a] * kC[e];
        for (int c = 0; c < d; ++c)
            S[(long)a * d + c] = g * S[(long)a * d + c] + (double)kt[a] * kt[c];
        for (int e = 0; e < dv; ++e)
            C[(long)a * dv + e] = g * C[(long)a * dv + e] + (double)qt[a] * vt[e];
    }
}

/*
 * Reverse sweep of the unnormalised recurrence.  With state adjoints (Sb, Cb, Gb)
 * arriving from token t+1, at token t:
 *   u = S_t^T q;  Cb += u dO^T;  ub = C_t dO;  Sb += q ub^T;  Gb -= q dO^T;
 *   dq += S_t ub - G_t dO;
 *   r = C_{t-1}^T k;  rb = g Gb^T k;  dk += g Gb r + C_{t-1} rb + (Sb + Sb^T) k;
 *   dq += Cb v;  dv += Cb^T q;
 *   Cb <- g Cb + k rb^T;  Sb <- g Sb;  Gb <- g^2 Gb.
 */
int hla2_oracle_backward(const float* q, const float* k, const float* v, const float* dout,
                         double* dq, double* dk, double* dvv, long BH, long H, long n, int d,
                         int dv, const double* gamma) {
    if (BH < 0 || n < 0 || d <= 0 || dv <= 0 || H <= 0) return -1;
    long ck = (long)ceil(sqrt((double)(n > 0 ? n : 1)));
    if (ck < 1) ck = 1;
    const long nblk = (n + ck - 1) / ck;
    const long dd = (long)d * d, ddv = (long)d * dv;
    const long ckpt_floats = dd + 2 * ddv; /* S, C, G before the block's first token */
    const long rec_floats = dd + 3 * ddv;  /* S_t, C_t, G_t, C_{t-1} */
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < BH; ++bh) {
        const double g = head_gamma(gamma, bh, H);
        const double g2 = g * g;
        double* ckpt = (double*)calloc((size_t)(nblk * ckpt_floats + 1), sizeof(double));
        double* blk = (double*)malloc((size_t)(ck * rec_floats + 1) * sizeof(double));
        double* adj = (double*)calloc((size_t)(dd + 2 * ddv + 2L * (d + dv)), sizeof(double));
        double* S = (double*)calloc((size_t)(dd + 2 * ddv + dv), sizeof(double));
        if (!ckpt || !blk || !adj || !S) {
            free(ckpt);
            free(blk);
            free(adj);
            free(S);
#pragma omp atomic write
            err = -2;
            continue;
        }
        memset(dq + bh * n * d, 0, (size_t)(n * d) * sizeof(double));
        memset(dk + bh * n * d, 0, (size_t)(n * d) * sizeof(double));
        memset(dvv + bh * n * dv, 0, (size_t)(n * dv) * sizeof(double));
        double *Sb = adj, *Cb = Sb + dd, *Gb = Cb + ddv;
        double *u = Gb + ddv, *ub = u + d, *r = ub + d, *rb = r + dv;
        double* C = S + dd;
        double* G = C + ddv;
        double* kC = G + ddv;
        /* forward sweep, saving (S, C, G) at each block start */
        for (long t = 0; t < n; ++t) {
            if (t % ck == 0)
                memcpy(ckpt + (t / ck) * ckpt_floats, S, (size_t)ckpt_floats * sizeof(double));
            const long row = bh * n + t;
            advance_SCG(S, C, G, kC, q + row * d, k + row * d, v + row * dv, d, dv, g);
        }
        /* reverse sweep over blocks, recomputing each block's states */
        for (long bi = nblk - 1; bi >= 0; --bi) {
            const long t0 = bi * ck;
            const long t1 = (t0 + ck < n) ? t0 + ck : n;
            memcpy(S, ckpt + bi * ckpt_floats, (size_t)ckpt_floats * sizeof(double));
            for (long t = t0; t < t1; ++t) {
                double* rec = blk + (t - t0) * rec_floats;
                const long row = bh * n + t;
                memcpy(rec + dd + 2 * ddv, C, (size_t)ddv * sizeof(double));
                advance_SCG(S, C, G, kC, q + row * d, k + row * d, v + row * dv, d, dv, g);
                memcpy(rec, S, (size_t)dd * sizeof(double));
                memcpy(rec + dd, C, (size_t)ddv * sizeof(double));
                memcpy(rec + dd + ddv, G, (size_t)ddv * sizeof(double));
            }
            for (long t = t1 - 1; t >= t0; --t) {
                const double* rec = blk + (t - t0) * rec_floats;
                const double *St = rec, *Ct = rec + dd, *Gt = rec + dd + ddv, *Cp = rec + dd + 2 * ddv;
                const long row = bh * n + t;
                const float *qt = q + row * d, *kt = k + row * d, *vt = v + row * dv;
                const float* dO = dout + row * dv;
                double *dqt = dq + row * d, *dkt = dk + row * d, *dvt = dvv + row * dv;
                for (int c = 0; c < d; ++c) u[c] = 0.0;
                for (int a = 0; a < d; ++a)
                    for (int c = 0; c < d; ++c) u[c] += St[(long)a * d + c] * qt[a];
                for (int a = 0; a < d; ++a) {
                    double acc = 0.0;
                    for (int e = 0; e < dv; ++e) acc += Ct[(long)a * dv + e] * dO[e];
                    ub[a] = acc;
                }
                for (int a = 0; a < d; ++a) {
                    for (int e = 0; e < dv; ++e) {
                        Cb[(long)a * dv + e] += u[a] * dO[e];
                        Gb[(long)a * dv + e] -= (double)qt[a] * dO[e];
                    }
                    for (int c = 0; c < d; ++c) Sb[(long)a * d + c] += (double)qt[a] * ub[c];
                }
                for (int a = 0; a < d; ++a) {
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c) acc += St[(long)a * d + c] * ub[c];
                    for (int e = 0; e < dv; ++e) acc -= Gt[(long)a * dv + e] * dO[e];
                    dqt[a] += acc;
                }
                for (int e = 0; e < dv; ++e) {
                    r[e] = 0.0;
                    rb[e] = 0.0;
                }
                for (int a = 0; a < d; ++a)
                    for (int e = 0; e < dv; ++e) {
                        r[e] += Cp[(long)a * dv + e] * kt[a];
                        rb[e] += Gb[(long)a * dv + e] * kt[a];
                    }
                for (int e = 0; e < dv; ++e) rb[e] *= g;
                for (int a = 0; a < d; ++a) {
                    double acc = 0.0;
                    for (int e = 0; e < dv; ++e)
                        acc += g * Gb[(long)a * dv + e] * r[e] + Cp[(long)a * dv + e] * rb[e];
                    for (int c = 0; c < d; ++c)
                        acc += (Sb[(long)a * d + c] + Sb[(long)c * d + a]) * kt[c];
                    dkt[a] += acc;
                }
                for (int a = 0; a < d; ++a) {
                    double acc = 0.0;
                    for (int e = 0; e < dv; ++e) acc += Cb[(long)a * dv + e] * vt[e];
                    dqt[a] += acc;
                }
                for (int e = 0; e < dv; ++e) {
                    double acc = 0.0;
                    for (int a = 0; a < d; ++a) acc += Cb[(long)a * dv + e] * qt[a];
                    dvt[e] += acc;
                }
                for (int a = 0; a < d; ++a) {
                    for (int e = 0; e < dv; ++e) {
                        Cb[(long)a * dv + e] = g * Cb[(long)a * dv + e] + (double)kt[a] * rb[e];
                        Gb[(long)a * dv + e] *= g2;
                    }
                    for (int c = 0; c < d; ++c) Sb[(long)a * d + c] *= g;
                }
            }
        }
        free(S);
        free(ckpt);
        free(blk);
        free(adj);
    }
    return err;
}
