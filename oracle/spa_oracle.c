/*
 * spa_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct fp64 CPU statement of projected-feature
 * softmax attention.  It exists so that tests, the smoke check and the CPU
 * baseline leg of the benchmark have something independent to compare the
 * CUDA library against.  Nothing in the product path may call it, and it
 * shares no code, header, table or constant with the CUDA sources.
 *
 * What it computes, per (batch b, head h):
 *   1. every input value is read exactly and widened to double;
 *   2. Qp = Q P_h and Kp = K P_h, with P_h in R^{d x m}
 *        ("Sparse Projection Attention: A Computationally Efficient Framework
 *         for Long Sequence Modeling", Sec. 3.1.2 and Algorithm 1 steps 2-3;
 *         "Projection-Decomposition Attention" page, Algorithm 2.1 step 1);
 *   3. s_ij = <Qp_i, Kp_j> / sqrt(m)
 *        (SPA Sec. 3.1.3 and Algorithm 1 step 4; PDA Algorithm 2.1 step 2);
 *   4. if causal, only keys j <= i take part (top-left aligned square mask;
 *      the pages do not define masking, this is the plain reading);
 *   5. row softmax: M_i = max_j s_ij, e_ij = exp(s_ij - M_i), l_i = sum_j e_ij
 *        (SPA Algorithm 1 step 5; PDA Algorithm 2.1 step 3, row-wise);
 *   6. O_i = (sum_j e_ij V_j) / l_i      (SPA Algorithm 1 step 6).
 *
 * The max subtraction in step 5 does not change the value of the softmax; it
 * only keeps exp() finite.  No tiling, no reordering, no fusion.
 *
 * Element types accepted for inputs: 0 = double, 1 = float, 2 = bfloat16
 * (raw 16-bit patterns).  Widening bf16 -> double is exact.
 *
 * Parity status: every entry point is pinned by the tests in
 * tests/test_oracle_pins.py (a library attention routine, closed forms,
 * brute-force cases, softmax/JL invariants stated on the pages; for the
 * gradients, central finite differences, automatic differentiation of a
 * plain restatement of the forward, and exact sum rules).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F64 = 0, ORC_F32 = 1, ORC_BF16 = 2 };

static double orc_load(const void *base, int dt, size_t idx)
{
    if (dt == ORC_F64) return ((const double *)base)[idx];
    if (dt == ORC_F32) return (double)((const float *)base)[idx];
    /* bfloat16: the upper 16 bits of an IEEE binary32 */
    uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Step 2 for one row: out[k] = sum_l x[row, l] * P_h[l, k]. */
static void orc_project_row(const void *x, int dt, size_t row_off, const void *P,
                            size_t p_off, int d, int m, double *out)
{
    for (int k = 0; k < m; ++k) {
        double acc = 0.0;
        for (int l = 0; l < d; ++l)
            acc += orc_load(x, dt, row_off + (size_t)l) *
                   orc_load(P, dt, p_off + (size_t)l * m + k);
        out[k] = acc;
    }
}

/*
 * Projection alone: xp[b][h][i][k] = sum_l x[b][h][i][l] * P[h][l][k].
 * x: [B][H][N][d], P: [H][d][m] (element type dt), xp: [B][H][N][m] double.
 */
int orc_project(const void *x, const void *P, int dt, double *xp,
                int B, int H, long N, int d, int m)
{
    if (!x || !P || !xp || B < 0 || H < 0 || N < 0 || d <= 0 || m <= 0) return 1;
    long BH = (long)B * H;
    #pragma omp parallel for schedule(static)
    for (long r = 0; r < BH * N; ++r) {
        long bh = r / N;
        int h = (int)(bh % H);
        orc_project_row(x, dt, (size_t)r * d, P, (size_t)h * d * m, d, m,
                        xp + (size_t)r * m);
    }
    return 0;
}

/*
 * Full forward for a chosen set of query rows (rows == NULL: all N rows).
 * q, k: [B][H][N][d]; v: [B][H][N][dv]; P: [H][d][m], all of element type dt.
 * out: [B][H][nrows][dv] double (nrows = N when rows == NULL).
 * lse (optional, may be NULL): [B][H][nrows], natural-log sum of exp(s_ij).
 */
int orc_attention(const void *q, const void *k, const void *v, const void *P, int dt,
                  double *out, double *lse, int B, int H, long N, int d, int m, int dv,
                  int causal, const long *rows, long nrows)
{
    if (!q || !k || !v || !P || !out || B < 0 || H < 0 || N < 0 || d <= 0 || m <= 0 ||
        dv <= 0)
        return 1;
    if (!rows) nrows = N;
    for (long t = 0; rows && t < nrows; ++t)
        if (rows[t] < 0 || rows[t] >= N) return 2;
    if (N == 0 || nrows == 0) return 0;

    double *kp = (double *)malloc(sizeof(double) * (size_t)N * m);
    if (!kp) return 3;
    const double inv_sqrt_m = 1.0 / sqrt((double)m);

    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            size_t bh = (size_t)b * H + h;
            size_t p_off = (size_t)h * d * m;
            /* step 2 for every key of this head */
            #pragma omp parallel for schedule(static)
            for (long j = 0; j < N; ++j)
                orc_project_row(k, dt, (bh * N + j) * d, P, p_off, d, m, kp + (size_t)j * m);

            #pragma omp parallel
            {
                double *qp = (double *)malloc(sizeof(double) * (size_t)m);
                double *s = (double *)malloc(sizeof(double) * (size_t)N);
                double *o = (double *)malloc(sizeof(double) * (size_t)dv);
                #pragma omp for schedule(dynamic, 4)
                for (long t = 0; t < nrows; ++t) {
                    long i = rows ? rows[t] : t;
                    orc_project_row(q, dt, (bh * N + i) * d, P, p_off, d, m, qp);
                    long nkeys = causal ? i + 1 : N;          /* step 4 */
                    double mx = -INFINITY;
                    for (long j = 0; j < nkeys; ++j) {         /* step 3 */
                        double acc = 0.0;
                        for (int c = 0; c < m; ++c) acc += qp[c] * kp[(size_t)j * m + c];
                        s[j] = acc * inv_sqrt_m;
                        if (s[j] > mx) mx = s[j];
                    }
                    double l = 0.0;                            /* step 5 */
                    for (long j = 0; j < nkeys; ++j) {
                        s[j] = exp(s[j] - mx);
                        l += s[j];
                    }
                    for (int c = 0; c < dv; ++c) o[c] = 0.0;   /* step 6 */
                    for (long j = 0; j < nkeys; ++j) {
                        size_t voff = (bh * N + j) * dv;
                        for (int c = 0; c < dv; ++c) o[c] += s[j] * orc_load(v, dt, voff + c);
                    }
                    double *dst = out + (bh * (size_t)nrows + t) * dv;
                    for (int c = 0; c < dv; ++c) dst[c] = o[c] / l;
                    if (lse) lse[bh * (size_t)nrows + t] = mx + log(l);
                }
                free(qp);
                free(s);
                free(o);
            }
        }
    }
    free(kp);
    return 0;
}

/*
 * Gradients of the forward above, for a given upstream gradient dO of the
 * output (same element type as the inputs), by the chain rule through each
 * step, per (batch b, head h):
 *   A_ij   = exp(s_ij - M_i) / l_i                 (the forward's softmax)
 *   O_i    = sum_j A_ij V_j
 *   dV_j   = sum_i A_ij dO_i                       (step 6, w.r.t. V)
 *   dA_ij  = <dO_i, V_j>                           (step 6, w.r.t. A)
 *   D_i    = sum_j A_ij dA_ij = <dO_i, O_i>
 *   dS_ij  = A_ij (dA_ij - D_i)                    (step 5: softmax Jacobian)
 *   dQp_i  = sum_j dS_ij Kp_j / sqrt(m)            (step 3)
 *   dKp_j  = sum_i dS_ij Qp_i / sqrt(m)
 *   dQ_i   = dQp_i P_h^T,  dK_j = dKp_j P_h^T      (step 2)
 *   dP_h  += sum_i Q_i^T dQp_i + sum_j K_j^T dKp_j  (step 2, w.r.t. P; P_h is
 *                                                    shared by every batch entry)
 * with the causal mask (j <= i) applied to every sum over j or i.
 * ("Sparse Projection Attention", Sec. 3.4.1 and Algorithm 2: the projection
 *  is trained through these gradients.)
 * Outputs (double): dq, dk [B][H][N][d]; dv_out [B][H][N][dv]; dP [H][d][m].
 */
int orc_attention_bwd(const void *q, const void *k, const void *v, const void *P,
                      const void *dO, int dt, double *dq, double *dk, double *dv_out,
                      double *dP, int B, int H, long N, int d, int m, int dv, int causal)
{
    if (!q || !k || !v || !P || !dO || !dq || !dk || !dv_out || !dP || B < 0 || H < 0 ||
        N < 0 || d <= 0 || m <= 0 || dv <= 0)
        return 1;
    memset(dP, 0, sizeof(double) * (size_t)H * d * m);
    if (N == 0) return 0;
    const double rsm = 1.0 / sqrt((double)m); /* 1/sqrt(m) */
    double *qp = (double *)malloc(sizeof(double) * (size_t)N * m);
    double *kp = (double *)malloc(sizeof(double) * (size_t)N * m);
    double *dqp = (double *)malloc(sizeof(double) * (size_t)N * m);
    double *dkp = (double *)malloc(sizeof(double) * (size_t)N * m);
    double *rmax = (double *)malloc(sizeof(double) * (size_t)N);
    double *rsum = (double *)malloc(sizeof(double) * (size_t)N);
    double *rdot = (double *)malloc(sizeof(double) * (size_t)N);
    if (!qp || !kp || !dqp || !dkp || !rmax || !rsum || !rdot) {
        free(qp); free(kp); free(dqp); free(dkp); free(rmax); free(rsum); free(rdot);
        return 3;
    }
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            const size_t bh = (size_t)b * H + h;
            const size_t p_off = (size_t)h * d * m;
            #pragma omp parallel for schedule(static)
            for (long i = 0; i < N; ++i) {
                orc_project_row(q, dt, (bh * N + i) * d, P, p_off, d, m, qp + (size_t)i * m);
                orc_project_row(k, dt, (bh * N + i) * d, P, p_off, d, m, kp + (size_t)i * m);
            }
            /* pass 1, per row: M_i, l_i and D_i = <dO_i, O_i> */
            #pragma omp parallel
            {
                double *o = (double *)malloc(sizeof(double) * (size_t)dv);
                #pragma omp for schedule(dynamic, 4)
                for (long i = 0; i < N; ++i) {
                    const long kcount = causal ? i + 1 : N; /* keys row i sees */
                    double mx = -INFINITY;
                    for (long j = 0; j < kcount; ++j) {
                        double acc = 0.0;
                        for (int c = 0; c < m; ++c) acc += qp[(size_t)i * m + c] * kp[(size_t)j * m + c];
                        if (acc * rsm > mx) mx = acc * rsm;
                    }
                    double l = 0.0;
                    for (int c = 0; c < dv; ++c) o[c] = 0.0;
                    for (long j = 0; j < kcount; ++j) {
                        double acc = 0.0;
                        for (int c = 0; c < m; ++c) acc += qp[(size_t)i * m + c] * kp[(size_t)j * m + c];
                        const double e = exp(acc * rsm - mx);
                        l += e;
                        for (int c = 0; c < dv; ++c) o[c] += e * orc_load(v, dt, (bh * N + j) * dv + c);
                    }
                    double dot = 0.0;
                    for (int c = 0; c < dv; ++c) dot += orc_load(dO, dt, (bh * N + i) * dv + c) * (o[c] / l);
                    rmax[i] = mx;
                    rsum[i] = l;
                    rdot[i] = dot;
                }
                free(o);
            }
            /* A_ij and dS_ij, recomputed where needed */
            #define ORC_A(i, j, out_a, out_ds)                                                 \
                do {                                                                           \
                    double acc_ = 0.0;                                                         \
                    for (int c_ = 0; c_ < m; ++c_)                                             \
                        acc_ += qp[(size_t)(i) * m + c_] * kp[(size_t)(j) * m + c_];           \
                    const double a_ = exp(acc_ * rsm - rmax[i]) / rsum[i];              \
                    double da_ = 0.0;                                                          \
                    for (int c_ = 0; c_ < dv; ++c_)                                            \
                        da_ += orc_load(dO, dt, (bh * N + (i)) * dv + c_) *                    \
                               orc_load(v, dt, (bh * N + (j)) * dv + c_);                      \
                    (out_a) = a_;                                                              \
                    (out_ds) = a_ * (da_ - rdot[i]);                                           \
                } while (0)
            /* pass 2a, per row: dQp_i */
            #pragma omp parallel for schedule(dynamic, 4)
            for (long i = 0; i < N; ++i) {
                double *g = dqp + (size_t)i * m;
                for (int c = 0; c < m; ++c) g[c] = 0.0;
                const long kcount = causal ? i + 1 : N; /* keys row i sees */
                for (long j = 0; j < kcount; ++j) {
                    double a, ds;
                    ORC_A(i, j, a, ds);
                    (void)a;
                    for (int c = 0; c < m; ++c) g[c] += ds * kp[(size_t)j * m + c] * rsm;
                }
            }
            /* pass 2b, per key: dKp_j and dV_j */
            #pragma omp parallel for schedule(dynamic, 4)
            for (long j = 0; j < N; ++j) {
                double *g = dkp + (size_t)j * m;
                double *gv = dv_out + (bh * N + j) * dv;
                for (int c = 0; c < m; ++c) g[c] = 0.0;
                for (int c = 0; c < dv; ++c) gv[c] = 0.0;
                for (long i = causal ? j : 0; i < N; ++i) {
                    double a, ds;
                    ORC_A(i, j, a, ds);
                    for (int c = 0; c < m; ++c) g[c] += ds * qp[(size_t)i * m + c] * rsm;
                    for (int c = 0; c < dv; ++c) gv[c] += a * orc_load(dO, dt, (bh * N + i) * dv + c);
                }
            }
            #undef ORC_A
            /* step 2 backwards: dQ = dQp P^T, dK = dKp P^T, dP_h += Q^T dQp + K^T dKp */
            #pragma omp parallel for schedule(static)
            for (long i = 0; i < N; ++i) {
                for (int l = 0; l < d; ++l) {
                    double aq = 0.0, ak = 0.0;
                    for (int c = 0; c < m; ++c) {
                        const double p = orc_load(P, dt, p_off + (size_t)l * m + c);
                        aq += dqp[(size_t)i * m + c] * p;
                        ak += dkp[(size_t)i * m + c] * p;
                    }
                    dq[(bh * N + i) * d + l] = aq;
                    dk[(bh * N + i) * d + l] = ak;
                }
            }
            #pragma omp parallel for schedule(static)
            for (int l = 0; l < d; ++l) {
                for (int c = 0; c < m; ++c) {
                    double acc = 0.0;
                    for (long i = 0; i < N; ++i)
                        acc += orc_load(q, dt, (bh * N + i) * d + l) * dqp[(size_t)i * m + c] +
                               orc_load(k, dt, (bh * N + i) * d + l) * dkp[(size_t)i * m + c];
                    dP[p_off + (size_t)l * m + c] += acc;
                }
            }
        }
    }
    free(qp); free(kp); free(dqp); free(dkp); free(rmax); free(rsum); free(rdot);
    return 0;
}
