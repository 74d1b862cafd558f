/*
 * Oracle for the causal dot product -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load or run this code.  The product path (the CUDA library and its
 * Python binding) never calls it and shares no code with it.
 *
 * What it computes (fp64 throughout, plain C, one (b,h) slice at a time):
 *
 *   Forward.  For one (b,h) with q,k in R^{N x D} and v in R^{N x M}:
 *       S_i   = sum_{j<=i} k_j v_j^T                 (a D x M matrix)
 *       out_i = S_i^T q_i  =  sum_{j<=i} (q_i . k_j) v_j
 *   This is the recurrent form of causal linear attention that
 *   triton-lang/triton issue #217 ("Dot Product Computes Wrong Values")
 *   sets out to batch-parallelise: the opening comment names Algorithm 1 of
 *   "Transformers are RNNs" and describes it as a prefix sum over the
 *   sequence; the loop body shown later in the same issue adds the outer
 *   product of the current key and value rows to a running state and then
 *   reads the output out of that state with the query (the comment there
 *   notes that the readout must use the query, not the key).  The state is
 *   updated before the readout, so row i sees itself (inclusive, j <= i).
 *   No normaliser and no 1/sqrt(D) scale are applied: neither appears in
 *   that loop.
 *
 *   Backward.  The pages print no backward; it follows from the definition.
 *   With g_i = dL/dout_i and L = sum_i <g_i, out_i>:
 *       dq_i = S_i g_i                         (forward sweep over i)
 *       R_j  = sum_{i>=j} q_i g_i^T            (reverse sweep over j)
 *       dk_j = R_j v_j,    dv_j = R_j^T k_j
 *
 *   Carried state.  The loop in the issue keeps its state across the
 *   sequence (the Triton port there takes the state as an argument), so a
 *   call may start from an initial state S_0 and hand on its final state:
 *       S_i = S_0 + sum_{j<=i} k_j v_j^T,      S_N = S_0 + sum_j k_j v_j^T.
 *   With L = sum_i <g_i, out_i> + <dS_N, S_N> the backward becomes
 *       dq_i = S_i g_i,    R_j = dS_N + sum_{i>=j} q_i g_i^T,
 *       dk_j = R_j v_j,    dv_j = R_j^T k_j,    dS_0 = R_0
 *   (S_0 enters every S_i, and dS_N every R_j).  Absent states are zero.
 *
 *   Normaliser.  Causal linear attention ("Transformers are RNNs", the
 *   paper the issue cites for the recurrence) divides each output row by
 *       z_i = q_i . c_i,       c_i = sum_{j<=i} k_j
 *   (the issue's loop leaves it out).  Its backward, from the definition
 *   with L = sum_i g_i z_i:
 *       dq_i = g_i c_i,        dk_j = sum_{i>=j} g_i q_i.
 *
 *   Feature map.  Causal linear attention feeds the product phi(q) and
 *   phi(k), with phi(x) = elu(x) + 1 (x + 1 for x > 0, e^x otherwise) in
 *   "Transformers are RNNs".  The feature entry points take the raw q, k,
 *   map them in double, run the same recurrences, and apply the chain rule
 *   dL/dx = dL/dphi * phi'(x), phi'(x) = 1 for x > 0, e^x otherwise.
 *
 *   Positive random features.  The issue names Performer-style models as
 *   users of the kernel.  Their feature map (positive random features of
 *   the softmax kernel) takes a raw row x in R^r and one projection W in
 *   R^{D x r}, shared by every row and slice, and gives a D-vector:
 *       phi(x)_d = exp(w_d . x - |x|^2 / 2) / sqrt(D).
 *   The product of phi(xq), phi(xk) and v runs the same recurrences.  With
 *   a = dL/dphi(x) for one row, the chain rule gives
 *       dL/dx = sum_d a_d phi_d (w_d - x) = W^T (a * phi) - x (a . phi).
 *   W is an input, not a trained parameter: no gradient is formed for it.
 *
 * Inputs are float32 arrays holding the exact values the GPU receives
 * (bfloat16 values are exactly representable in float32 and in double);
 * each slice is widened to double before any arithmetic.  Outputs are
 * double.  Layout: contiguous row-major [BH][N][D] / [BH][N][M].
 *
 * Parallelism: OpenMP over the independent (b,h) slices only; the sweep
 * inside a slice is the plain serial loop, in sequence order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Widen one [N][C] float slice to double. */
static void widen(const float *src, double *dst, int64_t n) {
    for (int64_t i = 0; i < n; ++i) dst[i] = (double)src[i];
}

/* The feature map (feature 1: elu + 1) and its derivative. */
static double phi(int feature, double x) {
    if (feature == 1) return x > 0.0 ? x + 1.0 : exp(x);
    return x;
}

static double dphi(int feature, double x) {
    if (feature == 1) return x > 0.0 ? 1.0 : exp(x);
    return 1.0;
}

/* Widen one [N][C] float slice to double, mapped by the feature map. */
static void widen_phi(const float *src, double *dst, int64_t n, int feature) {
    for (int64_t i = 0; i < n; ++i) dst[i] = phi(feature, (double)src[i]);
}

/* Forward recurrence on one (b,h) slice; all arrays double, row-major.
 * S0 (may be NULL: zero) is the initial state; the final state goes to SN
 * when SN is not NULL. */
static void fwd_slice(const double *q, const double *k, const double *v,
                      double *out, double *S, const double *S0, double *SN,
                      int64_t N, int64_t D, int64_t M) {
    /* start from the initial state */
    if (S0) memcpy(S, S0, sizeof(double) * (size_t)(D * M));
    else memset(S, 0, sizeof(double) * (size_t)(D * M));
    for (int64_t i = 0; i < N; ++i) {
        const double *ki = k + i * D, *vi = v + i * M, *qi = q + i * D;
        /* state update: S += k_i v_i^T */
        for (int64_t d = 0; d < D; ++d) {
            double kd = ki[d];
            double *Sd = S + d * M;
            for (int64_t m = 0; m < M; ++m) Sd[m] += kd * vi[m];
        }
        /* readout: out_i = S^T q_i */
        double *oi = out + i * M;
        for (int64_t m = 0; m < M; ++m) oi[m] = 0.0;
        for (int64_t d = 0; d < D; ++d) {
            double qd = qi[d];
            const double *Sd = S + d * M;
            for (int64_t m = 0; m < M; ++m) oi[m] += qd * Sd[m];
        }
    }
    if (SN) memcpy(SN, S, sizeof(double) * (size_t)(D * M));
}

/* Backward on one (b,h) slice.  S0 and dSN (may be NULL: zero) are the
 * initial state and the gradient of the final state; dS0 (when not NULL)
 * receives the gradient of the initial state. */
static void bwd_slice(const double *q, const double *k, const double *v,
                      const double *g, double *dq, double *dk, double *dv,
                      double *S, const double *S0, const double *dSN, double *dS0,
                      int64_t N, int64_t D, int64_t M) {
    /* forward sweep: S_i = S_0 + sum_{j<=i} k_j v_j^T ; dq_i = S_i g_i */
    if (S0) memcpy(S, S0, sizeof(double) * (size_t)(D * M));
    else memset(S, 0, sizeof(double) * (size_t)(D * M));
    for (int64_t i = 0; i < N; ++i) {
        const double *ki = k + i * D, *vi = v + i * M, *gi = g + i * M;
        for (int64_t d = 0; d < D; ++d) {
            double kd = ki[d];
            double *Sd = S + d * M;
            for (int64_t m = 0; m < M; ++m) Sd[m] += kd * vi[m];
        }
        double *dqi = dq + i * D;
        for (int64_t d = 0; d < D; ++d) {
            const double *Sd = S + d * M;
            double acc = 0.0;
            for (int64_t m = 0; m < M; ++m) acc += Sd[m] * gi[m];
            dqi[d] = acc;
        }
    }
    /* reverse sweep: R_j = dS_N + sum_{i>=j} q_i g_i^T ; dk_j = R_j v_j ; dv_j = R_j^T k_j */
    double *R = S;
    if (dSN) memcpy(R, dSN, sizeof(double) * (size_t)(D * M));
    else memset(R, 0, sizeof(double) * (size_t)(D * M));
    for (int64_t j = N - 1; j >= 0; --j) {
        const double *qj = q + j * D, *gj = g + j * M;
        const double *kj = k + j * D, *vj = v + j * M;
        for (int64_t d = 0; d < D; ++d) {
            double qd = qj[d];
            double *Rd = R + d * M;
            for (int64_t m = 0; m < M; ++m) Rd[m] += qd * gj[m];
        }
        double *dkj = dk + j * D;
        for (int64_t d = 0; d < D; ++d) {
            const double *Rd = R + d * M;
            double acc = 0.0;
            for (int64_t m = 0; m < M; ++m) acc += Rd[m] * vj[m];
            dkj[d] = acc;
        }
        double *dvj = dv + j * M;
        for (int64_t m = 0; m < M; ++m) dvj[m] = 0.0;
        for (int64_t d = 0; d < D; ++d) {
            double kd = kj[d];
            const double *Rd = R + d * M;
            for (int64_t m = 0; m < M; ++m) dvj[m] += kd * Rd[m];
        }
    }
    /* dS_0 = R_0 */
    if (dS0) memcpy(dS0, R, sizeof(double) * (size_t)(D * M));
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

/* Number of threads the oracle will use when called with `nthreads`
 * (<= 0 means the OpenMP default). */
int cpo_threads(int nthreads) { return set_threads(nthreads); }

/* Forward over BH slices.  state_in [BH][D][M] (may be NULL: zero) is the
 * initial state of every slice, state_out [BH][D][M] (may be NULL) receives
 * the final state.  Returns 0 on success, -1 on a bad argument, -2 when a
 * scratch allocation fails. */
int cpo_fwd_state(const float *q, const float *k, const float *v, double *out,
                  const double *state_in, double *state_out,
                  int64_t BH, int64_t N, int64_t D, int64_t M, int nthreads) {
    if (BH < 0 || N < 0 || D <= 0 || M <= 0) return -1;
    if (BH == 0) return 0;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *buf = (double *)malloc(sizeof(double) * (size_t)(N * (2 * D + M) + D * M));
        if (!buf) { err |= 1; continue; }
        double *qd = buf, *kd = qd + N * D, *vd = kd + N * D, *S = vd + N * M;
        widen(q + bh * N * D, qd, N * D);
        widen(k + bh * N * D, kd, N * D);
        widen(v + bh * N * M, vd, N * M);
        fwd_slice(qd, kd, vd, out + bh * N * M, S, state_in ? state_in + bh * D * M : NULL,
                  state_out ? state_out + bh * D * M : NULL, N, D, M);
        free(buf);
    }
    return err ? -2 : 0;
}

/* Forward over BH slices without carried state. */
int cpo_fwd(const float *q, const float *k, const float *v, double *out,
            int64_t BH, int64_t N, int64_t D, int64_t M, int nthreads) {
    if (N == 0) return (BH < 0 || D <= 0 || M <= 0) ? -1 : 0;
    return cpo_fwd_state(q, k, v, out, NULL, NULL, BH, N, D, M, nthreads);
}

/* Backward over BH slices: g is dL/dout; writes dq, dk, dv.  state_in and
 * grad_state_out [BH][D][M] (may be NULL: zero) are the initial state and
 * dL/dS_N; grad_state_in (may be NULL) receives dL/dS_0. */
int cpo_bwd_state(const float *q, const float *k, const float *v, const float *g,
                  const double *state_in, const double *grad_state_out,
                  double *dq, double *dk, double *dv, double *grad_state_in,
                  int64_t BH, int64_t N, int64_t D, int64_t M, int nthreads) {
    if (BH < 0 || N < 0 || D <= 0 || M <= 0) return -1;
    if (BH == 0) return 0;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *buf = (double *)malloc(sizeof(double) * (size_t)(N * (2 * D + 2 * M) + D * M));
        if (!buf) { err |= 1; continue; }
        double *qd = buf, *kd = qd + N * D, *vd = kd + N * D, *gd = vd + N * M;
        double *S = gd + N * M;
        widen(q + bh * N * D, qd, N * D);
        widen(k + bh * N * D, kd, N * D);
        widen(v + bh * N * M, vd, N * M);
        widen(g + bh * N * M, gd, N * M);
        bwd_slice(qd, kd, vd, gd, dq + bh * N * D, dk + bh * N * D, dv + bh * N * M, S,
                  state_in ? state_in + bh * D * M : NULL,
                  grad_state_out ? grad_state_out + bh * D * M : NULL,
                  grad_state_in ? grad_state_in + bh * D * M : NULL, N, D, M);
        free(buf);
    }
    return err ? -2 : 0;
}

/* Backward over BH slices without carried state. */
int cpo_bwd(const float *q, const float *k, const float *v, const float *g,
            double *dq, double *dk, double *dv,
            int64_t BH, int64_t N, int64_t D, int64_t M, int nthreads) {
    if (N == 0) return (BH < 0 || D <= 0 || M <= 0) ? -1 : 0;
    return cpo_bwd_state(q, k, v, g, NULL, NULL, dq, dk, dv, NULL, BH, N, D, M, nthreads);
}

/* Normaliser over BH slices: z [BH][N] (double) = q_i . sum_{j<=i} k_j. */
int cpo_norm(const float *q, const float *k, double *z, int64_t BH, int64_t N, int64_t D,
             int nthreads) {
    if (BH < 0 || N < 0 || D <= 0) return -1;
    if (BH == 0 || N == 0) return 0;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *c = (double *)calloc((size_t)D, sizeof(double));
        if (!c) { err |= 1; continue; }
        const float *qs = q + bh * N * D, *ks = k + bh * N * D;
        for (int64_t i = 0; i < N; ++i) {
            /* c += k_i, then z_i = q_i . c */
            for (int64_t d = 0; d < D; ++d) c[d] += (double)ks[i * D + d];
            double acc = 0.0;
            for (int64_t d = 0; d < D; ++d) acc += (double)qs[i * D + d] * c[d];
            z[bh * N + i] = acc;
        }
        free(c);
    }
    return err ? -2 : 0;
}

/* Backward of the normaliser: g [BH][N] is dL/dz; writes dq, dk [BH][N][D]. */
int cpo_norm_bwd(const float *q, const float *k, const float *g, double *dq, double *dk,
                 int64_t BH, int64_t N, int64_t D, int nthreads) {
    if (BH < 0 || N < 0 || D <= 0) return -1;
    if (BH == 0 || N == 0) return 0;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *c = (double *)calloc((size_t)D, sizeof(double));
        if (!c) { err |= 1; continue; }
        const float *qs = q + bh * N * D, *ks = k + bh * N * D, *gs = g + bh * N;
        double *dqs = dq + bh * N * D, *dks = dk + bh * N * D;
        /* forward sweep: c_i = sum_{j<=i} k_j ; dq_i = g_i c_i */
        for (int64_t i = 0; i < N; ++i) {
            for (int64_t d = 0; d < D; ++d) {
                c[d] += (double)ks[i * D + d];
                dqs[i * D + d] = (double)gs[i] * c[d];
            }
        }
        /* reverse sweep: r_j = sum_{i>=j} g_i q_i ; dk_j = r_j */
        memset(c, 0, sizeof(double) * (size_t)D);
        for (int64_t j = N - 1; j >= 0; j--) {
            for (int64_t d = 0; d < D; ++d) {
                c[d] += (double)gs[j] * (double)qs[j * D + d];
                dks[j * D + d] = c[d];
            }
        }
        free(c);
    }
    return err ? -2 : 0;
}

/* Forward of the causal product of phi(q), phi(k) and v (feature 0: q, k
 * as given, feature 1: elu + 1). */
int cpo_fwd_feature(const float *q, const float *k, const float *v, double *out, int feature,
                    int64_t BH, int64_t N, int64_t D, int64_t M, int nthreads) {
    if (BH < 0 || N < 0 || D <= 0 || M <= 0 || feature < 0 || feature > 1) return -1;
    if (BH == 0 || N == 0) return 0;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *buf = (double *)malloc(sizeof(double) * (size_t)(N * (2 * D + M) + D * M));
        if (!buf) { err |= 1; continue; }
        double *qd = buf, *kd = qd + N * D, *vd = kd + N * D, *S = vd + N * M;
        widen_phi(q + bh * N * D, qd, N * D, feature);
        widen_phi(k + bh * N * D, kd, N * D, feature);
        widen(v + bh * N * M, vd, N * M);
        fwd_slice(qd, kd, vd, out + bh * N * M, S, NULL, NULL, N, D, M);
        free(buf);
    }
    return err ? -2 : 0;
}

/* Backward of cpo_fwd_feature with respect to the raw q, k and v. */
int cpo_bwd_feature(const float *q, const float *k, const float *v, const float *g, double *dq,
                    double *dk, double *dv, int feature, int64_t BH, int64_t N, int64_t D,
                    int64_t M, int nthreads) {
    if (BH < 0 || N < 0 || D <= 0 || M <= 0 || feature < 0 || feature > 1) return -1;
    if (BH == 0 || N == 0) return 0;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *buf = (double *)malloc(sizeof(double) * (size_t)(N * (2 * D + 2 * M) + D * M));
        if (!buf) { err |= 1; continue; }
        double *qd = buf, *kd = qd + N * D, *vd = kd + N * D, *gd = vd + N * M;
        double *S = gd + N * M;
        const float *qs = q + bh * N * D, *ks = k + bh * N * D;
        widen_phi(qs, qd, N * D, feature);
        widen_phi(ks, kd, N * D, feature);
        widen(v + bh * N * M, vd, N * M);
        widen(g + bh * N * M, gd, N * M);
        double *dqs = dq + bh * N * D, *dks = dk + bh * N * D;
        bwd_slice(qd, kd, vd, gd, dqs, dks, dv + bh * N * M, S, NULL, NULL, NULL, N, D, M);
        /* chain rule through phi */
        for (int64_t e = 0; e < N * D; ++e) {
            dqs[e] *= dphi(feature, (double)qs[e]);
            dks[e] *= dphi(feature, (double)ks[e]);
        }
        free(buf);
    }
    return err ? -2 : 0;
}

/* phi of every row of one [N][r] slice into [N][D] (positive random
 * features, W row-major [D][r]). */
static void favor_slice(const float *x, const float *W, int64_t N, int64_t r, int64_t D,
                        double *phi) {
    const double scale = 1.0 / sqrt((double)D);
    for (int64_t i = 0; i < N; ++i) {
        const float *xi = x + i * r;
        double n2 = 0.0;
        for (int64_t t = 0; t < r; ++t) n2 += (double)xi[t] * (double)xi[t];
        for (int64_t d = 0; d < D; ++d) {
            double wx = 0.0;
            for (int64_t t = 0; t < r; ++t) wx += (double)W[d * r + t] * (double)xi[t];
            phi[i * D + d] = exp(wx - 0.5 * n2) * scale;
        }
    }
}

/* dL/dx of one slice from a = dL/dphi: W^T (a * phi) - x (a . phi) per row. */
static void favor_grad(const float *x, const float *W, const double *phi, const double *a,
                       int64_t N, int64_t r, int64_t D, double *dx) {
    for (int64_t i = 0; i < N; ++i) {
        const double *pi = phi + i * D, *ai = a + i * D;
        double s = 0.0;
        for (int64_t d = 0; d < D; ++d) s += ai[d] * pi[d];
        for (int64_t t = 0; t < r; ++t) {
            double acc = 0.0;
            for (int64_t d = 0; d < D; ++d) acc += (double)W[d * r + t] * (ai[d] * pi[d]);
            dx[i * r + t] = acc - (double)x[i * r + t] * s;
        }
    }
}

/* Forward of the causal product of phi(xq), phi(xk) and v with positive
 * random features: xq, xk [BH][N][r], W [D][r], v [BH][N][M] -> out
 * [BH][N][M]. */
int cpo_fwd_favor(const float *xq, const float *xk, const float *v, const float *W, double *out,
                  int64_t BH, int64_t N, int64_t r, int64_t D, int64_t M, int nthreads) {
    if (BH < 0 || N < 0 || r <= 0 || D <= 0 || M <= 0) return -1;
    if (BH == 0 || N == 0) return 0;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *buf = (double *)malloc(sizeof(double) * (size_t)(N * (2 * D + M) + D * M));
        if (!buf) { err |= 1; continue; }
        double *qd = buf, *kd = qd + N * D, *vd = kd + N * D, *S = vd + N * M;
        favor_slice(xq + bh * N * r, W, N, r, D, qd);
        favor_slice(xk + bh * N * r, W, N, r, D, kd);
        widen(v + bh * N * M, vd, N * M);
        fwd_slice(qd, kd, vd, out + bh * N * M, S, NULL, NULL, N, D, M);
        free(buf);
    }
    return err ? -2 : 0;
}

/* Backward of cpo_fwd_favor with respect to xq, xk and v (W fixed):
 * dxq, dxk [BH][N][r], dv [BH][N][M]. */
int cpo_bwd_favor(const float *xq, const float *xk, const float *v, const float *W,
                  const float *g, double *dxq, double *dxk, double *dv, int64_t BH, int64_t N,
                  int64_t r, int64_t D, int64_t M, int nthreads) {
    if (BH < 0 || N < 0 || r <= 0 || D <= 0 || M <= 0) return -1;
    if (BH == 0 || N == 0) return 0;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *buf = (double *)malloc(sizeof(double) * (size_t)(N * (4 * D + 2 * M) + D * M));
        if (!buf) { err |= 1; continue; }
        double *qd = buf, *kd = qd + N * D, *aq = kd + N * D, *ak = aq + N * D;
        double *vd = ak + N * D, *gd = vd + N * M, *S = gd + N * M;
        const float *xqs = xq + bh * N * r, *xks = xk + bh * N * r;
        favor_slice(xqs, W, N, r, D, qd);
        favor_slice(xks, W, N, r, D, kd);
        widen(v + bh * N * M, vd, N * M);
        widen(g + bh * N * M, gd, N * M);
        /* dL/dphi(q), dL/dphi(k) and dv from the plain recurrences */
        bwd_slice(qd, kd, vd, gd, aq, ak, dv + bh * N * M, S, NULL, NULL, NULL, N, D, M);
        favor_grad(xqs, W, qd, aq, N, r, D, dxq + bh * N * r);
        favor_grad(xks, W, kd, ak, N, r, D, dxk + bh * N * r);
        free(buf);
    }
    return err ? -2 : 0;
}

/* Normaliser of positive random features: z_i = phi(xq_i) . sum_{j<=i}
 * phi(xk_j), xq, xk [BH][N][r], W [D][r] -> z [BH][N]. */
int cpo_norm_favor(const float *xq, const float *xk, const float *W, double *z, int64_t BH,
                   int64_t N, int64_t r, int64_t D, int nthreads) {
    if (BH < 0 || N < 0 || r <= 0 || D <= 0) return -1;
    if (BH == 0 || N == 0) return 0;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *buf = (double *)malloc(sizeof(double) * (size_t)(2 * N * D + D));
        if (!buf) { err |= 1; continue; }
        double *pq = buf, *pk = pq + N * D, *c = pk + N * D;
        favor_slice(xq + bh * N * r, W, N, r, D, pq);
        favor_slice(xk + bh * N * r, W, N, r, D, pk);
        memset(c, 0, sizeof(double) * (size_t)D);
        for (int64_t i = 0; i < N; ++i) {
            /* c += phi(k_i), then z_i = phi(q_i) . c */
            for (int64_t d = 0; d < D; ++d) c[d] += pk[i * D + d];
            double acc = 0.0;
            for (int64_t d = 0; d < D; ++d) acc += pq[i * D + d] * c[d];
            z[bh * N + i] = acc;
        }
        free(buf);
    }
    return err ? -2 : 0;
}

/* Backward of cpo_norm_favor with respect to xq and xk (W fixed), from
 * g = dL/dz [BH][N]: dL/dphi(q_i) = g_i c_i, dL/dphi(k_j) = sum_{i>=j}
 * g_i phi(q_i), then the chain rule through phi. */
int cpo_norm_bwd_favor(const float *xq, const float *xk, const float *W, const float *g,
                       double *dxq, double *dxk, int64_t BH, int64_t N, int64_t r, int64_t D,
                       int nthreads) {
    if (BH < 0 || N < 0 || r <= 0 || D <= 0) return -1;
    if (BH == 0 || N == 0) return 0;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *buf = (double *)malloc(sizeof(double) * (size_t)(4 * N * D + D));
        if (!buf) { err |= 1; continue; }
        double *pq = buf, *pk = pq + N * D, *aq = pk + N * D, *ak = aq + N * D;
        double *c = ak + N * D;
        const float *xqs = xq + bh * N * r, *xks = xk + bh * N * r, *gs = g + bh * N;
        favor_slice(xqs, W, N, r, D, pq);
        favor_slice(xks, W, N, r, D, pk);
        memset(c, 0, sizeof(double) * (size_t)D);
        for (int64_t i = 0; i < N; ++i) {
            for (int64_t d = 0; d < D; ++d) c[d] += pk[i * D + d];
            for (int64_t d = 0; d < D; ++d) aq[i * D + d] = (double)gs[i] * c[d];
        }
        memset(c, 0, sizeof(double) * (size_t)D);
        for (int64_t j = N - 1; j >= 0; j -= 1) {
            for (int64_t d = 0; d < D; ++d) c[d] += (double)gs[j] * pq[j * D + d];
            for (int64_t d = 0; d < D; ++d) ak[j * D + d] = c[d];
        }
        favor_grad(xqs, W, pq, aq, N, r, D, dxq + bh * N * r);
        favor_grad(xks, W, pk, ak, N, r, D, dxk + bh * N * r);
        free(buf);
    }
    return err ? -2 : 0;
}

/* Normaliser of mapped features: z_i = phi(q_i) . sum_{j<=i} phi(k_j) from
 * the raw q, k (feature 0: as given, 1: elu + 1). */
int cpo_norm_feature(const float *q, const float *k, double *z, int feature, int64_t BH,
                     int64_t N, int64_t D, int nthreads) {
    if (BH < 0 || N < 0 || D <= 0 || feature < 0 || feature > 1) return -1;
    if (BH == 0 || N == 0) return 0;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *c = (double *)calloc((size_t)D, sizeof(double));
        if (!c) { err |= 1; continue; }
        const float *qs = q + bh * N * D, *ks = k + bh * N * D;
        for (int64_t i = 0; i < N; ++i) {
            /* c += phi(k_i), then z_i = phi(q_i) . c */
            for (int64_t d = 0; d < D; ++d) c[d] += phi(feature, (double)ks[i * D + d]);
            double acc = 0.0;
            for (int64_t d = 0; d < D; ++d) acc += phi(feature, (double)qs[i * D + d]) * c[d];
            z[bh * N + i] = acc;
        }
        free(c);
    }
    return err ? -2 : 0;
}

/* Backward of cpo_norm_feature with respect to the raw q, k:
 *   dq_i = phi'(q_i) * g_i sum_{j<=i} phi(k_j),
 *   dk_j = phi'(k_j) * sum_{i>=j} g_i phi(q_i). */
int cpo_norm_bwd_feature(const float *q, const float *k, const float *g, double *dq, double *dk,
                         int feature, int64_t BH, int64_t N, int64_t D, int nthreads) {
    if (BH < 0 || N < 0 || D <= 0 || feature < 0 || feature > 1) return -1;
    if (BH == 0 || N == 0) return 0;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *c = (double *)calloc((size_t)D, sizeof(double));
        if (!c) { err |= 1; continue; }
        const float *qs = q + bh * N * D, *ks = k + bh * N * D, *gs = g + bh * N;
        double *dqs = dq + bh * N * D, *dks = dk + bh * N * D;
        for (int64_t i = 0; i < N; ++i) {
            for (int64_t d = 0; d < D; ++d) {
                const double qx = (double)qs[i * D + d];
                c[d] += phi(feature, (double)ks[i * D + d]);
                dqs[i * D + d] = dphi(feature, qx) * ((double)gs[i] * c[d]);
            }
        }
        memset(c, 0, sizeof(double) * (size_t)D);
        for (int64_t j = N - 1; j >= 0; j -= 1) {
            for (int64_t d = 0; d < D; ++d) {
                c[d] += (double)gs[j] * phi(feature, (double)qs[j * D + d]);
                dks[j * D + d] = dphi(feature, (double)ks[j * D + d]) * c[d];
            }
        }
        free(c);
    }
    return err ? -2 : 0;
}
