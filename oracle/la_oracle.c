/*
 * la_oracle.c -- float64 CPU oracle for fused linear attention, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call this
 * file: only the tests, the smoke check and the timed CPU baseline of the benchmark do.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (module neuralops.core.triton_kernels.linear_attn, functions `fwd`
 * and `bwd`; feature list in the module docstring):
 *
 *   a_i^p = w_i^p * phi(q_i)        b_j^p = w_j^p * phi(k_j)        (p = one term, or the
 *                                                                    cos and sin terms)
 *   S_i^p = sum_{j in J(i)} b_j^p v_j^T     z_i^p = sum_{j in J(i)} b_j^p
 *   num_i = sum_p (a_i^p)^T S_i^p            den_i = sum_p a_i^p . z_i^p + eps
 *   out_i = num_i / den_i
 *
 * with J(i) = {j <= i} when causal and all j otherwise, phi(x) = elu(x)+1 (alpha = 1),
 * relu(x) or x ("identity": the caller's features are used as they are), and w^p = 1 without position weights, else w^cos = cos_weight, w^sin =
 * sin_weight (cosFormer modulation: one weight per position, applied to phi(q_i) and
 * phi(k_i), never to v).  The state is the running prefix sum, taken in token order, so
 * this is the plain recurrent definition with no chunking, blocking or reordering.
 *
 * Grouped-query attention (module neuralops.core.triton_kernels.gqa): query head h reads
 * key/value head h / n_rep, n_rep = Hq / Hkv, as `gqa.fwd` expands them; the key/value
 * gradients are computed per query head and then summed over each group of n_rep
 * consecutive query heads, as `gqa.bwd` reduces them with view(B, Hkv, n_rep, N, D).sum(2).
 *
 * Backward (the linear_attn page's `bwd` returns the autograd gradient of `fwd`): with
 * g_i the output gradient,
 *   gn_i = g_i / den_i,  gd_i = -(g_i . num_i) / den_i^2
 *   da_i^p = S_i^p gn_i + gd_i z_i^p
 *   R_j^p = sum_{i : j in J(i)} a_i^p gn_i^T,  r_j^p = sum_{i : j in J(i)} gd_i a_i^p
 *   db_j^p = R_j^p v_j + r_j^p,   dv_j = sum_p (R_j^p)^T b_j^p
 *   dq_i = phi'(q_i) * sum_p w_i^p da_i^p,   dk_j = phi'(k_j) * sum_p w_j^p db_j^p
 * obtained by differentiating the definition above by hand (chain rule through out =
 * num/den).  phi'(x) = (x > 0 ? 1 : exp(x)) for elu+1, (x > 0 ? 1 : 0) for relu and 1 for
 * identity.
 *
 * Layout: every tensor is a contiguous row-major float64 array: q, k, dq, dk [B, H, N, D] and
 * v, out, grad_out, dv [B, H, N, Dv].  The value width Dv may differ from D: `fwd` takes v
 * as a tensor of its own and reads only q's head dimension, and the state S = sum b v^T is
 * D x Dv (the `_v` entry points; la_oracle_fwd and la_oracle_bwd take Dv = D).
 * The weights, when given, are float64 arrays of length N (both or neither).
 * The outer loop over (batch, query head) runs under OpenMP when built with -fopenmp;
 * each iteration writes only its own rows, and the group sum runs afterwards in a fixed
 * order, so the result does not depend on the thread count.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_PHI_ELU1 = 0, ORACLE_PHI_RELU = 1, ORACLE_PHI_IDENTITY = 2 };

static double feature(double x, int phi)
{
    if (phi == ORACLE_PHI_ELU1) return x > 0.0 ? x + 1.0 : exp(x);
    if (phi == ORACLE_PHI_IDENTITY) return x;
    return x > 0.0 ? x : 0.0;
}

static double feature_grad(double x, int phi)
{
    if (phi == ORACLE_PHI_ELU1) return x > 0.0 ? 1.0 : exp(x);
    if (phi == ORACLE_PHI_IDENTITY) return 1.0;
    return x > 0.0 ? 1.0 : 0.0;
}

int la_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Position weight of term p at position i (1 without weights). */
static double weight(const double *cw, const double *sw, int p, int i)
{
    if (!cw) return 1.0;
    return p == 0 ? cw[i] : sw[i];
}

/* Add token j of one key/value head to the state: S^p += b_j^p v_j^T, z^p += b_j^p
 * (S^p is D x Dv). */
static void add_token(double *S, double *z, const double *kj, const double *vj, int D,
                      int Dv, int P, int phi, const double *cw, const double *sw, int j)
{
    for (int p = 0; p < P; ++p) {
        double w = weight(cw, sw, p, j);
        for (int d = 0; d < D; ++d) {
            double bd = w * feature(kj[d], phi);
            z[p * D + d] += bd;
            for (int e = 0; e < Dv; ++e) S[(p * D + d) * Dv + e] += bd * vj[e];
        }
    }
}

/* num_i (Dv values) and den_i for query row i against the current state. */
static void read_out(const double *S, const double *z, const double *qi, int D, int Dv, int P,
                     int phi, const double *cw, const double *sw, int i, double eps,
                     double *num, double *den)
{
    for (int e = 0; e < Dv; ++e) num[e] = 0.0;
    double dn = 0.0;
    for (int p = 0; p < P; ++p) {
        double w = weight(cw, sw, p, i);
        for (int d = 0; d < D; ++d) {
            double ad = w * feature(qi[d], phi);
            dn += ad * z[p * D + d];
            for (int e = 0; e < Dv; ++e) num[e] += ad * S[(p * D + d) * Dv + e];
        }
    }
    *den = dn + eps;
}

static void head_forward(const double *qh, const double *kh, const double *vh, double *oh,
                         int N, int D, int Dv, int causal, int phi, double eps, const double *cw,
                         const double *sw)
{
    int P = cw ? 2 : 1;
    double *S = calloc((size_t)P * D * Dv, sizeof(double));
    double *z = calloc((size_t)P * D, sizeof(double));
    double *num = malloc((size_t)Dv * sizeof(double));
    if (!causal)
        for (int j = 0; j < N; ++j)
            add_token(S, z, kh + (size_t)j * D, vh + (size_t)j * Dv, D, Dv, P, phi, cw, sw, j);
    for (int i = 0; i < N; ++i) {
        if (causal)
            add_token(S, z, kh + (size_t)i * D, vh + (size_t)i * Dv, D, Dv, P, phi, cw, sw, i);
        double den;
        read_out(S, z, qh + (size_t)i * D, D, Dv, P, phi, cw, sw, i, eps, num, &den);
        for (int e = 0; e < Dv; ++e) oh[(size_t)i * Dv + e] = num[e] / den;
    }
    free(S);
    free(z);
    free(num);
}

void la_oracle_fwd_v(const double *q, const double *k, const double *v, double *out, int B,
                     int Hq, int Hkv, int N, int D, int Dv, int causal, int phi, double eps,
                     const double *cos_weight, const double *sin_weight)
{
    int n_rep = Hq / Hkv;
    size_t head = (size_t)N * D, vhead = (size_t)N * Dv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < B * Hq; ++bh) {
        int b = bh / Hq, h = bh % Hq, g = h / n_rep;
        size_t kv = (size_t)b * Hkv + g;
        head_forward(q + (size_t)bh * head, k + kv * head, v + kv * vhead, out + (size_t)bh * vhead,
                     N, D, Dv, causal, phi, eps, cos_weight, sin_weight);
    }
}

void la_oracle_fwd(const double *q, const double *k, const double *v, double *out, int B,
                   int Hq, int Hkv, int N, int D, int causal, int phi, double eps,
                   const double *cos_weight, const double *sin_weight)
{
    la_oracle_fwd_v(q, k, v, out, B, Hq, Hkv, N, D, D, causal, phi, eps, cos_weight, sin_weight);
}

/* Backward for one query head.  dk_h and dv_h receive this head's own contribution to
 * the gradient of its key/value head (summed over the group by the caller). */
static void head_backward(const double *qh, const double *kh, const double *vh,
                          const double *gh, double *dqh, double *dkh, double *dvh, int N,
                          int D, int Dv, int causal, int phi, double eps, const double *cw,
                          const double *sw)
{
    int P = cw ? 2 : 1;
    double *S = calloc((size_t)P * D * Dv, sizeof(double));
    double *z = calloc((size_t)P * D, sizeof(double));
    double *num = malloc((size_t)Dv * sizeof(double));
    double *gn = malloc((size_t)N * Dv * sizeof(double));  /* gn_i per row */
    double *gd = malloc((size_t)N * sizeof(double));       /* gd_i per row */

    /* Forward over i: the state S_i, z_i; the row gradients gn, gd; dq. */
    if (!causal)
        for (int j = 0; j < N; ++j)
            add_token(S, z, kh + (size_t)j * D, vh + (size_t)j * Dv, D, Dv, P, phi, cw, sw, j);
    for (int i = 0; i < N; ++i) {
        const double *qi = qh + (size_t)i * D, *gi = gh + (size_t)i * Dv;
        if (causal)
            add_token(S, z, kh + (size_t)i * D, vh + (size_t)i * Dv, D, Dv, P, phi, cw, sw, i);
        double den;
        read_out(S, z, qi, D, Dv, P, phi, cw, sw, i, eps, num, &den);
        double g_dot_num = 0.0;
        for (int e = 0; e < Dv; ++e) {
            gn[(size_t)i * Dv + e] = gi[e] / den;
            g_dot_num += gi[e] * num[e];
        }
        gd[i] = -g_dot_num / (den * den);
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;  /* sum_p w_i^p da_i^p[d] */
            for (int p = 0; p < P; ++p) {
                double da = gd[i] * z[p * D + d];
                for (int e = 0; e < Dv; ++e) da += S[(p * D + d) * Dv + e] * gn[(size_t)i * Dv + e];
                acc += weight(cw, sw, p, i) * da;
            }
            dqh[(size_t)i * D + d] = feature_grad(qi[d], phi) * acc;
        }
    }

    /* Backward over j: R_j^p (D x Dv), r_j^p summed over the rows i that attend to j. */
    double *R = calloc((size_t)P * D * Dv, sizeof(double));
    double *r = calloc((size_t)P * D, sizeof(double));
    if (!causal)
        for (int i = 0; i < N; ++i)
            for (int p = 0; p < P; ++p) {
                double w = weight(cw, sw, p, i);
                for (int d = 0; d < D; ++d) {
                    double ad = w * feature(qh[(size_t)i * D + d], phi);
                    r[p * D + d] += gd[i] * ad;
                    for (int e = 0; e < Dv; ++e) R[(p * D + d) * Dv + e] += ad * gn[(size_t)i * Dv + e];
                }
            }
    for (int j = N - 1; j >= 0; --j) {
        if (causal)
            for (int p = 0; p < P; ++p) {  /* row i = j attends to j */
                double w = weight(cw, sw, p, j);
                for (int d = 0; d < D; ++d) {
                    double ad = w * feature(qh[(size_t)j * D + d], phi);
                    r[p * D + d] += gd[j] * ad;
                    for (int e = 0; e < Dv; ++e) R[(p * D + d) * Dv + e] += ad * gn[(size_t)j * Dv + e];
                }
            }
        const double *kj = kh + (size_t)j * D, *vj = vh + (size_t)j * Dv;
        for (int e = 0; e < Dv; ++e) dvh[(size_t)j * Dv + e] = 0.0;
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;  /* sum_p w_j^p db_j^p[d] */
            for (int p = 0; p < P; ++p) {
                double w = weight(cw, sw, p, j);
                double bd = w * feature(kj[d], phi);
                double db = r[p * D + d];
                for (int e = 0; e < Dv; ++e) {
                    db += R[(p * D + d) * Dv + e] * vj[e];
                    dvh[(size_t)j * Dv + e] += R[(p * D + d) * Dv + e] * bd;
                }
                acc += w * db;
            }
            dkh[(size_t)j * D + d] = feature_grad(kj[d], phi) * acc;
        }
    }
    free(S); free(z); free(num); free(gn); free(gd); free(R); free(r);
}

/* Returns 0 on success, 1 when scratch memory for the per-query-head key/value
 * gradients could not be allocated. */
int la_oracle_bwd_v(const double *q, const double *k, const double *v, const double *grad_out,
                    double *dq, double *dk, double *dv, int B, int Hq, int Hkv, int N, int D,
                    int Dv, int causal, int phi, double eps, const double *cos_weight,
                    const double *sin_weight)
{
    int n_rep = Hq / Hkv;
    size_t head = (size_t)N * D, vhead = (size_t)N * Dv;
    /* Key/value gradients per query head, [B, Hq, N, D] and [B, Hq, N, Dv], as the expanded
     * tensors of the gqa page before its group reduction. */
    double *dk_x = malloc((size_t)B * Hq * head * sizeof(double));
    double *dv_x = malloc((size_t)B * Hq * vhead * sizeof(double));
    if (!dk_x || !dv_x) { free(dk_x); free(dv_x); return 1; }
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < B * Hq; ++bh) {
        int b = bh / Hq, h = bh % Hq, g = h / n_rep;
        size_t kv = (size_t)b * Hkv + g;
        head_backward(q + (size_t)bh * head, k + kv * head, v + kv * vhead, grad_out + (size_t)bh * vhead,
                      dq + (size_t)bh * head, dk_x + (size_t)bh * head, dv_x + (size_t)bh * vhead,
                      N, D, Dv, causal, phi, eps, cos_weight, sin_weight);
    }
    /* view(B, Hkv, n_rep, N, D).sum(2) (and N, Dv for dv), in a fixed order. */
    for (int b = 0; b < B; ++b)
        for (int g = 0; g < Hkv; ++g) {
            double *dkg = dk + ((size_t)b * Hkv + g) * head, *dvg = dv + ((size_t)b * Hkv + g) * vhead;
            for (size_t t = 0; t < head; ++t) dkg[t] = 0.0;
            for (size_t t = 0; t < vhead; ++t) dvg[t] = 0.0;
            for (int rr = 0; rr < n_rep; ++rr) {
                size_t src = (size_t)b * Hq + (size_t)g * n_rep + rr;
                for (size_t t = 0; t < head; ++t) dkg[t] += dk_x[src * head + t];
                for (size_t t = 0; t < vhead; ++t) dvg[t] += dv_x[src * vhead + t];
            }
        }
    free(dk_x);
    free(dv_x);
    return 0;
}

int la_oracle_bwd(const double *q, const double *k, const double *v, const double *grad_out,
                  double *dq, double *dk, double *dv, int B, int Hq, int Hkv, int N, int D,
                  int causal, int phi, double eps, const double *cos_weight,
                  const double *sin_weight)
{
    return la_oracle_bwd_v(q, k, v, grad_out, dq, dk, dv, B, Hq, Hkv, N, D, D, causal, phi, eps,
                           cos_weight, sin_weight);
}
