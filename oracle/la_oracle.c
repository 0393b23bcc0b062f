/*
 * la_oracle.c -- fp64 CPU oracle for causal linear attention with a carried
 * running state.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * bench's CPU-baseline / reference arm may load this file's library.  The
 * product path (the CUDA kernels behind include/la.h) never calls it, and
 * this file includes nothing from the product.
 *
 * Source of the method: "Fractus-1B training optimization -- 2026-08-22".
 *   - Section 1, "Bottleneck #1": the running state is a causal cumulative
 *     sum of outer products, S_t = sum_{j<=t} outer_j (the masked einsum
 *     "tj,bjpq->btpq" with a lower-triangular mask), and the derivative of
 *     a cumsum is a reverse cumsum.
 *   - Section 2, "Opt 2": the chunked form -- a masked block x block score
 *     matrix inside a block plus the running state (S_run, z_run) across
 *     blocks, with the inclusive update done AFTER reading.
 *   - Section 2, "Opt 6": the state (carry) is threaded from one chunk to
 *     the next (carry_S_flat, carry_z_flat -> S_final, z_final).
 * The page does not print the output normalisation.  The reading used here
 * (stated once, used everywhere):
 *     S_t = S0 + sum_{j<=t} k_j v_j^T     (S[p][c], p = key dim, c = value dim)
 *     z_t = z0 + sum_{j<=t} k_j
 *     o_t[c] = sum_p q_t[p] S_t[p][c] / (q_t . z_t + eps)
 * eps is added (no clamp, no abs) and receives no gradient.
 *
 * Layouts (row-major, contiguous, fp64):
 *   q, k, v, o, dO, dq, dk, dv : [G][C][D]
 *   S0, S_out, dS_out, dS0     : [G][D][D]
 *   z0, z_out, dz_out, dz0     : [G][D]
 * A NULL S0 / z0 / dS_out / dz_out means all zeros.
 *
 * Every group g is independent; groups run in parallel under OpenMP.  The
 * arithmetic inside a group is plain sequential fp64 in the order written.
 */
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define IDX3(g, t, x, C, D) (((size_t)(g) * (size_t)(C) + (size_t)(t)) * (size_t)(D) + (size_t)(x))

int la_oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static void load_carry(int D, int g, const double* S0, const double* z0, double* S, double* z)
{
    size_t DD = (size_t)D * D;
    if (S0) memcpy(S, S0 + (size_t)g * DD, DD * sizeof(double));
    else memset(S, 0, DD * sizeof(double));
    if (z0) memcpy(z, z0 + (size_t)g * D, (size_t)D * sizeof(double));
    else memset(z, 0, (size_t)D * sizeof(double));
}

/*
 * Forward, per-token loop: the definition written out.  For each token the
 * state first absorbs k_t v_t^T (inclusive of t), then is read by q_t.
 */
void la_oracle_fwd(int G, int C, int D,
                   const double* q, const double* k, const double* v,
                   const double* S0, const double* z0, double eps,
                   double* o, double* S_out, double* z_out)
{
    #pragma omp parallel for schedule(dynamic, 1)
    for (int g = 0; g < G; ++g) {
        double* S = (double*)malloc((size_t)D * D * sizeof(double));
        double* z = (double*)malloc((size_t)D * sizeof(double));
        load_carry(D, g, S0, z0, S, z);
        for (int t = 0; t < C; ++t) {
            const double* qt = q + IDX3(g, t, 0, C, D);
            const double* kt = k + IDX3(g, t, 0, C, D);
            const double* vt = v + IDX3(g, t, 0, C, D);
            for (int p = 0; p < D; ++p) {
                for (int c = 0; c < D; ++c) S[(size_t)p * D + c] += kt[p] * vt[c];
                z[p] += kt[p];
            }
            double den = 0.0;
            for (int p = 0; p < D; ++p) den += qt[p] * z[p];
            den += eps;
            double* ot = o + IDX3(g, t, 0, C, D);
            for (int c = 0; c < D; ++c) {
                double num = 0.0;
                for (int p = 0; p < D; ++p) num += qt[p] * S[(size_t)p * D + c];
                ot[c] = num / den;
            }
        }
        if (S_out) memcpy(S_out + (size_t)g * D * D, S, (size_t)D * D * sizeof(double));
        if (z_out) memcpy(z_out + (size_t)g * D, z, (size_t)D * sizeof(double));
        free(S);
        free(z);
    }
}

/*
 * Backward of la_oracle_fwd, per token.  With n_t = S_t^T q_t and
 * den_t = q_t . z_t + eps:
 *   dn_t = dO_t / den_t,   dd_t = -(dO_t . n_t) / den_t^2
 *   dq_t = S_t dn_t + dd_t z_t
 * Every S_t, z_t (t >= j) contains k_j v_j^T and k_j, so the gradients that
 * reach token j are the reverse (suffix) cumsums
 *   R_j = dS_out + sum_{t>=j} q_t dn_t^T,   r_j = dz_out + sum_{t>=j} dd_t q_t
 * and dk_j = R_j v_j + r_j, dv_j = R_j^T k_j; dS0 = R_0, dz0 = r_0.
 */
void la_oracle_bwd(int G, int C, int D,
                   const double* q, const double* k, const double* v,
                   const double* S0, const double* z0,
                   const double* dO, const double* dS_out, const double* dz_out,
                   double eps,
                   double* dq, double* dk, double* dv, double* dS0, double* dz0)
{
    #pragma omp parallel for schedule(dynamic, 1)
    for (int g = 0; g < G; ++g) {
        size_t DD = (size_t)D * D;
        double* S = (double*)malloc(DD * sizeof(double));
        double* z = (double*)malloc((size_t)D * sizeof(double));
        double* dn = (double*)malloc((size_t)C * D * sizeof(double));
        double* dd = (double*)malloc((size_t)C * sizeof(double));
        double* n = (double*)malloc((size_t)D * sizeof(double));
        load_carry(D, g, S0, z0, S, z);
        /* forward in time: rebuild S_t, z_t; emit dq_t; keep dn_t, dd_t */
        for (int t = 0; t < C; ++t) {
            const double* qt = q + IDX3(g, t, 0, C, D);
            const double* kt = k + IDX3(g, t, 0, C, D);
            const double* vt = v + IDX3(g, t, 0, C, D);
            const double* gt = dO + IDX3(g, t, 0, C, D);
            for (int p = 0; p < D; ++p) {
                for (int c = 0; c < D; ++c) S[(size_t)p * D + c] += kt[p] * vt[c];
                z[p] += kt[p];
            }
            double den = 0.0;
            for (int p = 0; p < D; ++p) den += qt[p] * z[p];
            den += eps;
            double gn = 0.0;
            for (int c = 0; c < D; ++c) {
                double acc = 0.0;
                for (int p = 0; p < D; ++p) acc += qt[p] * S[(size_t)p * D + c];
                n[c] = acc;
                gn += gt[c] * acc;
            }
            double ddt = -gn / (den * den);
            dd[t] = ddt;
            for (int c = 0; c < D; ++c) dn[(size_t)t * D + c] = gt[c] / den;
            double* dqt = dq + IDX3(g, t, 0, C, D);
            for (int p = 0; p < D; ++p) {
                double acc = 0.0;
                for (int c = 0; c < D; ++c) acc += S[(size_t)p * D + c] * dn[(size_t)t * D + c];
                dqt[p] = acc + ddt * z[p];
            }
        }
        /* backward in time: suffix sums R, r */
        double* R = S; /* reuse */
        double* r = z;
        if (dS_out) memcpy(R, dS_out + (size_t)g * DD, DD * sizeof(double));
        else memset(R, 0, DD * sizeof(double));
        if (dz_out) memcpy(r, dz_out + (size_t)g * D, (size_t)D * sizeof(double));
        else memset(r, 0, (size_t)D * sizeof(double));
        for (int t = C - 1; t >= 0; --t) {
            const double* qt = q + IDX3(g, t, 0, C, D);
            const double* kt = k + IDX3(g, t, 0, C, D);
            const double* vt = v + IDX3(g, t, 0, C, D);
            const double* dnt = dn + (size_t)t * D;
            for (int p = 0; p < D; ++p) {
                for (int c = 0; c < D; ++c) R[(size_t)p * D + c] += qt[p] * dnt[c];
                r[p] += dd[t] * qt[p];
            }
            double* dkt = dk + IDX3(g, t, 0, C, D);
            double* dvt = dv + IDX3(g, t, 0, C, D);
            for (int p = 0; p < D; ++p) {
                double acc = 0.0;
                for (int c = 0; c < D; ++c) acc += R[(size_t)p * D + c] * vt[c];
                dkt[p] = acc + r[p];
            }
            for (int c = 0; c < D; ++c) {
                double acc = 0.0;
                for (int p = 0; p < D; ++p) acc += R[(size_t)p * D + c] * kt[p];
                dvt[c] = acc;
            }
        }
        if (dS0) memcpy(dS0 + (size_t)g * DD, R, DD * sizeof(double));
        if (dz0) memcpy(dz0 + (size_t)g * D, r, (size_t)D * sizeof(double));
        free(S);
        free(z);
        free(dn);
        free(dd);
        free(n);
    }
}

/*
 * Forward in the page's chunked form ("Opt 2"): blocks of `block` tokens.
 * Inside a block, a masked block x block score matrix A[i][j] = q_i . k_j
 * (kept for j <= i, the diagonal included); across blocks the running state
 * (S_run, z_run) that holds every earlier block.  For row i of the block:
 *   num_i = S_run^T q_i + sum_{j<=i} A[i][j] v_j
 *   den_i = q_i . z_run + sum_{j<=i} A[i][j] + eps
 * Only after all rows of the block have read it does the state absorb the
 * block: S_run += sum_j k_j v_j^T, z_run += sum_j k_j.  The last block may
 * be shorter than `block` (ragged); it is computed the same way.
 */
void la_oracle_fwd_chunked(int G, int C, int D, int block,
                           const double* q, const double* k, const double* v,
                           const double* S0, const double* z0, double eps,
                           double* o, double* S_out, double* z_out)
{
    #pragma omp parallel for schedule(dynamic, 1)
    for (int g = 0; g < G; ++g) {
        double* S = (double*)malloc((size_t)D * D * sizeof(double));
        double* z = (double*)malloc((size_t)D * sizeof(double));
        double* A = (double*)malloc((size_t)block * block * sizeof(double));
        load_carry(D, g, S0, z0, S, z);
        for (int b0 = 0; b0 < C; b0 += block) {
            int L = (C - b0 < block) ? (C - b0) : block;
            for (int i = 0; i < L; ++i) {
                const double* qi = q + IDX3(g, b0 + i, 0, C, D);
                for (int j = 0; j < L; ++j) {
                    double a = 0.0;
                    if (j <= i) {
                        const double* kj = k + IDX3(g, b0 + j, 0, C, D);
                        for (int p = 0; p < D; ++p) a += qi[p] * kj[p];
                    }
                    A[(size_t)i * block + j] = a;
                }
            }
            for (int i = 0; i < L; ++i) {
                const double* qi = q + IDX3(g, b0 + i, 0, C, D);
                double den = 0.0;
                for (int p = 0; p < D; ++p) den += qi[p] * z[p];
                for (int j = 0; j <= i; ++j) den += A[(size_t)i * block + j];
                den += eps;
                double* oi = o + IDX3(g, b0 + i, 0, C, D);
                for (int c = 0; c < D; ++c) {
                    double num = 0.0;
                    for (int p = 0; p < D; ++p) num += qi[p] * S[(size_t)p * D + c];
                    for (int j = 0; j <= i; ++j)
                        num += A[(size_t)i * block + j] * v[IDX3(g, b0 + j, c, C, D)];
                    oi[c] = num / den;
                }
            }
            for (int j = 0; j < L; ++j) {
                const double* kj = k + IDX3(g, b0 + j, 0, C, D);
                const double* vj = v + IDX3(g, b0 + j, 0, C, D);
                for (int p = 0; p < D; ++p) {
                    for (int c = 0; c < D; ++c) S[(size_t)p * D + c] += kj[p] * vj[c];
                    z[p] += kj[p];
                }
            }
        }
        if (S_out) memcpy(S_out + (size_t)g * D * D, S, (size_t)D * D * sizeof(double));
        if (z_out) memcpy(z_out + (size_t)g * D, z, (size_t)D * sizeof(double));
        free(S);
        free(z);
        free(A);
    }
}

/*
 * Backward in the chunked form: the reverse cumsum of la_oracle_bwd taken a
 * block at a time.  A forward sweep over blocks (state before the block:
 * S_run, z_run) gives, with A = masked Q_b K_b^T, P = dO_b V_b^T (same mask)
 * and U = dO_b S_run^T:
 *   den_i = q_i . z_run + sum_{j<=i} A_ij + eps
 *   dd_i  = -(q_i . U_i + sum_{j<=i} A_ij P_ij) / den_i^2
 *   dA_ij = P_ij / den_i + dd_i                  (j <= i, else 0)
 *   dq_i  = U_i / den_i + sum_j dA_ij k_j + dd_i z_run
 * A reverse sweep over blocks with (R, r) = suffix sums of every LATER block
 * (starting from dS_out, dz_out) gives
 *   dk_j = sum_i dA_ij q_i + R v_j + r
 *   dv_j = sum_i A_ij dO_i / den_i + R^T k_j
 * and then R += sum_i q_i dO_i^T / den_i, r += sum_i dd_i q_i.
 */
void la_oracle_bwd_chunked(int G, int C, int D, int block,
                           const double* q, const double* k, const double* v,
                           const double* S0, const double* z0,
                           const double* dO, const double* dS_out, const double* dz_out,
                           double eps,
                           double* dq, double* dk, double* dv, double* dS0, double* dz0)
{
    #pragma omp parallel for schedule(dynamic, 1)
    for (int g = 0; g < G; ++g) {
        size_t DD = (size_t)D * D;
        double* S = (double*)malloc(DD * sizeof(double));
        double* z = (double*)malloc((size_t)D * sizeof(double));
        double* A = (double*)malloc((size_t)block * block * sizeof(double));
        double* dA = (double*)malloc((size_t)block * block * sizeof(double));
        double* U = (double*)malloc((size_t)block * D * sizeof(double));
        double* den = (double*)malloc((size_t)C * sizeof(double));
        double* dd = (double*)malloc((size_t)C * sizeof(double));
        load_carry(D, g, S0, z0, S, z);
        /* forward sweep */
        for (int b0 = 0; b0 < C; b0 += block) {
            int L = (C - b0 < block) ? (C - b0) : block;
            for (int i = 0; i < L; ++i) {
                const double* qi = q + IDX3(g, b0 + i, 0, C, D);
                const double* gi = dO + IDX3(g, b0 + i, 0, C, D);
                double dsum = 0.0, apsum = 0.0, qu = 0.0, qz = 0.0;
                for (int j = 0; j <= i; ++j) {
                    const double* kj = k + IDX3(g, b0 + j, 0, C, D);
                    const double* vj = v + IDX3(g, b0 + j, 0, C, D);
                    double a = 0.0, pp = 0.0;
                    for (int p = 0; p < D; ++p) a += qi[p] * kj[p];
                    for (int c = 0; c < D; ++c) pp += gi[c] * vj[c];
                    A[(size_t)i * block + j] = a;
                    dA[(size_t)i * block + j] = pp; /* P for now */
                    dsum += a;
                    apsum += a * pp;
                }
                for (int p = 0; p < D; ++p) {
                    double u = 0.0;
                    for (int c = 0; c < D; ++c) u += gi[c] * S[(size_t)p * D + c];
                    U[(size_t)i * D + p] = u;
                    qu += qi[p] * u;
                    qz += qi[p] * z[p];
                }
                double dn_ = qz + dsum + eps;
                double ddi = -(qu + apsum) / (dn_ * dn_);
                den[b0 + i] = dn_;
                dd[b0 + i] = ddi;
                for (int j = 0; j <= i; ++j)
                    dA[(size_t)i * block + j] = dA[(size_t)i * block + j] / dn_ + ddi;
                double* dqi = dq + IDX3(g, b0 + i, 0, C, D);
                for (int p = 0; p < D; ++p) {
                    double acc = U[(size_t)i * D + p] / dn_ + ddi * z[p];
                    for (int j = 0; j <= i; ++j)
                        acc += dA[(size_t)i * block + j] * k[IDX3(g, b0 + j, p, C, D)];
                    dqi[p] = acc;
                }
            }
            for (int j = 0; j < L; ++j) {
                const double* kj = k + IDX3(g, b0 + j, 0, C, D);
                const double* vj = v + IDX3(g, b0 + j, 0, C, D);
                for (int p = 0; p < D; ++p) {
                    for (int c = 0; c < D; ++c) S[(size_t)p * D + c] += kj[p] * vj[c];
                    z[p] += kj[p];
                }
            }
        }
        /* reverse sweep */
        double* R = S;
        double* r = z;
        if (dS_out) memcpy(R, dS_out + (size_t)g * DD, DD * sizeof(double));
        else memset(R, 0, DD * sizeof(double));
        if (dz_out) memcpy(r, dz_out + (size_t)g * D, (size_t)D * sizeof(double));
        else memset(r, 0, (size_t)D * sizeof(double));
        int nb = (C + block - 1) / block;
        for (int b = nb - 1; b >= 0; --b) {
            int b0 = b * block;
            int L = (C - b0 < block) ? (C - b0) : block;
            /* rebuild A and dA of this block from the stored den, dd */
            for (int i = 0; i < L; ++i) {
                const double* qi = q + IDX3(g, b0 + i, 0, C, D);
                const double* gi = dO + IDX3(g, b0 + i, 0, C, D);
                for (int j = 0; j <= i; ++j) {
                    const double* kj = k + IDX3(g, b0 + j, 0, C, D);
                    const double* vj = v + IDX3(g, b0 + j, 0, C, D);
                    double a = 0.0, pp = 0.0;
                    for (int p = 0; p < D; ++p) a += qi[p] * kj[p];
                    for (int c = 0; c < D; ++c) pp += gi[c] * vj[c];
                    A[(size_t)i * block + j] = a;
                    dA[(size_t)i * block + j] = pp / den[b0 + i] + dd[b0 + i];
                }
            }
            for (int j = 0; j < L; ++j) {
                const double* kj = k + IDX3(g, b0 + j, 0, C, D);
                const double* vj = v + IDX3(g, b0 + j, 0, C, D);
                double* dkj = dk + IDX3(g, b0 + j, 0, C, D);
                double* dvj = dv + IDX3(g, b0 + j, 0, C, D);
                for (int p = 0; p < D; ++p) {
                    double acc = r[p];
                    for (int c = 0; c < D; ++c) acc += R[(size_t)p * D + c] * vj[c];
                    for (int i = j; i < L; ++i)
                        acc += dA[(size_t)i * block + j] * q[IDX3(g, b0 + i, p, C, D)];
                    dkj[p] = acc;
                }
                for (int c = 0; c < D; ++c) {
                    double acc = 0.0;
                    for (int p = 0; p < D; ++p) acc += R[(size_t)p * D + c] * kj[p];
                    for (int i = j; i < L; ++i)
                        acc += A[(size_t)i * block + j] * dO[IDX3(g, b0 + i, c, C, D)] / den[b0 + i];
                    dvj[c] = acc;
                }
            }
            for (int i = 0; i < L; ++i) {
                const double* qi = q + IDX3(g, b0 + i, 0, C, D);
                const double* gi = dO + IDX3(g, b0 + i, 0, C, D);
                for (int p = 0; p < D; ++p) {
                    for (int c = 0; c < D; ++c) R[(size_t)p * D + c] += qi[p] * gi[c] / den[b0 + i];
                    r[p] += dd[b0 + i] * qi[p];
                }
            }
        }
        if (dS0) memcpy(dS0 + (size_t)g * DD, R, DD * sizeof(double));
        if (dz0) memcpy(dz0 + (size_t)g * D, r, (size_t)D * sizeof(double));
        free(S);
        free(z);
        free(A);
        free(dA);
        free(U);
        free(den);
        free(dd);
    }
}
