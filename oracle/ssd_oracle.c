/*
 * ssd_oracle.c -- plain CPU reference for the Mamba-2 selective state-space
 * recurrence, forward and reverse mode, in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no header, helper or constant with the
 * CUDA library.
 *
 * What it computes (burn-mamba, "Recompute-based gradient math for the
 * Mamba-2 SSD", combined_backward.rs: the K3/K4/K5 formulas unrolled to one
 * token at a time).  For every (batch b, head h), with group g = h / (H/G) and
 * valid length V = valid_len[b] (default L), a state S in R^{P x N} starts at
 * init[b,h] (zero when init is NULL) and for t = 0 .. V-1
 *
 *     a_t   = exp(dt[b,h,t] * A[h])
 *     S     = a_t * S + dt[b,h,t] * x[b,t,h,:] (outer) B[b,t,g,:]
 *     y[b,t,h,p] = sum_r S[p,r] * C[b,t,g,r] + D[h] * x[b,t,h,p]
 *
 * Tokens t >= V are absent: y = 0 there and no state update happens.
 * final_state[b,h] = S after token V-1.
 *
 * The backward is the reverse-mode derivative of exactly that loop for the
 * scalar  Loss = sum dy*y + sum d_final*final_state :
 *
 *     G := d_final (or 0); for t = V-1 .. 0:
 *        G += dy_t (outer) C_t                       (G = dLoss/dS_t)
 *        dC_t[r] += sum_p dy_t[p] S_t[p,r]
 *        dx_t[p]  = D dy_t[p] + dt_t sum_r G[p,r] B_t[r]
 *        dB_t[r] += dt_t sum_p G[p,r] x_t[p]
 *        s_a      = sum_{p,r} G[p,r] S_{t-1}[p,r]
 *        ddt_t    = sum_{p,r} G[p,r] x_t[p] B_t[r] + A a_t s_a
 *        dA      += dt_t a_t s_a ;   dD += sum_p dy_t[p] x_t[p]
 *        G *= a_t
 *     d_init = G.
 *
 * dB and dC sum over the heads of a group; dA and dD sum over batch and time.
 * Gradients at padded tokens (t >= V) are 0.
 *
 * States S_{t-1}, S_t are re-derived in reverse order by checkpointing the
 * state every `seg` tokens and replaying one segment forward at a time, so no
 * full per-token trajectory is held.
 *
 * Layouts (row-major, contiguous): x, y, dx, dy [b, L, H, P]; dt, ddt [b, H, L];
 * A, D, dA, dD [H]; B, C, dB, dC [b, L, G, N]; init, final, d_final, d_init
 * [b, H, P, N]; valid_len int32 [b].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int64_t clamp_len(const int32_t *valid_len, int64_t bi, int64_t L) {
    if (!valid_len) return L;
    int64_t v = valid_len[bi];
    if (v < 0) v = 0;
    if (v > L) v = L;
    return v;
}

static int check_dims(int64_t nb, int64_t L, int64_t H, int64_t P, int64_t N, int64_t G) {
    if (nb < 0 || L < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0) return 1;
    if (H % G != 0) return 1;
    return 0;
}

int ssd_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One token of the recurrence for one (b, h): S <- a S + dt x (outer) B. */
static void step_state(double *S, int64_t P, int64_t N, double a, double dtt,
                       const double *xt, const double *Bt) {
    for (int64_t p = 0; p < P; ++p) {
        double xp = dtt * xt[p];
        double *row = S + p * N;
        for (int64_t r = 0; r < N; ++r) row[r] = a * row[r] + xp * Bt[r];
    }
}

int ssd_oracle_forward(int64_t nb, int64_t L, int64_t H, int64_t P, int64_t N, int64_t G,
                       const double *x, const double *dt, const double *A, const double *Bm,
                       const double *Cm, const double *D, const double *init,
                       const int32_t *valid_len, double *y, double *final_state, int nthreads) {
    if (check_dims(nb, L, H, P, N, G)) return 1;
    const int64_t hpg = H / G;
    const int64_t ntask = nb * H;
    int err = 0;
    if (nthreads <= 0) nthreads = ssd_oracle_num_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t task = 0; task < ntask; ++task) {
        const int64_t bi = task / H, h = task % H, g = h / hpg;
        const int64_t V = clamp_len(valid_len, bi, L);
        double *S = (double *)malloc(sizeof(double) * P * N);
        if (!S) {
#pragma omp atomic write
            err = 2;
            continue;
        }
        if (init)
            memcpy(S, init + (bi * H + h) * P * N, sizeof(double) * P * N);
        else
            memset(S, 0, sizeof(double) * P * N);
        for (int64_t t = 0; t < L; ++t) {
            double *yt = y + ((bi * L + t) * H + h) * P;
            if (t >= V) {
                for (int64_t p = 0; p < P; ++p) yt[p] = 0.0;
                continue;
            }
            const double dtt = dt[(bi * H + h) * L + t];
            const double a = exp(dtt * A[h]);
            const double *xt = x + ((bi * L + t) * H + h) * P;
            const double *Bt = Bm + ((bi * L + t) * G + g) * N;
            const double *Ct = Cm + ((bi * L + t) * G + g) * N;
            step_state(S, P, N, a, dtt, xt, Bt);
            for (int64_t p = 0; p < P; ++p) {
                const double *row = S + p * N;
                double acc = 0.0;
                for (int64_t r = 0; r < N; ++r) acc += row[r] * Ct[r];
                yt[p] = acc + D[h] * xt[p];
            }
        }
        if (final_state) memcpy(final_state + (bi * H + h) * P * N, S, sizeof(double) * P * N);
        free(S);
    }
    return err;
}

int ssd_oracle_backward(int64_t nb, int64_t L, int64_t H, int64_t P, int64_t N, int64_t G,
                        const double *x, const double *dt, const double *A, const double *Bm,
                        const double *Cm, const double *D, const double *init,
                        const int32_t *valid_len, const double *dy, const double *d_final,
                        double *dx, double *ddt, double *dA, double *dB, double *dC, double *dD,
                        double *d_init, int nthreads) {
    if (check_dims(nb, L, H, P, N, G)) return 1;
    const int64_t hpg = H / G;
    const int64_t ntask = nb * H;
    const int64_t PN = P * N;
    int err = 0;
    if (nthreads <= 0) nthreads = ssd_oracle_num_threads();

    memset(dB, 0, sizeof(double) * nb * L * G * N);
    memset(dC, 0, sizeof(double) * nb * L * G * N);
    double *dA_part = (double *)calloc((size_t)(ntask > 0 ? ntask : 1), sizeof(double));
    double *dD_part = (double *)calloc((size_t)(ntask > 0 ? ntask : 1), sizeof(double));
    if (!dA_part || !dD_part) {
        free(dA_part);
        free(dD_part);
        return 2;
    }

#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t task = 0; task < ntask; ++task) {
        const int64_t bi = task / H, h = task % H, g = h / hpg;
        const int64_t V = clamp_len(valid_len, bi, L);
        const double Ah = A[h], Dh = D[h];
        const double *dtrow = dt + (bi * H + h) * L;

        /* padded tokens: every per-token gradient is zero */
        for (int64_t t = V; t < L; ++t) {
            double *dxt = dx + ((bi * L + t) * H + h) * P;
            for (int64_t p = 0; p < P; ++p) dxt[p] = 0.0;
            ddt[(bi * H + h) * L + t] = 0.0;
        }

        /* checkpoint spacing ~ sqrt(V) keeps memory at O(sqrt(V) P N) */
        int64_t seg = (int64_t)ceil(sqrt((double)(V > 0 ? V : 1)));
        if (seg < 1) seg = 1;
        const int64_t nseg = (V + seg - 1) / seg;
        double *ck = (double *)malloc(sizeof(double) * PN * (nseg > 0 ? nseg : 1));
        double *buf = (double *)malloc(sizeof(double) * PN * (seg + 1));
        double *Gs = (double *)malloc(sizeof(double) * PN);
        double *gb = (double *)malloc(sizeof(double) * P); /* sum_r G[p,r] B_t[r] */
        if (!ck || !buf || !Gs || !gb) {
            free(ck);
            free(buf);
            free(Gs);
            free(gb);
#pragma omp atomic write
            err = 2;
            continue;
        }

        /* forward pass, storing the state before every segment start */
        double *S = buf;
        if (init)
            memcpy(S, init + (bi * H + h) * PN, sizeof(double) * PN);
        else
            memset(S, 0, sizeof(double) * PN);
        for (int64_t t = 0; t < V; ++t) {
            if (t % seg == 0) memcpy(ck + (t / seg) * PN, S, sizeof(double) * PN);
            const double dtt = dtrow[t];
            step_state(S, P, N, exp(dtt * Ah), dtt, x + ((bi * L + t) * H + h) * P,
                       Bm + ((bi * L + t) * G + g) * N);
        }

        if (d_final)
            memcpy(Gs, d_final + (bi * H + h) * PN, sizeof(double) * PN);
        else
            memset(Gs, 0, sizeof(double) * PN);
        double dA_acc = 0.0, dD_acc = 0.0;

        for (int64_t k = nseg - 1; k >= 0; --k) {
            const int64_t t0 = k * seg;
            const int64_t t1 = (t0 + seg < V) ? t0 + seg : V;
            /* buf[j] = state after token t0 + j - 1 (buf[0] = state before t0) */
            memcpy(buf, ck + k * PN, sizeof(double) * PN);
            for (int64_t t = t0; t < t1; ++t) {
                double *nxt = buf + (t - t0 + 1) * PN;
                memcpy(nxt, buf + (t - t0) * PN, sizeof(double) * PN);
                const double dtt = dtrow[t];
                step_state(nxt, P, N, exp(dtt * Ah), dtt, x + ((bi * L + t) * H + h) * P,
                           Bm + ((bi * L + t) * G + g) * N);
            }
            for (int64_t t = t1 - 1; t >= t0; --t) {
                const double *Sprev = buf + (t - t0) * PN;
                const double *Scur = buf + (t - t0 + 1) * PN;
                const double dtt = dtrow[t];
                const double a = exp(dtt * Ah);
                const double *xt = x + ((bi * L + t) * H + h) * P;
                const double *dyt = dy + ((bi * L + t) * H + h) * P;
                const double *Bt = Bm + ((bi * L + t) * G + g) * N;
                const double *Ct = Cm + ((bi * L + t) * G + g) * N;
                double *dBt = dB + ((bi * L + t) * G + g) * N;
                double *dCt = dC + ((bi * L + t) * G + g) * N;
                double *dxt = dx + ((bi * L + t) * H + h) * P;

                /* G = dLoss/dS_t: carried part plus this token's output */
                for (int64_t p = 0; p < P; ++p) {
                    double *grow = Gs + p * N;
                    for (int64_t r = 0; r < N; ++r) grow[r] += dyt[p] * Ct[r];
                }
                /* dC_t[r] = sum_p dy[p] S_t[p,r] */
                for (int64_t r = 0; r < N; ++r) {
                    double acc = 0.0;
                    for (int64_t p = 0; p < P; ++p) acc += dyt[p] * Scur[p * N + r];
#pragma omp atomic
                    dCt[r] += acc;
                }
                double s_w = 0.0, s_a = 0.0, dd = 0.0;
                for (int64_t p = 0; p < P; ++p) {
                    const double *grow = Gs + p * N;
                    const double *prow = Sprev + p * N;
                    double accb = 0.0, acca = 0.0;
                    for (int64_t r = 0; r < N; ++r) {
                        accb += grow[r] * Bt[r];
                        acca += grow[r] * prow[r];
                    }
                    gb[p] = accb;
                    s_w += accb * xt[p];
                    s_a += acca;
                    dd += dyt[p] * xt[p];
                }
                for (int64_t p = 0; p < P; ++p) dxt[p] = Dh * dyt[p] + dtt * gb[p];
                for (int64_t r = 0; r < N; ++r) {
                    double acc = 0.0;
                    for (int64_t p = 0; p < P; ++p) acc += Gs[p * N + r] * xt[p];
#pragma omp atomic
                    dBt[r] += dtt * acc;
                }
                ddt[(bi * H + h) * L + t] = s_w + Ah * a * s_a;
                dA_acc += dtt * a * s_a;
                dD_acc += dd;
                for (int64_t i = 0; i < PN; ++i) Gs[i] *= a;
            }
        }
        if (d_init) memcpy(d_init + (bi * H + h) * PN, Gs, sizeof(double) * PN);
        dA_part[task] = dA_acc;
        dD_part[task] = dD_acc;
        free(ck);
        free(buf);
        free(Gs);
        free(gb);
    }
    /* fixed-order reduction over the batch */
    for (int64_t h = 0; h < H; ++h) {
        double sa = 0.0, sd = 0.0;
        for (int64_t bi = 0; bi < nb; ++bi) {
            sa += dA_part[bi * H + h];
            sd += dD_part[bi * H + h];
        }
        dA[h] = sa;
        dD[h] = sd;
    }
    free(dA_part);
    free(dD_part);
    return err;
}

/*
 * Raw moments of the per-token states (burn-mamba, "modules/state_moments.rs",
 * StateMoments: each state row, one (token, p) pair, is a sample in R^N).  For
 * every (b, h), with S_t the state after token t of the recurrence above
 * (t < V = valid_len[b]):
 *
 *     m2[b,h] = sum_t S_t^T S_t            (N x N; the transpose pools the P rows)
 *     m1[b,h] = sum_t sum_p S_t[p, :]      (N)
 *
 * The sample count of a (b, h) slice is V * P.  Layouts: m2 [b, H, N, N],
 * m1 [b, H, N]; the other arguments as ssd_oracle_forward.
 */
int ssd_oracle_state_moments(int64_t nb, int64_t L, int64_t H, int64_t P, int64_t N, int64_t G,
                             const double *x, const double *dt, const double *A, const double *Bm,
                             const double *init, const int32_t *valid_len, double *m2, double *m1,
                             int nthreads) {
    if (check_dims(nb, L, H, P, N, G)) return 1;
    const int64_t hpg = H / G;
    const int64_t ntask = nb * H;
    int err = 0;
    if (nthreads <= 0) nthreads = ssd_oracle_num_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t task = 0; task < ntask; ++task) {
        const int64_t bi = task / H, h = task % H, g = h / hpg;
        const int64_t V = clamp_len(valid_len, bi, L);
        double *S = (double *)malloc(sizeof(double) * P * N);
        if (!S) {
#pragma omp atomic write
            err = 2;
            continue;
        }
        if (init)
            memcpy(S, init + (bi * H + h) * P * N, sizeof(double) * P * N);
        else
            memset(S, 0, sizeof(double) * P * N);
        double *M2 = m2 + task * N * N, *M1 = m1 + task * N;
        memset(M2, 0, sizeof(double) * N * N);
        memset(M1, 0, sizeof(double) * N);
        for (int64_t t = 0; t < V; ++t) {
            const double dtt = dt[(bi * H + h) * L + t];
            step_state(S, P, N, exp(dtt * A[h]), dtt, x + ((bi * L + t) * H + h) * P,
                       Bm + ((bi * L + t) * G + g) * N);
            for (int64_t p = 0; p < P; ++p) {
                const double *row = S + p * N;
                for (int64_t r = 0; r < N; ++r) {
                    M1[r] += row[r];
                    const double v = row[r];
                    double *mr = M2 + r * N;
                    for (int64_t r2 = 0; r2 < N; ++r2) mr[r2] += v * row[r2];
                }
            }
        }
        free(S);
    }
    return err;
}

