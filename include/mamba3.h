/* mamba3.h -- C ABI of the two Mamba-3 pieces on the burn-mamba pages, built
 * beside the Mamba-2 SSD scan in the same library (libssd.so, ssd.h):
 *
 *   - the quaternion cumulative-product scan of the rotated states and its
 *     recompute backward (burn-mamba, "mamba3/quat_scan/backward.rs",
 *     module doc "Gradient math");
 *   - the same-step gamma correction y_diag and its analytic backward, MIMO
 *     and the SISO fast path (burn-mamba,
 *     "mamba3/single_ssd/ssd/serial_recalculated/diag.rs").
 *
 * Conventions as in ssd.h: plain device pointers, row-major contiguous
 * tensors, caller-owned memory (the library allocates nothing; the scan takes
 * a caller workspace sized by m3_quat_workspace_bytes), work enqueued on
 * `stream` (a cudaStream_t, NULL = the legacy default stream) without
 * synchronising.  Argument errors return before any launch; ssd_last_error()
 * describes the last failure. */
#ifndef MAMBA3_H
#define MAMBA3_H

#include <stddef.h>
#include <stdint.h>

#include "ssd.h"

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- quaternion scan
 * Quaternions are 4 fp32 components (w, x, y, z), the order of the pages'
 * QuaternionBlocks; products are Hamilton products.
 *   q     [b, L, H, J, 4]  per-step quaternions (the page's q_bshj4)
 *   init  [b, H, J, 4]     carry before step 0, or NULL for the identity (1, 0, 0, 0)
 *   cum   [b, L, H, J, 4]  cum[t] = q[t] (x) cum[t-1], cum[-1] = init
 * Every pointer 16-byte aligned.  Errors: SSD_ERR_INVALID_ARG (NULL or
 * misaligned pointer, a dimension < 1), SSD_ERR_WORKSPACE, SSD_ERR_CUDA. */
size_t m3_quat_workspace_bytes(int64_t b, int64_t L, int64_t H, int64_t J, int backward);

ssd_status m3_quat_cumprod(const float *q, const float *init, float *cum, int64_t b, int64_t L, int64_t H,
                           int64_t J, void *workspace, size_t workspace_bytes, void *stream);

/* Backward of m3_quat_cumprod for the upstream cotangent d_cum [b, L, H, J, 4]
 * (which already holds the final carry's gradient at the last step), the
 * page's closed form, exact for unit quaternions (the rotation always
 * produces them): with the prefix product P[t] = q[t] (x) ... (x) q[0],
 *   S[t] = sum_{s >= t} conj(P[s]) (x) d_cum[s],  G[t] = P[t] (x) S[t],
 *   d_q[t] = G[t] (x) conj(cum[t-1])  (cum[-1] = init),   d_init = S[0].
 * Only the leaves q and init are read; the prefix products are recomputed.
 *   d_q [b, L, H, J, 4] (overwritten);  d_init [b, H, J, 4] or NULL (not written). */
ssd_status m3_quat_cumprod_backward(const float *q, const float *init, const float *d_cum, float *d_q,
                                    float *d_init, int64_t b, int64_t L, int64_t H, int64_t J, void *workspace,
                                    size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------- gamma correction
 * Per token t (the page's (b, n, l) axes flattened into T tokens) and head h:
 *   qk[o, i]   = sum_r C[t, o, h, r] B[t, i, h, r]          (o, i < m, the MIMO rank)
 *   y[t, o, h, p] = gamma[t, h] sum_i qk[o, i] V[t, i, h, p]
 *   V, y [T, m, H, P];  B, C [T, m, H, N];  gamma [T, H] fp32.
 * dtype SSD_F32: V, B, C, y fp32; SSD_BF16: V, B, C, y bf16 (fp32 arithmetic).
 * m = 1 is the page's SISO fast path (one scalar qk).  Limits: 1 <= m <= 4,
 * P and N even; every pointer 16-byte aligned.  Errors as above
 * (SSD_ERR_UNSUPPORTED for m > 4 or odd P / N). */
ssd_status m3_y_diag(ssd_dtype dtype, const void *V, const void *B, const void *C, const float *gamma, void *y,
                     int64_t T, int64_t m, int64_t H, int64_t P, int64_t N, void *stream);

/* Backward of m3_y_diag for dY [T, m, H, P] (the page's DiagGrads): with
 * e = gamma dY,  d_gamma[t, h] = sum_{o, p} dY (qk V),  dV = qk^T e,
 * d_qk = e V^T,  dC = d_qk B,  dB = d_qk^T C.  dV, dB, dC in the dtype of V,
 * d_gamma fp32 [T, H]; all overwritten. */
ssd_status m3_y_diag_backward(ssd_dtype dtype, const void *dY, const void *V, const void *B, const void *C,
                              const float *gamma, void *dV, void *dB, void *dC, float *d_gamma, int64_t T,
                              int64_t m, int64_t H, int64_t P, int64_t N, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA3_H */
