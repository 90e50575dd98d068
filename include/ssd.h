/*
 * ssd.h -- C ABI of the GB300 (sm_103a) Mamba-2 SSD chunked selective scan.
 *
 * The operation (burn-mamba, page "combined_backward.rs" under
 * burn_mamba/mamba2/ssd/serial_recalculated/: the five-kernel chunked scan
 * K1 chunk cumsum of dt*A, K2 C.B^T per chunk, K3 chunk-end states, K4
 * inter-chunk state passing, K5 chunk scan with the D skip; and its
 * recompute-based analytic backward, section "Recompute-based gradient math
 * for the Mamba-2 SSD") is, per batch b and head h with group g = h/(H/G):
 *
 *     S_{-1} = init[b,h];   S_t = exp(dt[b,h,t] * A[h]) * S_{t-1}
 *                                 + dt[b,h,t] * x[b,t,h,:] (outer) B[b,t,g,:]
 *     y[b,t,h,p] = sum_r S_t[p,r] C[b,t,g,r] + D[h] x[b,t,h,p]
 *     final_state[b,h] = S_{V-1}
 *
 * where V = valid_len[b] (default L).  Tokens t >= V are absent: no state
 * update, y = 0, and every per-token gradient there is 0.  ssd_backward
 * returns the gradient of  Loss = <dy, y> + <d_final_state, final_state>
 * with respect to x, dt, A, B, C, D and init, recomputing every forward
 * intermediate from those inputs (nothing is saved between the two calls).
 *
 * Layouts: all tensors are dense, row-major, contiguous.
 *     x, y, dy, dx           [batch, seqlen, nheads, headdim]     (T)
 *     B, C, dB, dC           [batch, seqlen, ngroups, dstate]     (T)
 *     dt, ddt                [batch, nheads, seqlen]              (fp32)
 *     A, D, dA, dD           [nheads]                             (fp32)
 *     init_state, final_state, d_final_state, d_init_state
 *                            [batch, nheads, headdim, dstate]     (fp32)
 *     valid_len              [batch]                              (int32)
 * T is fp32 for SSD_F32 and bf16 for SSD_BF16.  A is the (negative) decay
 * rate used as given; dt is the already-discretised step used as given.
 *
 * Ownership and memory: every pointer is a DEVICE pointer owned by the
 * caller.  Apart from one exception, the library allocates no device memory
 * and keeps no data between calls; scratch lives in the caller's `workspace`,
 * sized by ssd_workspace_bytes().  The exception is ssd_forward_noalloc (end
 * of this file): its scratch is a fixed array of SSD_NOALLOC_SCRATCH_BYTES
 * held on every GPU that loads the library, whose contents outlive each call.
 * Outputs are overwritten, never accumulated into.  Tensor pointers and the
 * workspace must be 16-byte aligned.
 *
 * Streams and errors: work is enqueued on `stream` (a cudaStream_t; NULL is
 * the legacy default stream) and the call returns without synchronising.
 * The tensor-core backward forks part of its kernels onto a second stream
 * that the library creates once per (device, caller stream) pair
 * (non-blocking, with three events, kept until the process exits) and joins
 * it back into `stream` before returning, so to the caller every call is
 * ordered on `stream` as if all its kernels ran there.  Calls that share a
 * caller stream enqueue one at a time (a lock per caller stream); calls on
 * different streams do not wait for each other.
 * Argument errors are detected on the host and returned before anything is
 * enqueued.  Launch failures return SSD_ERR_CUDA.  Three conditions can only be
 * seen on the device; each call clears the start of its workspace (its status
 * words in the first 16 bytes, and, when few long (batch, head) chains take
 * the time-segmented state passing, that pass's ticket counter and ready
 * flags after them) and the kernels record them there, readable with
 * ssd_workspace_status() once the call's work has finished:
 *   - a wait on a shared-memory barrier, or on another block's ready flag,
 *     that gives up after its time limit (SSD_ERR_TIMEOUT; the call's outputs
 *     are then undefined);
 *   - valid_len entries outside [0, seqlen]: such an entry is clamped into the
 *     range, the call completes with the clamped value, and the count of
 *     clamped entries is reported (SSD_ERR_INVALID_ARG);
 *   - with SSD_FLAG_CHECK_FINITE, NaN or infinite values in any output or in
 *     the intermediates the call writes in full (SSD_ERR_NONFINITE).
 */
#ifndef SSD_GB300_H
#define SSD_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1,  /* null required pointer, bad dims, H % G != 0, misalignment */
    SSD_ERR_UNSUPPORTED = 2,  /* shape outside the supported range (see ssd_supported) */
    SSD_ERR_WORKSPACE = 3,    /* workspace smaller than ssd_workspace_bytes() */
    SSD_ERR_CUDA = 4,         /* a CUDA call or kernel launch failed */
    SSD_ERR_TIMEOUT = 5,      /* a bounded device-side wait expired */
    SSD_ERR_NONFINITE = 6     /* SSD_FLAG_CHECK_FINITE found NaN / Inf values */
} ssd_status;

typedef enum {
    SSD_F32 = 0,   /* every tensor fp32; CUDA-core kernels, fp32 arithmetic */
    SSD_BF16 = 1   /* x, B, C, dy, y, dx, dB, dC bf16; fp32 accumulate and state */
} ssd_dtype;

/* Execution-path flags (ssd_dims.flags). */
#define SSD_FLAG_NONE 0u
#define SSD_FLAG_SIMT 1u   /* SSD_BF16 only: use the CUDA-core kernels instead of
                              the tcgen05 tensor-core kernels for the contractions */
#define SSD_FLAG_SPLIT_SCAN 4u     /* tensor-core path: compute the chunk states
                              with the chunk-parallel K3 and a separate K4 pass
                              (the intra-chunk states round-trip through the
                              workspace) even where the fused chunk-state scan,
                              which carries the state on chip along each (b, h)
                              chain, would be chosen; the scan is chosen when
                              batch * nheads >= 64.  Same results up to rounding. */
#define SSD_FLAG_CHECK_FINITE 2u  /* debug: one extra kernel at the end of the call
                              counts NaN / Inf elements of every output and of
                              cumA, endA, the chunk states (and, in the backward,
                              the chunk-state gradients); ssd_workspace_status then
                              returns SSD_ERR_NONFINITE.  The page passes every
                              intermediate of combined_backward through `san`;
                              this flag is that check.  Off: no cost at all. */

typedef struct {
    int64_t batch;      /* b  >= 1 */
    int64_t seqlen;     /* L  >= 1 (need not be a multiple of chunk_len) */
    int64_t nheads;     /* H  >= 1 */
    int64_t headdim;    /* P  (the page's per_head_dim) */
    int64_t dstate;     /* N  (the page's state_rank) */
    int64_t ngroups;    /* G, divides H; B and C are shared by the H/G heads of a group */
    int64_t chunk_len;  /* Q, one of 16, 32, 64, 128, 256 */
    uint32_t flags;     /* SSD_FLAG_* */
    uint32_t reserved;  /* must be 0 */
} ssd_dims;

/* Shape support: returns SSD_OK when (dims, dtype) can run, else
 * SSD_ERR_INVALID_ARG / SSD_ERR_UNSUPPORTED.  Limits: headdim <= 128 and a
 * multiple of 4; dstate <= 256 and a multiple of 4.  The tcgen05 path of
 * SSD_BF16 covers chunk_len in {128, 256}, headdim == 64 and dstate == 128;
 * other SSD_BF16 shapes run on the CUDA-core kernels. */
ssd_status ssd_supported(const ssd_dims *dims, ssd_dtype dtype);

/* Bytes of device workspace ssd_forward (backward = 0) or ssd_backward
 * (backward = 1) needs; 0 when the arguments are invalid. */
size_t ssd_workspace_bytes(const ssd_dims *dims, ssd_dtype dtype, int backward);

/* Forward: y (and optionally final_state).
 * burn-mamba, "combined_backward.rs": the forward intermediates that its
 * "RECOMPUTE FORWARD INTERMEDIATES" block rebuilds (K1 k1_ssd_chunk_cumsum,
 * K2 k2_ssd_bmm, K3 k3_ssd_chunk_state_extended, K4 k4_ssd_state_passing)
 * followed by the chunk scan whose pieces its "BLUE backward" (C times the
 * chunk-input state, scaled by exp(cumA)), "ORANGE backward" (the causal
 * C.B^T decay-weighted sum over earlier tokens, scaled by dt) and "SKIP
 * backward" (D x) blocks differentiate.
 *   init_state   may be NULL (zeros);  valid_len may be NULL (= seqlen);
 *   final_state  may be NULL (not written).
 *   Errors: SSD_ERR_INVALID_ARG / _UNSUPPORTED / _WORKSPACE before any work is
 *   enqueued; SSD_ERR_CUDA if a launch fails (work already enqueued by the
 *   call may then have run).  Device-side conditions: ssd_workspace_status. */
ssd_status ssd_forward(const ssd_dims *dims, ssd_dtype dtype,
                       const void *x, const float *dt, const float *A,
                       const void *B, const void *C, const float *D,
                       const float *init_state, const int32_t *valid_len,
                       void *y, float *final_state,
                       void *workspace, size_t workspace_bytes, void *stream);

/* Backward with recompute: gradients of <dy,y> + <d_final_state,final_state>.
 * burn-mamba, "combined_backward.rs": the function combined_backward(d_y,
 * d_final, x, dt, b, c, d, initial_state, a_decay) and its result struct
 * CombinedGrads, whose fields d_x, d_dt, d_b, d_c, d_d, d_initial_state and
 * d_a_decay are the outputs dx, ddt, dB, dC, dD, d_init_state and dA here
 * (B and C per group instead of per head: their gradients are summed over the
 * group's heads).  Like the page, it saves nothing from the forward: every
 * intermediate is recomputed from the leaves.
 *   d_final_state may be NULL (zeros);  d_init_state may be NULL (not written).
 *   dA and dD are reduced over batch and time in a fixed order (deterministic).
 *   Errors: as ssd_forward. */
ssd_status ssd_backward(const ssd_dims *dims, ssd_dtype dtype,
                        const void *x, const float *dt, const float *A,
                        const void *B, const void *C, const float *D,
                        const float *init_state, const int32_t *valid_len,
                        const void *dy, const float *d_final_state,
                        void *dx, float *ddt, float *dA, void *dB, void *dC, float *dD,
                        float *d_init_state,
                        void *workspace, size_t workspace_bytes, void *stream);

/* Reads (synchronously, on `stream`) the status words that the last call on
 * this workspace left and returns, in this order of precedence:
 * SSD_ERR_TIMEOUT, SSD_ERR_NONFINITE (with the count in ssd_last_error()),
 * SSD_ERR_INVALID_ARG for clamped valid_len entries (count in
 * ssd_last_error()), else SSD_OK.  workspace_bytes must be >= 16. */
ssd_status ssd_workspace_status(const void *workspace, size_t workspace_bytes, void *stream);

/* ---- Diagnostics (no counterpart on the pages; used by the benchmark) ----
 *
 * ssd_last_launch_count: number of kernels the most recent ssd_forward /
 * ssd_backward call on the calling host thread enqueued.
 *
 * ssd_profile_begin / ssd_profile_end: while active on the calling host
 * thread, every kernel the library enqueues is bracketed by two
 * cudaEventRecord calls on the call's stream, taken in order from `events`
 * (an array of `capacity` cudaEvent_t created by the caller); recording stops
 * silently when the array is full.  ssd_profile_end deactivates it and
 * returns how many events were recorded (2 per kernel); ssd_profile_name(i)
 * names the i-th recorded kernel (i < 4096).  Timing events add no device
 * work besides the records themselves.  While every kernel is recorded (no
 * ssd_profile_only filter), the kernels the library otherwise runs on its
 * second stream beside the caller's chain (K2, and the backward's d_cb and
 * dB/dC kernels) run on the call's stream instead, so that each event pair
 * brackets one kernel running alone; with a filter the schedule is unchanged
 * and a second-stream kernel's pair is recorded on that stream, spanning any
 * overlap with the caller's chain.
 *
 * ssd_profile_only: restricts the recording to kernels whose name (as
 * ssd_profile_name reports it) equals `name`; NULL or "" records every
 * kernel again.  The string is copied (at most 63 characters).  Applies to
 * the calling host thread until changed. */
int ssd_last_launch_count(void);
ssd_status ssd_profile_begin(void **events, int capacity);
int ssd_profile_end(void);
const char *ssd_profile_name(int i);
void ssd_profile_only(const char *name);

/* ---- Forward without any device allocation (no counterpart on the pages) ----
 *
 * For callers that cannot call cudaMalloc themselves or have it called for
 * them: code whose device memory is owned by an arena or pool it may not
 * grow, plug-ins whose host framework forbids allocation on the hot path,
 * and code running while another component captures or replays work.
 * ssd_forward_noalloc computes exactly what ssd_forward computes, with the
 * same arguments minus the workspace: its scratch is a fixed array of
 * SSD_NOALLOC_SCRATCH_BYTES bytes in this library's device memory, created
 * on every GPU that loads the library and held until the process exits.
 *
 *  - Size limit: shapes whose forward workspace (ssd_workspace_bytes(dims,
 *    dtype, 0)) exceeds SSD_NOALLOC_SCRATCH_BYTES are rejected with
 *    SSD_ERR_UNSUPPORTED and a message in ssd_last_error(); nothing is
 *    enqueued.
 *  - First call per device: it looks up the array's device address for the
 *    current device (cudaGetSymbolAddress, which may load the library's code
 *    onto that device).  Make that first call before any stream capture.  The
 *    address is kept per CUDA context: after a device reset (a new primary
 *    context) the next call looks it up again, and is again a first call.
 *  - Status: the call's status words (see the file header) live at the start
 *    of the array; read them with ssd_noalloc_status() on the same device.
 *  - Sharing: every call on a device uses the same array and leaves its
 *    contents behind; the call clears what must start at zero itself.  Calls
 *    whose GPU work overlaps (different streams, or different host threads
 *    without ordering) race on the array and give wrong results: serialise
 *    them on one stream.
 *  - It calls no cudaMalloc, cudaFree or allocating library routine. */
#define SSD_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
ssd_status ssd_forward_noalloc(const ssd_dims *dims, ssd_dtype dtype,
                               const void *x, const float *dt, const float *A,
                               const void *B, const void *C, const float *D,
                               const float *init_state, const int32_t *valid_len,
                               void *y, float *final_state, void *stream);

/* Status of the last ssd_forward_noalloc call on the current device, as
 * ssd_workspace_status() reports it for a workspace (synchronises `stream`;
 * allocates nothing).  SSD_ERR_INVALID_ARG with "no call yet" in
 * ssd_last_error() if the array has not been used on this device. */
ssd_status ssd_noalloc_status(void *stream);

/* Self-test of the device-side timeout path (no counterpart on the pages).
 * Every wait of the library's kernels is a bounded wait on a shared-memory
 * barrier that gives up after 2 s and records SSD_ERR_TIMEOUT in the call's
 * status words.  This call runs that same wait in a one-thread kernel, on a
 * barrier that one arrival completes (arrive = 1) or that nothing completes
 * (arrive = 0), with a limit of limit_us microseconds (1 <= limit_us <=
 * 2,000,000), after clearing the workspace's status words.  With arrive = 0
 * the wait runs out, the kernel records the timeout and returns, the stream
 * and context stay usable, and ssd_workspace_status then returns
 * SSD_ERR_TIMEOUT; with arrive = 1 it returns SSD_OK.  The kernel holds no
 * copies or tensor memory, so giving up leaves nothing in flight.
 *   workspace: device memory, workspace_bytes >= 16 (only the status words are
 *   written);  stream: cudaStream_t or NULL.
 *   Errors: SSD_ERR_INVALID_ARG (before any work) for a bad workspace, limit
 *   or arrive; SSD_ERR_CUDA if the launch fails. */
ssd_status ssd_wait_selftest(void *workspace, size_t workspace_bytes, uint32_t limit_us, int arrive,
                             void *stream);

/* Static description of a status code. */
const char *ssd_status_str(ssd_status status);

/* Detail of the most recent failure on the calling host thread ("" if none). */
const char *ssd_last_error(void);

/* ABI version (major * 10000 + minor * 100 + patch). */
int ssd_version(void);

/* ---------------------------------------------------------------- state moments
 * Raw first and second moments of every per-token state of the forward
 * (burn-mamba, "modules/state_moments.rs": StateMoments, produced in closed
 * form for Mamba-2 by Mamba2SsdInput::state_moments).  Each state row -- one
 * (token, p) pair of S_t in R^{P x N}, S_t the state after token t < valid_len
 * -- is one sample in R^N:
 *   m2[b, h] = sum_t S_t^T S_t      [b, H, N, N] fp32
 *   m1[b, h] = sum_t sum_p S_t[p,:] [b, H, N] fp32
 *   count[b] = valid_len[b] * P     int64 (device), or NULL
 * Computed without forming any per-token state: the chunk-input states are
 * recomputed from the leaves (x, dt, A, B, init; C and D do not enter) at
 * chunk 128 whatever dims->chunk_len says, then each 128-token chunk adds
 * c0 s^T s + U^T D B + B^T D U + B^T (K o G) B (see the kernel) by three
 * tensor-core products.  SSD_BF16 with headdim 64 and dstate 128 only
 * (SSD_ERR_UNSUPPORTED otherwise).  Workspace from ssd_moments_workspace_bytes;
 * m2, m1 overwritten; status words as ssd_forward's (ssd_workspace_status). */
size_t ssd_moments_workspace_bytes(const ssd_dims *dims, ssd_dtype dtype);
ssd_status ssd_state_moments(const ssd_dims *dims, ssd_dtype dtype, const void *x, const float *dt,
                             const float *A, const void *B, const float *init_state,
                             const int32_t *valid_len, float *m2, float *m1, int64_t *count,
                             void *workspace, size_t workspace_bytes, void *stream);

/* Participation ratio of pooled state moments (StateMoments::pr / ::pr_complex
 * / ::trace): per (b, h), Sigma = m2 / n, minus mu mu^T with mu = m1 / n when
 * `center`; PR = tr(Sigma)^2 / tr(Sigma^2) evaluated, as the page does, on
 * Sigma / max(tr Sigma, FLT_MIN) with the denominator floored at 1e-12.  With a
 * complex or quaternionic `pairing` the state axis is read as realified
 * coordinates and tr(Sigma^2) is that of the Hermitian moment (one complex or
 * quaternion direction counts once; unrotated coordinates join as a real
 * block).  `pool_batch` first sums m2, m1 and count over the batch (the page's
 * pool_batch); outputs are then [1, H].  trace[b, h] = tr(m2) / n (the raw mean
 * squared state magnitude), or NULL.  All pointers are device pointers;
 * N = dstate <= 224; num = complex pairs or quaternion blocks (ignored for
 * SSD_PAIR_REAL).  PR of a slice with no samples is not defined (NaN/Inf). */
#define SSD_PAIR_REAL 0
#define SSD_PAIR_COMPLEX_INTERLEAVED 1  /* coordinate 2a real, 2a+1 imaginary part of pair a */
#define SSD_PAIR_COMPLEX_HALF_HALF 2    /* coordinate a real, N/2 + a imaginary part of pair a */
#define SSD_PAIR_QUATERNION 3           /* coordinates 4j .. 4j+3: quaternion block j (w, x, y, z) */
ssd_status ssd_state_pr(const float *m2, const float *m1, const int64_t *count, int64_t batch,
                        int64_t nheads, int64_t dstate, int center, int pairing, int64_t num,
                        int pool_batch, float *pr, float *trace, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* SSD_GB300_H */
