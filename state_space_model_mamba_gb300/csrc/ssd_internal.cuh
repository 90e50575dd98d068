// ssd_internal.cuh -- shared definitions of the SSD kernels (not part of the ABI).
//
// Index conventions (all row-major):
//   x/y/dy/dx  [b, L, H, P]      B/C/dB/dC  [b, L, G, N]      dt/ddt [b, H, L]
//   cumA, per-token chunk quantities     [b, H, n, Q]   (n = ceil(L / Q))
//   endA                                 [b, H, n]
//   CB (per chunk and group)             [b, n, G, Q, Q]
//   chunk states (intra -> s_in, d_s_in -> d_intra)   [b, n, H, P, N]
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd.h"

namespace ssd {

typedef __nv_bfloat16 bf16;

struct Params {
    // shape
    int b, L, H, P, N, G, Q, n, hpg;
    // leaves
    const void *x;
    const float *dt, *A, *D, *init;
    const void *B, *C;
    const int32_t *valid_len;
    // forward outputs
    void *y;
    float *final_state;
    // backward inputs / outputs
    const void *dy;
    const float *d_final;
    void *dx, *dB, *dC;
    float *ddt, *dA, *dD, *d_init;
    // workspace
    float *cumA, *endA, *CB, *states, *dstates;
    bf16 *CBh;           // bf16 CB  [b, n, G, Q(t), Q(s)] in the CB region (tensor-core path)
    bf16 *CBt;           // bf16 CB^T [b, n, G, Q(s), Q(t)] right after it
    bf16 *states_bf, *dstates_bf;
    float *dcum_blue, *dcum_main, *d_delta, *ddt_main;
    float *d_endA_part;  // [b, H, n, k4_nblk]
    int k4_nblk;
    float *dD_part;      // [b, n, H, dD_per]
    int dD_per;
    float *dA_part;      // [b, H, n]
    float *d_cb;         // [nslice_cb, b, n, G, Q, Q] d_cb (partial sums per head slice)
    int nslice_cb;
    bf16 *d_cb_bf;       // [b, n, G, Q, Q] summed d_cb in bf16 (tensor-core group path)
    int *cb_count;       // [n_count] arrival counters of the d_cb partial blocks
    int *fin_count;      // [H] arrival counters of the K1-backward warps of each head
    int n_count;
    float *dBC_part;     // [nslice, 2, b, n, G, Q, N]  (tensor-core group path)
    int nslice;
    int nslice_k5;       // head slices of the persistent per-group kernels (tensor-core path)
    int nslice_k3;       // head slices of the streaming K3 / BLUE kernels (tensor-core path)
    int *status;         // device status words, kStatusWords ints (below)
    float *mom_A;        // [mom_ranges, b, H, N, N] state-moment partials (A stored transposed)
    float *mom_m1;       // [mom_ranges, b, H, N]
    int mom_ranges;      // chunk ranges per (b, h) of the state-moment kernel
    int cumA_given;      // the chunk-state scan reads cumA / endA (K1 ran before it)
    // time-segmented state passing (few, long (b, h) chains; K4SegGeom below)
    int *k4s_sync;       // ticket counter and ready flags, zeroed by every call with the status words
    float *k4s_agg;      // [pairs, K, kK4Threads * kK4Vec] each segment's state change from zero
    float *k4s_carry;    // [pairs, KG, kK4Threads * kK4Vec] carry into each group's first segment
    float *k4s_dec;      // [pairs, K] each segment's decay (product of its chunks' exp(endA))
};

// The workspace's status words (cleared by every call before its first kernel):
//   [kStatusCode]      SSD_OK, or SSD_ERR_TIMEOUT once a bounded wait gave up
//   [kStatusValidLen]  number of valid_len entries outside [0, seqlen] (clamped)
//   [kStatusNonFinite] non-finite elements seen by the SSD_FLAG_CHECK_FINITE check
constexpr int kStatusCode = 0, kStatusValidLen = 1, kStatusNonFinite = 2, kStatusWords = 4;

// ---------------------------------------------------------------- small helpers
// valid_len[bi] clamped to [0, L] (an entry outside is counted by K1, below).
__device__ __forceinline__ int valid_len_of(const Params &p, int bi) {
    int V = p.L;
    if (p.valid_len) {
        V = p.valid_len[bi];
        V = V < 0 ? 0 : (V > p.L ? p.L : V);
    }
    return V;
}

// True when valid_len[bi] lies outside [0, L] (the kernels then use the clamped value).
__device__ __forceinline__ bool valid_len_out_of_range(const Params &p, int bi) {
    if (!p.valid_len) return false;
    const int V = p.valid_len[bi];
    return V < 0 || V > p.L;
}

__device__ __forceinline__ float ldf(const float *a, size_t i) { return a[i]; }
__device__ __forceinline__ float ldf(const bf16 *a, size_t i) { return __bfloat162float(a[i]); }
__device__ __forceinline__ void stf(float *a, size_t i, float v) { a[i] = v; }
__device__ __forceinline__ void stf(bf16 *a, size_t i, float v) { a[i] = __float2bfloat16_rn(v); }

__device__ __forceinline__ size_t ix_x(const Params &p, int bi, int t, int h, int pp) {
    return ((size_t)((size_t)bi * p.L + t) * p.H + h) * p.P + pp;
}
__device__ __forceinline__ size_t ix_bc(const Params &p, int bi, int t, int g, int r) {
    return ((size_t)((size_t)bi * p.L + t) * p.G + g) * p.N + r;
}
__device__ __forceinline__ size_t ix_dt(const Params &p, int bi, int h, int t) {
    return ((size_t)bi * p.H + h) * p.L + t;
}
__device__ __forceinline__ size_t ix_chunk(const Params &p, int bi, int h, int c) {  // [b,H,n]
    return ((size_t)bi * p.H + h) * p.n + c;
}
__device__ __forceinline__ size_t ix_state(const Params &p, int bi, int c, int h) {  // start of P x N
    return (((size_t)bi * p.n + c) * p.H + h) * (size_t)p.P * p.N;
}
__device__ __forceinline__ size_t ix_cb(const Params &p, int bi, int c, int g) {  // start of Q x Q
    return (((size_t)bi * p.n + c) * p.G + g) * (size_t)p.Q * p.Q;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Fixed-order block sum (deterministic for a fixed blockDim); red has >= 32 floats.
__device__ __forceinline__ float block_sum(float v, float *red) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[wid] = v;
    __syncthreads();
    const int nw = (blockDim.x + 31) >> 5;
    float s = 0.f;
    if (wid == 0) {
        s = lane < nw ? red[lane] : 0.f;
        s = warp_sum(s);
    }
    return s;  // valid in warp 0
}

// Sets the message ssd_last_error() returns on the calling host thread.
void record_error(const char *msg);
// Reads kStatusWords device ints at `words` (synchronising `s`) and turns them
// into the status ssd_workspace_status reports.
ssd_status read_status_words(const void *words, cudaStream_t s);

// ---------------------------------------------------------------- launchers
// Shared by both execution paths (ssd_scan.cu).
cudaError_t launch_k1_cumsum(const Params &p, cudaStream_t s);
cudaError_t launch_k4_state_passing(const Params &p, bool write_final, cudaStream_t s);
cudaError_t launch_bwd_k4(const Params &p, cudaStream_t s);
cudaError_t launch_bwd_k1(const Params &p, cudaStream_t s);

// CUDA-core kernels for the contractions (ssd_simt.cu), T = float or bf16.
template <typename T> cudaError_t launch_simt_k2(const Params &p, cudaStream_t s);
template <typename T> cudaError_t launch_simt_k3(const Params &p, cudaStream_t s);
template <typename T> cudaError_t launch_simt_k5(const Params &p, cudaStream_t s);
template <typename T> cudaError_t launch_simt_bwd_blue(const Params &p, cudaStream_t s);
template <typename T> cudaError_t launch_simt_bwd_main(const Params &p, cudaStream_t s);
template <typename T> cudaError_t launch_simt_bwd_group(const Params &p, cudaStream_t s);

// State moments (ssd_moments.cu): sum of the per-range partials into m2 / m1 /
// count, and the participation ratio of pooled moments.
constexpr int kMomN = 128;  // dstate of the tensor-core state-moment kernel
cudaError_t launch_moments_reduce(const Params &p, float *m2, float *m1, int64_t *count, cudaStream_t s);
cudaError_t launch_state_pr(const float *m2, const float *m1, const int64_t *count, int nb, int H, int N,
                            int center, int pairing, int num, int pool, float *pr, float *trace_out,
                            cudaStream_t s);

// Geometry constants of the CUDA-core kernels that size workspace buffers.
constexpr int kK4Threads = 128;             // threads per block of the state-passing kernels
constexpr int kK4Vec = 16;                   // state entries per thread of the state-passing kernels
constexpr int kMaxQ = 256;                   // largest supported chunk length
constexpr int kMainRows = 16;               // source rows per block of the backward main kernel

// Time-segmented state passing (forward).  With few (b, h) chains the
// chunk-serial K4 grid holds a fraction of the GPU and its speed is set by
// memory latency; the recurrence s_{c+1} = a_c s_c + v_c is linear, so the
// chunks are cut into segments of T, each (chain, slice, segment) ticket
// reduces its segment from a zero state, and the carry into a segment is
// rebuilt from the earlier segments' reductions in one fixed order
// (deterministic results).  Used when the chunk-serial grid has at most
// kK4SegMaxBlocks blocks, P * N fills whole 2048-entry slices and the chains
// have at least two segments.
constexpr int kK4SegGroup = 8;               // segments per group (carry published at each group's start)
constexpr int kK4SegMaxBlocks = 304;         // two 128-thread blocks per SM on a 152-SM GPU
constexpr int kK4SegSyncHead = 64;           // ints before the ready flags: [0] the ticket counter
struct K4SegGeom {
    int on;            // 1: the segmented kernel runs
    int T;             // chunks per segment
    int K;             // segments per chain
    int KG;            // segment groups per chain, ceil(K / kK4SegGroup)
    int slices;        // kK4Threads-thread slices of one (b, h) state
    long long pairs;   // b * H * slices
};
// Geometry of the forward state passing; fp32_states selects the CUDA-core
// path's fp32 chunk states.
K4SegGeom k4_seg_geom(long long b, long long H, long long P, long long N, long long n, bool fp32_states);
// Ints of the sync region (ticket counter, then the ready flags) for these
// dims; 0 when the state passing is not segmented.
size_t k4_seg_sync_ints(long long b, long long H, long long P, long long N, long long n, bool fp32_states);

}  // namespace ssd
