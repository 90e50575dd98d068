// ssd_moments.cu -- the CUDA-core kernels around the state-moment path
// (burn-mamba, "modules/state_moments.rs"): the fixed-order sum of the
// tensor-core kernel's per-range partials into m2, m1 and the sample counts,
// and the participation ratio (StateMoments::pr, ::pr_complex, ::trace).
#include <float.h>

#include "ssd_internal.cuh"

namespace ssd {
namespace {

// m2[bh][r][r'] = sum over ranges of (A[r][r'] + A[r'][r]) / 2, in range order;
// m1[bh][r] likewise; count[b] = valid tokens * P.
__global__ void moments_reduce(const float *__restrict__ A, const float *__restrict__ M1, int ranges, int bh_count,
                               int N, float *__restrict__ m2, float *__restrict__ m1, int64_t *__restrict__ count,
                               const int32_t *__restrict__ valid_len, int nb, int L, int P) {
    const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    const long long NN = (long long)N * N, tot = (long long)bh_count * NN;
    if (i < tot) {
        const long long bh = i / NN, rr = i % NN, r = rr / N, q = rr % N;
        float s = 0.f;
        for (int k = 0; k < ranges; ++k) {
            const float *a = A + ((long long)k * bh_count + bh) * NN;
            s += 0.5f * (a[r * N + q] + a[q * N + r]);
        }
        m2[i] = s;
    }
    if (i < (long long)bh_count * N && m1) {
        float s = 0.f;
        for (int k = 0; k < ranges; ++k) s += M1[(long long)k * bh_count * N + i];
        m1[i] = s;
    }
    if (i < nb && count) {
        int V = L;
        if (valid_len) {
            V = valid_len[i];
            V = V < 0 ? 0 : (V > L ? L : V);
        }
        count[i] = (int64_t)V * P;
    }
}

__device__ __forceinline__ float block_sum_f(float v, float *red) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[wid] = v;
    __syncthreads();
    float s = 0.f;
    if (wid == 0) {
        s = lane < nw ? red[lane] : 0.f;
        s = warp_sum(s);
        if (lane == 0) red[32] = s;
    }
    __syncthreads();
    return red[32];
}

// One block per (b or pooled, h).  Sigma = m2 / n (- mu mu^T when centred), its
// trace normalised away (floored at the smallest fp32 normal), and
// PR = tr(Sigma^)^2 / max(tr(Sigma^2 of the pairing's Hermitian form), 1e-12).
// Coordinates: `perm` maps the canonical order [x-pairs | y-pairs | real] (or
// quaternion blocks then real) to the state index.
__global__ void state_pr_kernel(const float *__restrict__ m2, const float *__restrict__ m1,
                                const int64_t *__restrict__ count, int nb, int H, int N, int center, int pairing,
                                int num, int pool, float *__restrict__ pr, float *__restrict__ trace_out) {
    extern __shared__ float sh[];  // Sigma [N][N] (canonical order), mu [N]
    __shared__ float red[33];
    __shared__ int perm[256];
    float *S = sh, *mu = sh + N * N;
    const int ob = blockIdx.x / H, h = blockIdx.x % H;  // output (batch or pooled), head
    const int b0 = pool ? 0 : ob, b1 = pool ? nb : ob + 1;
    double n = 0.0;
    for (int b = b0; b < b1; ++b) n += (double)count[b];
    const float inv = n > 0.0 ? (float)(1.0 / n) : 0.f;
    // canonical coordinate order
    if (threadIdx.x == 0) {
        int k = 0;
        if (pairing == 1) {  // interleaved complex pairs
            for (int a = 0; a < num; ++a) perm[k++] = 2 * a;
            for (int a = 0; a < num; ++a) perm[k++] = 2 * a + 1;
            for (int r = 2 * num; r < N; ++r) perm[k++] = r;
        } else if (pairing == 2) {  // half-and-half complex pairs
            const int half = N / 2;
            for (int a = 0; a < num; ++a) perm[k++] = a;
            for (int a = 0; a < num; ++a) perm[k++] = half + a;
            for (int r = num; r < half; ++r) perm[k++] = r;
            for (int r = half + num; r < N; ++r) perm[k++] = r;
        } else {
            for (int r = 0; r < N; ++r) perm[k++] = r;
        }
    }
    for (int r = threadIdx.x; r < N; r += blockDim.x) {
        float s = 0.f;
        for (int b = b0; b < b1; ++b) s += m1[((long long)b * H + h) * N + r];
        mu[r] = s * inv;
    }
    __syncthreads();
    float tr_raw = 0.f;
    for (int e = threadIdx.x; e < N * N; e += blockDim.x) {
        const int i = e / N, j = e % N, pi = perm[i], pj = perm[j];
        float s = 0.f;
        for (int b = b0; b < b1; ++b) s += m2[(((long long)b * H + h) * N + pi) * N + pj];
        if (i == j) tr_raw += s;
        float v = s * inv;
        if (center) v -= mu[pi] * mu[pj];
        S[e] = v;
    }
    tr_raw = block_sum_f(tr_raw, red);
    float tr = 0.f;
    for (int i = threadIdx.x; i < N; i += blockDim.x) tr += S[i * N + i];
    tr = block_sum_f(tr, red);
    const float scale = fmaxf(tr, FLT_MIN), is = 1.f / scale;
    const float tr1 = tr * is;
    float sq = 0.f;
    const int rot = pairing == 1 || pairing == 2 ? 2 * num : (pairing == 3 ? 4 * num : 0);
    if (pairing == 0) {
        for (int e = threadIdx.x; e < N * N; e += blockDim.x) {
            const float v = S[e] * is;
            sq += v * v;
        }
    } else {
        if (pairing == 3) {
            for (int e = threadIdx.x; e < num * num; e += blockDim.x) {
                const int jj = e / num, kk = e % num;
                auto c = [&](int a, int b) { return S[(4 * jj + a) * N + 4 * kk + b] * is; };
                const float w = c(0, 0) + c(1, 1) + c(2, 2) + c(3, 3);
                const float x = c(0, 1) - c(1, 0) - c(2, 3) + c(3, 2);
                const float y = c(0, 2) + c(1, 3) - c(2, 0) - c(3, 1);
                const float z = c(0, 3) - c(1, 2) + c(2, 1) - c(3, 0);
                sq += w * w + x * x + y * y + z * z;
            }
        } else {
            for (int e = threadIdx.x; e < num * num; e += blockDim.x) {
                const int a = e / num, b = e % num;
                const float A_ = (S[a * N + b] + S[(num + a) * N + num + b]) * is;
                const float S_ = (S[a * N + num + b] - S[b * N + num + a]) * is;
                sq += A_ * A_ + S_ * S_;
            }
        }
        // the real tail: twice the cross block, once the tail block
        for (int e = threadIdx.x; e < N * N; e += blockDim.x) {
            const int i = e / N, j = e % N;
            if (j < rot) continue;
            const float v = S[e] * is;
            if (i < rot) sq += 2.f * v * v;
            else sq += v * v;
        }
    }
    sq = block_sum_f(sq, red);
    if (threadIdx.x == 0) {
        const int o = ob * H + h;
        pr[o] = tr1 * tr1 / fmaxf(sq, 1e-12f);
        if (trace_out) trace_out[o] = tr_raw * inv;
    }
}

}  // namespace

cudaError_t launch_moments_reduce(const Params &p, float *m2, float *m1, int64_t *count, cudaStream_t s) {
    const long long tot = (long long)p.b * p.H * kMomN * kMomN;
    const unsigned grid = (unsigned)((tot + 255) / 256);
    moments_reduce<<<grid, 256, 0, s>>>(p.mom_A, p.mom_m1, p.mom_ranges, p.b * p.H, kMomN, m2, m1, count,
                                         p.valid_len, p.b, p.L, p.P);
    return cudaGetLastError();
}

cudaError_t launch_state_pr(const float *m2, const float *m1, const int64_t *count, int nb, int H, int N,
                            int center, int pairing, int num, int pool, float *pr, float *trace_out,
                            cudaStream_t s) {
    const size_t smem = sizeof(float) * ((size_t)N * N + N);
    cudaError_t e = cudaFuncSetAttribute(state_pr_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)((pool ? 1 : nb) * H);
    state_pr_kernel<<<grid, 256, smem, s>>>(m2, m1, count, nb, H, N, center, pairing, num, pool, pr, trace_out);
    return cudaGetLastError();
}

}  // namespace ssd
