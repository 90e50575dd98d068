// ssd_scan.cu -- the chunk-cumsum (K1), state-passing (K4) and reduction kernels,
// forward and backward.  These are HBM/latency-bound streams shared by every
// execution path; they carry fp32 throughout.
//
// burn-mamba, "combined_backward.rs": K1 recompute (dA = dt * A, inclusive
// cumsum per chunk), K4 recurrence s_{i+1} = exp(dA_end_i) s_i + intra_i, the
// "K4 backward step" of the reverse chunk loop, and "SUM GRADIENT
// CONTRIBUTIONS + K1 BACKWARD" (suffix sum, d_dt += d_da * A, dA = sum d_da dt).
#include "ssd_internal.cuh"

namespace ssd {

// ------------------------------------------------------------------ K1 forward
// One warp per (b, h, chunk): inclusive warp-shuffle scan of dt*A over the
// chunk's Q tokens, 32 at a time with a running carry.  Tokens at or past the
// sample's valid length contribute dt = 0.
__global__ void k1_chunk_cumsum(Params p) {
    const int warp = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (warp >= p.b * p.H * p.n) return;
    const int c = warp % p.n, bh = warp / p.n, h = bh % p.H, bi = bh / p.H;
    const int V = valid_len_of(p, bi);
    const float Ah = p.A[h];
    const float *dtrow = p.dt + ix_dt(p, bi, h, 0);
    float *out = p.cumA + (size_t)warp * p.Q;
    float carry = 0.f;
    for (int q0 = 0; q0 < p.Q; q0 += 32) {
        const int q = q0 + lane, t = c * p.Q + q;
        float v = (q < p.Q && t < V) ? dtrow[t] * Ah : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        v += carry;
        if (q < p.Q) out[q] = v;
        carry = __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) p.endA[warp] = carry;
}

cudaError_t launch_k1_cumsum(const Params &p, cudaStream_t s) {
    const long long warps = (long long)p.b * p.H * p.n;
    const int threads = 256;
    const long long blocks = (warps * 32 + threads - 1) / threads;
    k1_chunk_cumsum<<<(unsigned)blocks, threads, 0, s>>>(p);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ K4 forward
// One thread per 4 consecutive (p, r) entries of one (b, h) state.  The chunk
// loop is serial; the chunk-state reads do not depend on the carry, so they
// are issued kUnroll chunks ahead.  The slot holding intra_c is overwritten
// with the chunk-input state s_c (and a bf16 copy when requested).
constexpr int kUnroll = 8;

__device__ __forceinline__ float4 fma4(float a, float4 s, float4 b) {
    return make_float4(fmaf(a, s.x, b.x), fmaf(a, s.y, b.y), fmaf(a, s.z, b.z), fmaf(a, s.w, b.w));
}

__device__ __forceinline__ void store_bf4(bf16 *dst, float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&lo);
    u.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(dst) = u;
}

__global__ void k4_state_passing(Params p, int write_final) {
    const size_t PN = (size_t)p.P * p.N, nvec = PN / 4;
    const size_t gid = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    if (gid >= (size_t)p.b * p.H * nvec) return;
    const size_t e = gid % nvec, bh = gid / nvec;
    const int h = (int)(bh % p.H), bi = (int)(bh / p.H);
    float4 s = p.init ? reinterpret_cast<const float4 *>(p.init)[bh * nvec + e]
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    const float *endA = p.endA + ix_chunk(p, bi, h, 0);
    for (int c0 = 0; c0 < p.n; c0 += kUnroll) {
        float4 in[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (c0 + u < p.n)
                in[u] = reinterpret_cast<const float4 *>(p.states + ix_state(p, bi, c0 + u, h))[e];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int c = c0 + u;
            if (c < p.n) {
                const size_t off = ix_state(p, bi, c, h) + 4 * e;
                *reinterpret_cast<float4 *>(p.states + off) = s;
                if (p.states_bf) store_bf4(p.states_bf + off, s);
                s = fma4(__expf(endA[c]), s, in[u]);
            }
        }
    }
    if (write_final && p.final_state) reinterpret_cast<float4 *>(p.final_state)[bh * nvec + e] = s;
}

cudaError_t launch_k4_state_passing(const Params &p, bool write_final, cudaStream_t s) {
    const long long nthr = (long long)p.b * p.H * ((long long)p.P * p.N / 4);
    const long long blocks = (nthr + kK4Threads - 1) / kK4Threads;
    k4_state_passing<<<(unsigned)blocks, kK4Threads, 0, s>>>(p, write_final ? 1 : 0);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ K4 backward
// Reverse chunk loop over the carried state gradient d (seeded with
// d_final_state):  d_intra_c = d;  d_endA_c = exp(endA_c) * <d, s_c>;
// d <- exp(endA_c) d + d_s_in_c.  Block = kK4Threads threads x 4 entries of one
// (b, h); the per-chunk dot product is reduced in a fixed order inside the
// block and written as one partial per block (summed later by the K1 backward).
__global__ void bwd_k4_state_passing(Params p) {
    __shared__ float red[2][32];
    const size_t PN = (size_t)p.P * p.N, nvec = PN / 4;
    const int nblk = p.k4_nblk;
    const int bh = blockIdx.x / nblk, slab = blockIdx.x % nblk;
    const int h = bh % p.H, bi = bh / p.H;
    const size_t e = (size_t)slab * blockDim.x + threadIdx.x;
    const bool active = e < nvec;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    float4 d = make_float4(0.f, 0.f, 0.f, 0.f);
    if (active && p.d_final) d = reinterpret_cast<const float4 *>(p.d_final)[(size_t)bh * nvec + e];
    const float *endA = p.endA + ix_chunk(p, bi, h, 0);
    for (int c0 = p.n - 1; c0 >= 0; c0 -= kUnroll) {
        float4 dsin[kUnroll], sin_[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int c = c0 - u;
            if (c >= 0 && active) {
                const size_t off = ix_state(p, bi, c, h) + 4 * e;
                dsin[u] = *reinterpret_cast<const float4 *>(p.dstates + off);
                sin_[u] = *reinterpret_cast<const float4 *>(p.states + off);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int c = c0 - u;
            if (c < 0) break;
            const float a = __expf(endA[c]);
            float part = 0.f;
            if (active) {
                const size_t off = ix_state(p, bi, c, h) + 4 * e;
                *reinterpret_cast<float4 *>(p.dstates + off) = d;
                if (p.dstates_bf) store_bf4(p.dstates_bf + off, d);
                part = d.x * sin_[u].x + d.y * sin_[u].y + d.z * sin_[u].z + d.w * sin_[u].w;
                d = fma4(a, d, dsin[u]);
            }
            part = warp_sum(part);
            float *r = red[c & 1];
            if (lane == 0) r[wid] = part;
            __syncthreads();
            if (wid == 0) {
                float v = lane < nw ? r[lane] : 0.f;
                v = warp_sum(v);
                if (lane == 0) p.d_endA_part[ix_chunk(p, bi, h, c) * nblk + slab] = v * a;
            }
        }
    }
    if (active && p.d_init) reinterpret_cast<float4 *>(p.d_init)[(size_t)bh * nvec + e] = d;
}

cudaError_t launch_bwd_k4(const Params &p, cudaStream_t s) {
    const long long blocks = (long long)p.b * p.H * p.k4_nblk;
    bwd_k4_state_passing<<<(unsigned)blocks, kK4Threads, 0, s>>>(p);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ K1 backward
// One warp per (b, h, chunk).  d_cumA = blue + (orange - d_delta) per token,
// plus, at the chunk's last position, the K4 term d_endA and the K3 term
// sum_l d_delta[l].  d_da = suffix sum of d_cumA (reverse warp scan);
// ddt = ddt_main + d_da * A on valid tokens (0 past valid_len); the dA partial
// of the chunk is sum_l d_da[l] * dt_eff[l].
__global__ void bwd_k1_chunk_cumsum(Params p) {
    const int warp = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (warp >= p.b * p.H * p.n) return;
    const int c = warp % p.n, bh = warp / p.n, h = bh % p.H, bi = bh / p.H;
    const int V = valid_len_of(p, bi);
    const float Ah = p.A[h];
    const size_t base = (size_t)warp * p.Q;
    // chunk-end terms
    float endterm = 0.f;
    for (int k = lane; k < p.k4_nblk; k += 32) endterm += p.d_endA_part[(size_t)warp * p.k4_nblk + k];
    for (int q = lane; q < p.Q; q += 32) endterm += p.d_delta[base + q];
    endterm = warp_sum(endterm);
    float carry = 0.f, dA_acc = 0.f;
    const int nseg = (p.Q + 31) / 32;
    for (int sg = nseg - 1; sg >= 0; --sg) {
        const int q = sg * 32 + lane;
        float v = 0.f;
        if (q < p.Q) {
            v = p.dcum_blue[base + q] + p.dcum_main[base + q];
            if (q == p.Q - 1) v += endterm;
        }
        // inclusive suffix scan within the 32 lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_down_sync(0xffffffffu, v, o);
            if (lane + o < 32) v += u;
        }
        v += carry;
        carry = __shfl_sync(0xffffffffu, v, 0);
        const int t = c * p.Q + q;
        if (q < p.Q && t < p.L) {
            const bool valid = t < V;
            const float dtt = valid ? p.dt[ix_dt(p, bi, h, t)] : 0.f;
            p.ddt[ix_dt(p, bi, h, t)] = valid ? p.ddt_main[base + q] + v * Ah : 0.f;
            dA_acc += v * dtt;
        }
    }
    dA_acc = warp_sum(dA_acc);
    if (lane == 0) p.dA_part[warp] = dA_acc;
}

cudaError_t launch_bwd_k1(const Params &p, cudaStream_t s) {
    const long long warps = (long long)p.b * p.H * p.n;
    const int threads = 256;
    bwd_k1_chunk_cumsum<<<(unsigned)((warps * 32 + threads - 1) / threads), threads, 0, s>>>(p);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ dA / dD
// One block per head; fixed-order sums of the per-(b, chunk) partials.
__global__ void bwd_finalize(Params p) {
    __shared__ float red[32];
    const int h = blockIdx.x;
    float a = 0.f, d = 0.f;
    for (int i = threadIdx.x; i < p.b * p.n; i += blockDim.x) {
        const int bi = i / p.n, c = i % p.n;
        a += p.dA_part[ix_chunk(p, bi, h, c)];
        const float *dp = p.dD_part + (((size_t)bi * p.n + c) * p.H + h) * p.dD_per;
        for (int k = 0; k < p.dD_per; ++k) d += dp[k];
    }
    a = block_sum(a, red);
    if (threadIdx.x == 0) p.dA[h] = a;
    d = block_sum(d, red);
    if (threadIdx.x == 0) p.dD[h] = d;
}

cudaError_t launch_bwd_finalize(const Params &p, cudaStream_t s) {
    bwd_finalize<<<p.H, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace ssd
