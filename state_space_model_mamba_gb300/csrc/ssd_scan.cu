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
// chunk's Q tokens, 32 at a time with a running carry.  All of the warp's loads
// are issued before the first scan step (Q <= 256: at most 8 per lane), so
// their latencies overlap.  Tokens at or past the sample's valid length
// contribute dt = 0; a valid_len entry outside [0, L] is clamped and counted
// in the status words.  (The grid has b*H*n*32 >= n_count threads, so the
// counter clear needs no extra launch.)
__global__ void k1_chunk_cumsum(Params p) {
    const size_t gid = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    // the backward's first kernel also clears the arrival counters
    if (p.cb_count && gid < (size_t)p.n_count) p.cb_count[gid] = 0;
    if (p.fin_count && gid < (size_t)p.H) p.fin_count[gid] = 0;
    const int warp = (int)(gid >> 5);
    const int lane = threadIdx.x & 31;
    if (warp >= p.b * p.H * p.n) return;
    const int c = warp % p.n, bh = warp / p.n, h = bh % p.H, bi = bh / p.H;
    const int V = valid_len_of(p, bi);
    // one warp per sample reports a valid_len entry outside [0, L] (it is clamped)
    if (h == 0 && c == 0 && lane == 0 && valid_len_out_of_range(p, bi))
        atomicAdd(p.status + kStatusValidLen, 1);
    const float Ah = p.A[h];
    const float *dtrow = p.dt + ix_dt(p, bi, h, 0);
    float *out = p.cumA + (size_t)warp * p.Q;
    float v[kMaxQ / 32];
#pragma unroll
    for (int sg = 0; sg < kMaxQ / 32; ++sg) {
        const int q = sg * 32 + lane, t = c * p.Q + q;
        v[sg] = (q < p.Q && t < V) ? dtrow[t] * Ah : 0.f;
    }
    float carry = 0.f;
#pragma unroll
    for (int sg = 0; sg < kMaxQ / 32; ++sg) {
        if (sg * 32 >= p.Q) break;
        float u = v[sg];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float w = __shfl_up_sync(0xffffffffu, u, o);
            if (lane >= o) u += w;
        }
        u += carry;
        if (sg * 32 + lane < p.Q) out[sg * 32 + lane] = u;
        carry = __shfl_sync(0xffffffffu, u, 31);
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
// One thread per 16 consecutive (p, r) entries of one (b, h) state, 128-thread
// blocks, sized so that the whole grid is resident at once: the chain over
// chunks is serial, so a second wave would double the kernel's time.  The
// chunk-state reads do not depend on the carry; they are issued a fixed number
// of chunks ahead (the forward refills a slot as soon as it is consumed) and
// held packed (8 registers per 16 bf16) until used.  The slot
// holding intra_c is overwritten with the chunk-input state s_c.  The carry is
// fp32; the stored states are S (fp32 on the CUDA-core path, bf16 on the
// tensor-core path, whose every consumer reads bf16 operands).
constexpr int kVec = kK4Vec;

template <typename S>
struct Packed;
template <>
struct Packed<bf16> {
    uint4 u[2];
};
template <>
struct Packed<float> {
    float4 u[4];
};

__device__ __forceinline__ Packed<bf16> load16(const bf16 *src) {
    const uint4 *q = reinterpret_cast<const uint4 *>(src);
    return Packed<bf16>{{q[0], q[1]}};
}
__device__ __forceinline__ Packed<float> load16(const float *src) {
    const float4 *q = reinterpret_cast<const float4 *>(src);
    return Packed<float>{{q[0], q[1], q[2], q[3]}};
}
__device__ __forceinline__ void unpack16(const Packed<bf16> &x, float *v) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint32_t w[4] = {x.u[j].x, x.u[j].y, x.u[j].z, x.u[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[8 * j + 2 * i] = __uint_as_float(w[i] << 16);
            v[8 * j + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
}
__device__ __forceinline__ void unpack16(const Packed<float> &x, float *v) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        v[4 * j] = x.u[j].x;
        v[4 * j + 1] = x.u[j].y;
        v[4 * j + 2] = x.u[j].z;
        v[4 * j + 3] = x.u[j].w;
    }
}
__device__ __forceinline__ void store16(float *dst, const float *v) {
    float4 *q = reinterpret_cast<float4 *>(dst);
#pragma unroll
    for (int j = 0; j < 4; ++j) q[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}
__device__ __forceinline__ void store16(bf16 *dst, const float *v) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        __nv_bfloat162 t = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t *>(&t);
    }
    uint4 *q = reinterpret_cast<uint4 *>(dst);
    q[0] = make_uint4(w[0], w[1], w[2], w[3]);
    q[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// Chunks read ahead (U): bounded by registers, since the grid must stay one
// wave.  A grid of at most one block per SM (few (b, h) chains: the 131k-token
// workload has 32, 128 blocks) takes a deep read-ahead and the registers it
// needs; larger grids keep five blocks per SM and a short one.  MB: the blocks
// per SM the launch bounds promise.
constexpr int k4_min_blocks(int U, int bytes) { return U * bytes >= 32 ? 1 : (U * bytes >= 16 ? 2 : 5); }

template <typename S, int U>
__global__ void __launch_bounds__(kK4Threads, k4_min_blocks(U, sizeof(S)))
    k4_state_passing(Params p, S *st, int write_final) {
    const size_t PN = (size_t)p.P * p.N, nvec = PN / kVec;
    const size_t gid = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    if (gid >= (size_t)p.b * p.H * nvec) return;
    const size_t e = gid % nvec, bh = gid / nvec;
    const int h = (int)(bh % p.H), bi = (int)(bh / p.H);
    float s[kVec];
    if (p.init) unpack16(load16(p.init + bh * PN + kVec * e), s);
    else {
#pragma unroll
        for (int i = 0; i < kVec; ++i) s[i] = 0.f;
    }
    const float *endA = p.endA + ix_chunk(p, bi, h, 0);
    // rolling read-ahead: slot u holds chunk c (c % U == u) and is refilled with
    // chunk c + U as soon as it is consumed, so U chunk loads stay in flight
    Packed<S> in[U];
    float ea[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (u < p.n) {
            in[u] = load16(st + ix_state(p, bi, u, h) + kVec * e);
            ea[u] = endA[u];
        }
    for (int c0 = 0; c0 < p.n; c0 += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + u;
            if (c < p.n) {
                const Packed<S> cur = in[u];
                const float a = __expf(ea[u]);
                if (c + U < p.n) {
                    in[u] = load16(st + ix_state(p, bi, c + U, h) + kVec * e);
                    ea[u] = endA[c + U];
                }
                store16(st + ix_state(p, bi, c, h) + kVec * e, s);
                float v[kVec];
                unpack16(cur, v);
#pragma unroll
                for (int i = 0; i < kVec; ++i) s[i] = fmaf(a, s[i], v[i]);
            }
        }
    }
    if (write_final && p.final_state) store16(p.final_state + bh * PN + kVec * e, s);
}

// blocks per SM of a K4 grid on this device (1: at most one block on every SM)
static int k4_per_sm(long long blocks) {
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return (int)((blocks + sms - 1) / sms);
}

cudaError_t launch_k4_state_passing(const Params &p, bool write_final, cudaStream_t s) {
    const long long nthr = (long long)p.b * p.H * ((long long)p.P * p.N / kVec);
    const long long blocks = (nthr + kK4Threads - 1) / kK4Threads;
    const int per_sm = k4_per_sm(blocks), wf = write_final ? 1 : 0;
    const unsigned g = (unsigned)blocks;
    if (p.states) {  // fp32 states: 16 registers per chunk read ahead
        if (per_sm <= 1) k4_state_passing<float, 8><<<g, kK4Threads, 0, s>>>(p, p.states, wf);
        else if (per_sm <= 2) k4_state_passing<float, 4><<<g, kK4Threads, 0, s>>>(p, p.states, wf);
        else k4_state_passing<float, 2><<<g, kK4Threads, 0, s>>>(p, p.states, wf);
    } else {         // bf16 states: 8 registers per chunk
        if (per_sm <= 1) k4_state_passing<bf16, 16><<<g, kK4Threads, 0, s>>>(p, p.states_bf, wf);
        else if (per_sm <= 2) k4_state_passing<bf16, 8><<<g, kK4Threads, 0, s>>>(p, p.states_bf, wf);
        else k4_state_passing<bf16, 4><<<g, kK4Threads, 0, s>>>(p, p.states_bf, wf);
    }
    return cudaGetLastError();
}

// ------------------------------------------------------------------ K4 backward
// Reverse chunk loop over the carried state gradient d (seeded with
// d_final_state):  d_intra_c = d;  d_endA_c = exp(endA_c) * <d, s_c>;
// d <- exp(endA_c) d + d_s_in_c.  One thread per 16 entries of one (b, h),
// laid out as in the forward; the per-chunk dot product is reduced inside
// each warp and written as one partial per warp (k4_nblk partials per
// (b, h, chunk), summed in a fixed order by the K1 backward), so the chunk
// loop has no block barrier.  `dst` holds d_s_in on entry and d_intra on
// exit; `st` holds s_in.
template <typename S, int U, int MB>
__global__ void __launch_bounds__(kK4Threads, MB) bwd_k4_state_passing(Params p, S *dst, const S *st) {
    const size_t PN = (size_t)p.P * p.N, nvec = PN / kVec;
    const int nblk = (int)((nvec + kK4Threads - 1) / kK4Threads);
    const int bh = blockIdx.x / nblk, slab = blockIdx.x % nblk;
    const int h = bh % p.H, bi = bh / p.H;
    const size_t e = (size_t)slab * blockDim.x + threadIdx.x;
    const bool active = e < nvec;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int part_idx = slab * (kK4Threads / 32) + wid;  // < k4_nblk
    float d[kVec];
    if (active && p.d_final) unpack16(load16(p.d_final + (size_t)bh * PN + kVec * e), d);
    else {
#pragma unroll
        for (int i = 0; i < kVec; ++i) d[i] = 0.f;
    }
    const float *endA = p.endA + ix_chunk(p, bi, h, 0);
    for (int c0 = p.n - 1; c0 >= 0; c0 -= U) {
        Packed<S> dsin[U], sin_[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 - u;
            if (c >= 0 && active) {
                const size_t off = ix_state(p, bi, c, h) + kVec * e;
                dsin[u] = load16(dst + off);
                sin_[u] = load16(st + off);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 - u;
            if (c < 0) break;
            const float a = __expf(endA[c]);
            float part = 0.f;
            if (active) {
                store16(dst + ix_state(p, bi, c, h) + kVec * e, d);
                float sv[kVec], dv[kVec];
                unpack16(sin_[u], sv);
                unpack16(dsin[u], dv);
#pragma unroll
                for (int i = 0; i < kVec; ++i) {
                    part = fmaf(d[i], sv[i], part);
                    d[i] = fmaf(a, d[i], dv[i]);
                }
            }
            part = warp_sum(part);
            if (lane == 0) p.d_endA_part[ix_chunk(p, bi, h, c) * p.k4_nblk + part_idx] = part * a;
        }
    }
    if (active && p.d_init) store16(p.d_init + (size_t)bh * PN + kVec * e, d);
}

cudaError_t launch_bwd_k4(const Params &p, cudaStream_t s) {
    const long long nvec = (long long)p.P * p.N / kVec;
    const long long blocks = (long long)p.b * p.H * ((nvec + kK4Threads - 1) / kK4Threads);
    const int per_sm = k4_per_sm(blocks);
    const unsigned g = (unsigned)blocks;
    // two chunks (d_s_in and s_in) per step read ahead; one block per SM: deep, else five per SM
    if (p.dstates) {
        if (per_sm <= 1) bwd_k4_state_passing<float, 4, 1><<<g, kK4Threads, 0, s>>>(p, p.dstates, p.states);
        else bwd_k4_state_passing<float, 2, 5><<<g, kK4Threads, 0, s>>>(p, p.dstates, p.states);
    } else {
        if (per_sm <= 1) bwd_k4_state_passing<bf16, 8, 1><<<g, kK4Threads, 0, s>>>(p, p.dstates_bf, p.states_bf);
        else bwd_k4_state_passing<bf16, 4, 5><<<g, kK4Threads, 0, s>>>(p, p.dstates_bf, p.states_bf);
    }
    return cudaGetLastError();
}

// ------------------------------------------------------------------ K1 backward
// One warp per (b, h, chunk).  d_cumA = blue + (orange - d_delta) per token,
// plus, at the chunk's last position, the K4 term d_endA and the K3 term
// sum_l d_delta[l].  d_da = suffix sum of d_cumA (reverse warp scan);
// ddt = ddt_main + d_da * A on valid tokens (0 past valid_len); the dA partial
// of the chunk is sum_l d_da[l] * dt_eff[l].  The last warp of a head to finish
// reduces the head's dA and dD partials (fixed order).
__global__ void bwd_k1_chunk_cumsum(Params p) {
    const int warp = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (warp >= p.b * p.H * p.n) return;
    const int c = warp % p.n, bh = warp / p.n, h = bh % p.H, bi = bh / p.H;
    const int V = valid_len_of(p, bi);
    const float Ah = p.A[h];
    const size_t base = (size_t)warp * p.Q;
    constexpr int NS = kMaxQ / 32;
    // every load of the warp first (at most 8 tokens per lane), then the scans
    float v[NS], dtt[NS], ddm[NS];
    float endterm = 0.f;
#pragma unroll
    for (int sg = 0; sg < NS; ++sg) {
        const int q = sg * 32 + lane, t = c * p.Q + q;
        const bool in = q < p.Q;
        v[sg] = in ? p.dcum_blue[base + q] + p.dcum_main[base + q] : 0.f;
        endterm += in ? p.d_delta[base + q] : 0.f;
        const bool valid = in && t < V;
        dtt[sg] = valid ? p.dt[ix_dt(p, bi, h, t)] : 0.f;
        ddm[sg] = valid ? p.ddt_main[base + q] : 0.f;
    }
    // chunk-end terms: the K4 partials and the K3 sum of d_delta
    for (int k = lane; k < p.k4_nblk; k += 32) endterm += p.d_endA_part[(size_t)warp * p.k4_nblk + k];
    endterm = warp_sum(endterm);
    float carry = 0.f, dA_acc = 0.f;
#pragma unroll
    for (int sg = NS - 1; sg >= 0; --sg) {
        if (sg * 32 >= p.Q) continue;
        const int q = sg * 32 + lane;
        float u = v[sg];
        if (q == p.Q - 1) u += endterm;
        // inclusive suffix scan within the 32 lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float w = __shfl_down_sync(0xffffffffu, u, o);
            if (lane + o < 32) u += w;
        }
        u += carry;
        carry = __shfl_sync(0xffffffffu, u, 0);
        const int t = c * p.Q + q;
        if (q < p.Q && t < p.L) {
            const bool valid = t < V;
            p.ddt[ix_dt(p, bi, h, t)] = valid ? ddm[sg] + u * Ah : 0.f;
            dA_acc += u * dtt[sg];
        }
    }
    dA_acc = warp_sum(dA_acc);
    // dA[h], dD[h]: the last warp of head h to finish sums the head's partials
    // (its b * n dA partials, and the dD partials the ORANGE kernel wrote) in a
    // fixed order, so the result does not depend on which warp that is
    int last = 0;
    if (lane == 0) {
        p.dA_part[warp] = dA_acc;
        __threadfence();
        last = atomicAdd(p.fin_count + h, 1) == p.b * p.n - 1;
    }
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    __threadfence();
    float a = 0.f, d = 0.f;
    for (int i = lane; i < p.b * p.n; i += 32) {
        const int bb = i / p.n, cc = i % p.n;
        a += __ldcg(p.dA_part + ix_chunk(p, bb, h, cc));
        const float *dp = p.dD_part + (((size_t)bb * p.n + cc) * p.H + h) * p.dD_per;
        for (int k = 0; k < p.dD_per; ++k) d += __ldcg(dp + k);
    }
    a = warp_sum(a);
    d = warp_sum(d);
    if (lane == 0) {
        p.dA[h] = a;
        p.dD[h] = d;
        p.fin_count[h] = 0;  // ready for the next call
    }
}

cudaError_t launch_bwd_k1(const Params &p, cudaStream_t s) {
    const long long warps = (long long)p.b * p.H * p.n;
    const int threads = 256;
    bwd_k1_chunk_cumsum<<<(unsigned)((warps * 32 + threads - 1) / threads), threads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace ssd
