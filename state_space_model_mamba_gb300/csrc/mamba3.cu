// mamba3.cu -- the Mamba-3 pieces of include/mamba3.h: the quaternion
// cumulative-product scan with its closed-form recompute backward (burn-mamba,
// "mamba3/quat_scan/backward.rs", "Gradient math") and the same-step gamma
// correction with its backward (burn-mamba,
// "mamba3/single_ssd/ssd/serial_recalculated/diag.rs").  Both are HBM-bound
// streams: coalesced 16-byte (quaternion) or pair loads, fp32 arithmetic.
//
// Quaternion scan.  A chain is one (b, h, j); its L steps are cut into
// segments of kSeg steps so that b * L / kSeg * H * J threads share the work.
//   forward:  pass 1, per segment: the product of its steps;
//             carries, one warp per chain: the carry into each segment (init
//             times the earlier segments' products, in order) by a warp scan
//             whose combine is the ordered product, written over pass 1's
//             products;
//             pass 2, per segment: its steps from that carry.
//   backward: pass 1, per segment: the local prefix products LP (from the
//             identity at the segment start), their product, and
//             T = sum_s conj(LP[s]) (x) d_cum[s];
//             carries, one warp per chain: P_in (product of the earlier
//             segments) and the suffix sum over the later segments
//             sum_{later} conj(P_in') (x) T';
//             pass 2, per segment: one forward walk in which
//             S[t] = suffix + conj(P_in) (x) (T - running sum of the segment's
//             terms before t) -- the page's reverse cumsum without a reverse
//             walk -- and G, d_q as on the page.
#include <cuda_bf16.h>
#include <stdio.h>

#include "mamba3.h"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kSeg = 32;  // steps per segment of the quaternion scan

struct Qt {
    float w, x, y, z;
};
__device__ __forceinline__ Qt qmul(Qt a, Qt b) {
    return {a.w * b.w - a.x * b.x - a.y * b.y - a.z * b.z, a.w * b.x + a.x * b.w + a.y * b.z - a.z * b.y,
            a.w * b.y - a.x * b.z + a.y * b.w + a.z * b.x, a.w * b.z + a.x * b.y - a.y * b.x + a.z * b.w};
}
__device__ __forceinline__ Qt qconj(Qt a) { return {a.w, -a.x, -a.y, -a.z}; }
__device__ __forceinline__ Qt qadd(Qt a, Qt b) { return {a.w + b.w, a.x + b.x, a.y + b.y, a.z + b.z}; }
__device__ __forceinline__ Qt qsub(Qt a, Qt b) { return {a.w - b.w, a.x - b.x, a.y - b.y, a.z - b.z}; }
__device__ __forceinline__ Qt qld(const float *p) {
    const float4 v = __ldg(reinterpret_cast<const float4 *>(p));
    return {v.x, v.y, v.z, v.w};
}
__device__ __forceinline__ void qst(float *p, Qt a) { *reinterpret_cast<float4 *>(p) = make_float4(a.w, a.x, a.y, a.z); }
__device__ __forceinline__ Qt qld_rw(const float *p) {  // plain load: data this kernel also writes
    const float4 v = *reinterpret_cast<const float4 *>(p);
    return {v.x, v.y, v.z, v.w};
}
__device__ __forceinline__ Qt qshfl_up(Qt a, int o) {
    return {__shfl_up_sync(0xffffffffu, a.w, o), __shfl_up_sync(0xffffffffu, a.x, o),
            __shfl_up_sync(0xffffffffu, a.y, o), __shfl_up_sync(0xffffffffu, a.z, o)};
}
__device__ __forceinline__ Qt qshfl_down(Qt a, int o) {
    return {__shfl_down_sync(0xffffffffu, a.w, o), __shfl_down_sync(0xffffffffu, a.x, o),
            __shfl_down_sync(0xffffffffu, a.y, o), __shfl_down_sync(0xffffffffu, a.z, o)};
}
__device__ __forceinline__ Qt qone() { return {1.f, 0.f, 0.f, 0.f}; }
__device__ __forceinline__ Qt qzero() { return {0.f, 0.f, 0.f, 0.f}; }

struct QShape {
    long long b, L, C, S;  // C = H * J chains per sample, S segments
};

// thread -> (sample, segment, chain), the chain fastest (coalesced 16-byte accesses)
__device__ __forceinline__ bool qmap(const QShape &s, long long &bi, long long &sg, long long &c) {
    const long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (idx >= s.b * s.S * s.C) return false;
    c = idx % s.C;
    sg = (idx / s.C) % s.S;
    bi = idx / (s.C * s.S);
    return true;
}

__global__ void quat_seg_product(const float *__restrict__ q, float *__restrict__ segp, QShape s) {
    long long bi, sg, c;
    if (!qmap(s, bi, sg, c)) return;
    const long long t0 = sg * kSeg, t1 = min(s.L, t0 + kSeg);
    const float *qp = q + ((bi * s.L + t0) * s.C + c) * 4;
    Qt acc = qone();
#pragma unroll 8
    for (long long t = t0; t < t1; ++t, qp += s.C * 4) acc = qmul(qld(qp), acc);
    qst(segp + ((bi * s.S + sg) * s.C + c) * 4, acc);
}

// One warp per chain (b, c): lane l takes segments [l K, l K + K), K = ceil(S / 32).
// The product of a lane's segments, a warp scan in lane order (later (x) earlier),
// then a walk that overwrites each segment's product with the carry into it.
// The segments are read in batches of kCB into registers, every load of a batch
// before any store; a lane with one batch (K <= kCB) reads them once.
constexpr int kCB = 8;

__global__ void quat_seg_carry(float *__restrict__ segp, const float *__restrict__ init, QShape s) {
    const long long wid = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= s.b * s.C) return;  // warp-uniform
    const long long c = wid % s.C, bi = wid / s.C;
    const long long K = (s.S + 31) / 32, k0 = lane * K, k1 = min(s.S, k0 + K);
    auto at = [&](long long k) { return ((bi * s.S + k) * s.C + c) * 4; };
    Qt v[kCB];
    Qt a = qone();
    for (long long kb = k0; kb < k1; kb += kCB) {
#pragma unroll
        for (int i = 0; i < kCB; ++i) v[i] = kb + i < k1 ? qld_rw(segp + at(kb + i)) : qone();
#pragma unroll
        for (int i = 0; i < kCB; ++i) a = qmul(v[i], a);
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const Qt y = qshfl_up(a, o);
        if (lane >= o) a = qmul(a, y);
    }
    Qt run = qshfl_up(a, 1);  // the earlier lanes' segments
    if (lane == 0) run = qone();
    const Qt in = init ? qld(init + (bi * s.C + c) * 4) : qone();
    const bool reuse = k1 - k0 <= kCB;
    for (long long kb = k0; kb < k1; kb += kCB) {
        if (!reuse) {
#pragma unroll
            for (int i = 0; i < kCB; ++i) v[i] = kb + i < k1 ? qld_rw(segp + at(kb + i)) : qone();
        }
#pragma unroll
        for (int i = 0; i < kCB; ++i) {
            if (kb + i < k1) qst(segp + at(kb + i), qmul(run, in));
            run = qmul(v[i], run);
        }
    }
}

__global__ void quat_seg_scan(const float *__restrict__ q, const float *__restrict__ carries,
                              float *__restrict__ cum, QShape s) {
    long long bi, sg, c;
    if (!qmap(s, bi, sg, c)) return;
    Qt carry = qld(carries + ((bi * s.S + sg) * s.C + c) * 4);
    const long long t0 = sg * kSeg, t1 = min(s.L, t0 + kSeg);
    const long long off = ((bi * s.L + t0) * s.C + c) * 4;
    const float *qp = q + off;
    float *cp = cum + off;
#pragma unroll 8
    for (long long t = t0; t < t1; ++t, qp += s.C * 4, cp += s.C * 4) {
        carry = qmul(qld(qp), carry);
        qst(cp, carry);
    }
}

__global__ void quat_bwd_segments(const float *__restrict__ q, const float *__restrict__ d_cum,
                                  float *__restrict__ segp, float *__restrict__ segT, QShape s) {
    long long bi, sg, c;
    if (!qmap(s, bi, sg, c)) return;
    const long long t0 = sg * kSeg, t1 = min(s.L, t0 + kSeg);
    const long long off = ((bi * s.L + t0) * s.C + c) * 4;
    const float *qp = q + off, *dp = d_cum + off;
    Qt lp = qone(), acc = qzero();
#pragma unroll 4
    for (long long t = t0; t < t1; ++t, qp += s.C * 4, dp += s.C * 4) {
        lp = qmul(qld(qp), lp);
        acc = qadd(acc, qmul(qconj(lp), qld(dp)));
    }
    const long long so = ((bi * s.S + sg) * s.C + c) * 4;
    qst(segp + so, lp);
    qst(segT + so, acc);
}

// One warp per chain, lanes over segments as in quat_seg_carry: segp's products
// become P_in[k] (the product of segments 0 .. k-1, without init), and
// later[k] = sum_{k' > k} conj(P_in[k']) (x) T[k'] (a suffix sum over lanes, then
// a reverse walk over the lane's own segments).  A lane with one batch of
// segments holds its products, P_in and T in registers throughout.
__global__ void quat_bwd_carry(float *__restrict__ segp, const float *__restrict__ segT, float *__restrict__ later,
                               QShape s) {
    const long long wid = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= s.b * s.C) return;  // warp-uniform
    const long long c = wid % s.C, bi = wid / s.C;
    const long long K = (s.S + 31) / 32, k0 = lane * K, k1 = min(s.S, k0 + K);
    auto at = [&](long long k) { return ((bi * s.S + k) * s.C + c) * 4; };
    const bool reuse = k1 - k0 <= kCB;
    Qt v[kCB], tv[kCB], pin[kCB];
    Qt a = qone();
    for (long long kb = k0; kb < k1; kb += kCB) {
#pragma unroll
        for (int i = 0; i < kCB; ++i) {
            v[i] = kb + i < k1 ? qld_rw(segp + at(kb + i)) : qone();
            tv[i] = kb + i < k1 ? qld(segT + at(kb + i)) : qzero();
        }
#pragma unroll
        for (int i = 0; i < kCB; ++i) a = qmul(v[i], a);
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const Qt y = qshfl_up(a, o);
        if (lane >= o) a = qmul(a, y);
    }
    Qt run = qshfl_up(a, 1);
    if (lane == 0) run = qone();
    Qt u = qzero();  // sum over the lane's segments of conj(P_in) (x) T
    for (long long kb = k0; kb < k1; kb += kCB) {
        if (!reuse) {
#pragma unroll
            for (int i = 0; i < kCB; ++i) {
                v[i] = kb + i < k1 ? qld_rw(segp + at(kb + i)) : qone();
                tv[i] = kb + i < k1 ? qld(segT + at(kb + i)) : qzero();
            }
        }
#pragma unroll
        for (int i = 0; i < kCB; ++i) {
            pin[i] = run;
            if (kb + i < k1) qst(segp + at(kb + i), run);
            u = qadd(u, qmul(qconj(run), tv[i]));
            run = qmul(v[i], run);
        }
    }
    Qt r = u;  // inclusive suffix sum over lanes, then exclusive
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const Qt y = qshfl_down(r, o);
        if (lane + o < 32) r = qadd(r, y);
    }
    r = qsub(r, u);
    // the lane's segments in reverse, batch by batch from the last
    const long long nb = (k1 - k0 + kCB - 1) / kCB;
    for (long long bb = nb - 1; bb >= 0; --bb) {
        const long long kb = k0 + bb * kCB;
        if (!reuse) {
#pragma unroll
            for (int i = 0; i < kCB; ++i) {
                pin[i] = kb + i < k1 ? qld_rw(segp + at(kb + i)) : qone();
                tv[i] = kb + i < k1 ? qld(segT + at(kb + i)) : qzero();
            }
        }
#pragma unroll
        for (int i = kCB - 1; i >= 0; --i) {
            if (kb + i < k1) {
                qst(later + at(kb + i), r);
                r = qadd(r, qmul(qconj(pin[i]), tv[i]));
            }
        }
    }
}

__global__ void quat_bwd_apply(const float *__restrict__ q, const float *__restrict__ init,
                               const float *__restrict__ d_cum, const float *__restrict__ p_ins,
                               const float *__restrict__ segT, const float *__restrict__ laters,
                               float *__restrict__ d_q, float *__restrict__ d_init, QShape s) {
    long long bi, sg, c;
    if (!qmap(s, bi, sg, c)) return;
    const long long so = ((bi * s.S + sg) * s.C + c) * 4;
    const Qt p_in = qld(p_ins + so), later = qld(laters + so), own = qld(segT + so);
    const Qt in = init ? qld(init + (bi * s.C + c) * 4) : qone();
    const Qt cin = qconj(p_in);
    const long long t0 = sg * kSeg, t1 = min(s.L, t0 + kSeg);
    const long long off = ((bi * s.L + t0) * s.C + c) * 4;
    const float *qp = q + off, *dp = d_cum + off;
    float *gp = d_q + off;
    Qt lp = qone(), run = qzero(), p_prev = p_in;
#pragma unroll 4
    for (long long t = t0; t < t1; ++t, qp += s.C * 4, dp += s.C * 4, gp += s.C * 4) {
        const Qt S_t = qadd(later, qmul(cin, qsub(own, run)));  // sum_{s >= t} conj(P[s]) (x) d_cum[s]
        lp = qmul(qld(qp), lp);
        const Qt P_t = qmul(lp, p_in);
        const Qt G = qmul(P_t, S_t);
        qst(gp, qmul(G, qconj(qmul(p_prev, in))));  // cum[t-1] = P[t-1] (x) init
        run = qadd(run, qmul(qconj(lp), qld(dp)));
        if (t == 0 && d_init) qst(d_init + (bi * s.C + c) * 4, S_t);
        p_prev = P_t;
    }
}

// ---------------------------------------------------------------- gamma correction
template <typename T>
struct Pair;
template <>
struct Pair<float> {
    static __device__ __forceinline__ float2 ld(const float *p) { return __ldg(reinterpret_cast<const float2 *>(p)); }
    static __device__ __forceinline__ void st(float *p, float2 v) { *reinterpret_cast<float2 *>(p) = v; }
    static __device__ __forceinline__ float4 ld4(const float *p) { return __ldg(reinterpret_cast<const float4 *>(p)); }
    static __device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
};
template <>
struct Pair<bf16> {
    static __device__ __forceinline__ float2 ld(const bf16 *p) {
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
    }
    static __device__ __forceinline__ void st(bf16 *p, float2 v) {
        *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(v.x, v.y);
    }
    static __device__ __forceinline__ float4 ld4(const bf16 *p) {
        const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
        return make_float4(a.x, a.y, b.x, b.y);
    }
    static __device__ __forceinline__ void st4(bf16 *p, float4 v) {
        __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t *>(&a);
        u.y = *reinterpret_cast<uint32_t *>(&b);
        *reinterpret_cast<uint2 *>(p) = u;
    }
};
__device__ __forceinline__ float dot4(float4 a, float4 b) { return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w; }

struct DShape {
    long long T;
    int H, P, N;
};

// one warp per (token, head); lanes take pairs of the state / head axis, the
// m x m products are reduced across the warp
template <typename T, int M>
__device__ __forceinline__ void qk_of(const T *C, const T *B, const DShape &s, long long t, int h, int lane,
                                      float (&qk)[M][M]) {
#pragma unroll
    for (int o = 0; o < M; ++o)
#pragma unroll
        for (int i = 0; i < M; ++i) qk[o][i] = 0.f;
    if ((s.N & 3) == 0) {  // 8- or 16-byte loads: four elements per lane
        for (int e = 4 * lane; e < s.N; e += 128) {
            float4 cv[M], bv[M];
#pragma unroll
            for (int i = 0; i < M; ++i) {
                const long long row = ((t * M + i) * s.H + h) * (long long)s.N + e;
                cv[i] = Pair<T>::ld4(C + row);
                bv[i] = Pair<T>::ld4(B + row);
            }
#pragma unroll
            for (int o = 0; o < M; ++o)
#pragma unroll
                for (int i = 0; i < M; ++i) qk[o][i] += dot4(cv[o], bv[i]);
        }
    } else {
        for (int e = 2 * lane; e < s.N; e += 64) {
            float2 cv[M], bv[M];
#pragma unroll
            for (int i = 0; i < M; ++i) {
                const long long row = ((t * M + i) * s.H + h) * (long long)s.N + e;
                cv[i] = Pair<T>::ld(C + row);
                bv[i] = Pair<T>::ld(B + row);
            }
#pragma unroll
            for (int o = 0; o < M; ++o)
#pragma unroll
                for (int i = 0; i < M; ++i) qk[o][i] += cv[o].x * bv[i].x + cv[o].y * bv[i].y;
        }
    }
#pragma unroll
    for (int o = 0; o < M; ++o)
#pragma unroll
        for (int i = 0; i < M; ++i) qk[o][i] = warp_sum(qk[o][i]);
}

template <typename T, int M>
__global__ void y_diag_fwd(const T *__restrict__ V, const T *__restrict__ B, const T *__restrict__ C,
                           const float *__restrict__ gamma, T *__restrict__ y, DShape s) {
    const long long w = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= s.T * s.H) return;
    const int h = (int)(w % s.H);
    const long long t = w / s.H;
    float qk[M][M];
    qk_of<T, M>(C, B, s, t, h, lane, qk);
    const float g = gamma[w];
    for (int e = 2 * lane; e < s.P; e += 64) {
        float2 vv[M];
#pragma unroll
        for (int i = 0; i < M; ++i) vv[i] = Pair<T>::ld(V + ((t * M + i) * s.H + h) * (long long)s.P + e);
#pragma unroll
        for (int o = 0; o < M; ++o) {
            float2 a = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < M; ++i) {
                a.x += qk[o][i] * vv[i].x;
                a.y += qk[o][i] * vv[i].y;
            }
            Pair<T>::st(y + ((t * M + o) * s.H + h) * (long long)s.P + e, make_float2(g * a.x, g * a.y));
        }
    }
}

template <typename T, int M>
__global__ void y_diag_bwd(const T *__restrict__ dY, const T *__restrict__ V, const T *__restrict__ B,
                           const T *__restrict__ C, const float *__restrict__ gamma, T *__restrict__ dV,
                           T *__restrict__ dB, T *__restrict__ dC, float *__restrict__ d_gamma, DShape s) {
    const long long w = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= s.T * s.H) return;
    const int h = (int)(w % s.H);
    const long long t = w / s.H;
    float qk[M][M], dyv[M][M];
    qk_of<T, M>(C, B, s, t, h, lane, qk);
    // dyv[o, i] = sum_p dY[o, p] V[i, p]
#pragma unroll
    for (int o = 0; o < M; ++o)
#pragma unroll
        for (int i = 0; i < M; ++i) dyv[o][i] = 0.f;
    for (int e = 2 * lane; e < s.P; e += 64) {
        float2 dv[M], vv[M];
#pragma unroll
        for (int i = 0; i < M; ++i) {
            const long long row = ((t * M + i) * s.H + h) * (long long)s.P + e;
            dv[i] = Pair<T>::ld(dY + row);
            vv[i] = Pair<T>::ld(V + row);
        }
#pragma unroll
        for (int o = 0; o < M; ++o)
#pragma unroll
            for (int i = 0; i < M; ++i) dyv[o][i] += dv[o].x * vv[i].x + dv[o].y * vv[i].y;
    }
    float dg = 0.f;
#pragma unroll
    for (int o = 0; o < M; ++o)
#pragma unroll
        for (int i = 0; i < M; ++i) {
            dyv[o][i] = warp_sum(dyv[o][i]);
            dg += qk[o][i] * dyv[o][i];
        }
    const float g = gamma[w];
    if (lane == 0) d_gamma[w] = dg;
    // dV[i, p] = g sum_o qk[o, i] dY[o, p]
    for (int e = 2 * lane; e < s.P; e += 64) {
        float2 dv[M];
#pragma unroll
        for (int o = 0; o < M; ++o) dv[o] = Pair<T>::ld(dY + ((t * M + o) * s.H + h) * (long long)s.P + e);
#pragma unroll
        for (int i = 0; i < M; ++i) {
            float2 a = make_float2(0.f, 0.f);
#pragma unroll
            for (int o = 0; o < M; ++o) {
                a.x += qk[o][i] * dv[o].x;
                a.y += qk[o][i] * dv[o].y;
            }
            Pair<T>::st(dV + ((t * M + i) * s.H + h) * (long long)s.P + e, make_float2(g * a.x, g * a.y));
        }
    }
    // d_qk = g dyv;  dC[o, r] = sum_i d_qk[o, i] B[i, r];  dB[i, r] = sum_o d_qk[o, i] C[o, r]
    if ((s.N & 3) == 0) {
        for (int e = 4 * lane; e < s.N; e += 128) {
            float4 cv[M], bv[M];
#pragma unroll
            for (int i = 0; i < M; ++i) {
                const long long row = ((t * M + i) * s.H + h) * (long long)s.N + e;
                cv[i] = Pair<T>::ld4(C + row);
                bv[i] = Pair<T>::ld4(B + row);
            }
#pragma unroll
            for (int o = 0; o < M; ++o) {
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b2 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int i = 0; i < M; ++i) {
                    a.x += dyv[o][i] * bv[i].x;
                    a.y += dyv[o][i] * bv[i].y;
                    a.z += dyv[o][i] * bv[i].z;
                    a.w += dyv[o][i] * bv[i].w;
                    b2.x += dyv[i][o] * cv[i].x;
                    b2.y += dyv[i][o] * cv[i].y;
                    b2.z += dyv[i][o] * cv[i].z;
                    b2.w += dyv[i][o] * cv[i].w;
                }
                const long long row = ((t * M + o) * s.H + h) * (long long)s.N + e;
                Pair<T>::st4(dC + row, make_float4(g * a.x, g * a.y, g * a.z, g * a.w));
                Pair<T>::st4(dB + row, make_float4(g * b2.x, g * b2.y, g * b2.z, g * b2.w));
            }
        }
    } else {
        for (int e = 2 * lane; e < s.N; e += 64) {
            float2 cv[M], bv[M];
#pragma unroll
            for (int i = 0; i < M; ++i) {
                const long long row = ((t * M + i) * s.H + h) * (long long)s.N + e;
                cv[i] = Pair<T>::ld(C + row);
                bv[i] = Pair<T>::ld(B + row);
            }
#pragma unroll
            for (int o = 0; o < M; ++o) {
                float2 a = make_float2(0.f, 0.f), b2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < M; ++i) {
                    a.x += dyv[o][i] * bv[i].x;
                    a.y += dyv[o][i] * bv[i].y;
                    b2.x += dyv[i][o] * cv[i].x;
                    b2.y += dyv[i][o] * cv[i].y;
                }
                const long long row = ((t * M + o) * s.H + h) * (long long)s.N + e;
                Pair<T>::st(dC + row, make_float2(g * a.x, g * a.y));
                Pair<T>::st(dB + row, make_float2(g * b2.x, g * b2.y));
            }
        }
    }
}

// The same two kernels when the state axis fits one 4-wide piece per lane
// (N <= 128, N % 4 == 0) and the head axis one pair per lane (P <= 64, P
// even): every row the warp needs is loaded at the start, so a warp waits for
// one memory round trip instead of two (forward) or four (backward), and
// nothing is read twice.
template <typename T, int M>
__global__ void y_diag_fwd_fast(const T *__restrict__ V, const T *__restrict__ B, const T *__restrict__ C,
                                const float *__restrict__ gamma, T *__restrict__ y, DShape s) {
    const long long w = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= s.T * s.H) return;
    const int h = (int)(w % s.H);
    const long long t = w / s.H;
    const bool hn = 4 * lane < s.N, hp = 2 * lane < s.P;
    float4 cv[M], bv[M];
    float2 vv[M];
#pragma unroll
    for (int i = 0; i < M; ++i) {
        const long long rn = ((t * M + i) * s.H + h) * (long long)s.N + 4 * lane;
        const long long rp = ((t * M + i) * s.H + h) * (long long)s.P + 2 * lane;
        cv[i] = hn ? Pair<T>::ld4(C + rn) : make_float4(0.f, 0.f, 0.f, 0.f);
        bv[i] = hn ? Pair<T>::ld4(B + rn) : make_float4(0.f, 0.f, 0.f, 0.f);
        vv[i] = hp ? Pair<T>::ld(V + rp) : make_float2(0.f, 0.f);
    }
    const float g = gamma[w];
    float qk[M][M];
#pragma unroll
    for (int o = 0; o < M; ++o)
#pragma unroll
        for (int i = 0; i < M; ++i) qk[o][i] = warp_sum(dot4(cv[o], bv[i]));
    if (!hp) return;
#pragma unroll
    for (int o = 0; o < M; ++o) {
        float2 a = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < M; ++i) {
            a.x += qk[o][i] * vv[i].x;
            a.y += qk[o][i] * vv[i].y;
        }
        Pair<T>::st(y + ((t * M + o) * s.H + h) * (long long)s.P + 2 * lane, make_float2(g * a.x, g * a.y));
    }
}

template <typename T, int M>
__global__ void y_diag_bwd_fast(const T *__restrict__ dY, const T *__restrict__ V, const T *__restrict__ B,
                                const T *__restrict__ C, const float *__restrict__ gamma, T *__restrict__ dV,
                                T *__restrict__ dB, T *__restrict__ dC, float *__restrict__ d_gamma, DShape s) {
    const long long w = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= s.T * s.H) return;
    const int h = (int)(w % s.H);
    const long long t = w / s.H;
    const bool hn = 4 * lane < s.N, hp = 2 * lane < s.P;
    float4 cv[M], bv[M];
    float2 dv[M], vv[M];
#pragma unroll
    for (int i = 0; i < M; ++i) {
        const long long rn = ((t * M + i) * s.H + h) * (long long)s.N + 4 * lane;
        const long long rp = ((t * M + i) * s.H + h) * (long long)s.P + 2 * lane;
        cv[i] = hn ? Pair<T>::ld4(C + rn) : make_float4(0.f, 0.f, 0.f, 0.f);
        bv[i] = hn ? Pair<T>::ld4(B + rn) : make_float4(0.f, 0.f, 0.f, 0.f);
        dv[i] = hp ? Pair<T>::ld(dY + rp) : make_float2(0.f, 0.f);
        vv[i] = hp ? Pair<T>::ld(V + rp) : make_float2(0.f, 0.f);
    }
    const float g = gamma[w];
    float qk[M][M], dyv[M][M];
    float dg = 0.f;
#pragma unroll
    for (int o = 0; o < M; ++o)
#pragma unroll
        for (int i = 0; i < M; ++i) {
            qk[o][i] = warp_sum(dot4(cv[o], bv[i]));
            dyv[o][i] = warp_sum(dv[o].x * vv[i].x + dv[o].y * vv[i].y);
            dg += qk[o][i] * dyv[o][i];
        }
    if (lane == 0) d_gamma[w] = dg;
    if (hp) {  // dV[i, p] = g sum_o qk[o, i] dY[o, p]
#pragma unroll
        for (int i = 0; i < M; ++i) {
            float2 a = make_float2(0.f, 0.f);
#pragma unroll
            for (int o = 0; o < M; ++o) {
                a.x += qk[o][i] * dv[o].x;
                a.y += qk[o][i] * dv[o].y;
            }
            Pair<T>::st(dV + ((t * M + i) * s.H + h) * (long long)s.P + 2 * lane, make_float2(g * a.x, g * a.y));
        }
    }
    if (hn) {  // d_qk = g dyv;  dC[o, r] = sum_i d_qk[o, i] B[i, r];  dB[o, r] = sum_i d_qk[i, o] C[i, r]
#pragma unroll
        for (int o = 0; o < M; ++o) {
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b2 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < M; ++i) {
                a.x += dyv[o][i] * bv[i].x;
                a.y += dyv[o][i] * bv[i].y;
                a.z += dyv[o][i] * bv[i].z;
                a.w += dyv[o][i] * bv[i].w;
                b2.x += dyv[i][o] * cv[i].x;
                b2.y += dyv[i][o] * cv[i].y;
                b2.z += dyv[i][o] * cv[i].z;
                b2.w += dyv[i][o] * cv[i].w;
            }
            const long long row = ((t * M + o) * s.H + h) * (long long)s.N + 4 * lane;
            Pair<T>::st4(dC + row, make_float4(g * a.x, g * a.y, g * a.z, g * a.w));
            Pair<T>::st4(dB + row, make_float4(g * b2.x, g * b2.y, g * b2.z, g * b2.w));
        }
    }
}

// ---------------------------------------------------------------- host side
ssd_status m3_fail(ssd_status st, const char *msg) {
    record_error(msg);
    return st;
}
bool al16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
bool y_diag_fits_lanes(const DShape &s) { return s.N <= 128 && (s.N & 3) == 0 && s.P <= 64 && (s.P & 1) == 0; }

ssd_status quat_check(const void *const *ptrs, int nreq, int64_t b, int64_t L, int64_t H, int64_t J) {
    if (b < 1 || L < 1 || H < 1 || J < 1) return m3_fail(SSD_ERR_INVALID_ARG, "every dimension must be >= 1");
    if ((double)b * L * H * J * 4 > 4.0e15) return m3_fail(SSD_ERR_UNSUPPORTED, "problem too large");
    for (int i = 0; i < nreq; ++i)
        if (!ptrs[i] || !al16(ptrs[i])) return m3_fail(SSD_ERR_INVALID_ARG, "a required pointer is NULL or not 16-byte aligned");
    return SSD_OK;
}

QShape qshape(int64_t b, int64_t L, int64_t H, int64_t J) {
    return QShape{b, L, H * J, (L + kSeg - 1) / kSeg};
}

unsigned qgrid(const QShape &s) { return (unsigned)((s.b * s.S * s.C + 255) / 256); }
unsigned cgrid(const QShape &s) { return (unsigned)((s.b * s.C * 32 + 255) / 256); }  // a warp per chain

template <typename T, int M>
cudaError_t launch_y_fwd(const DShape &s, const void *V, const void *B, const void *C, const float *g, void *y,
                         cudaStream_t st) {
    const long long threads = s.T * s.H * 32;
    const unsigned grid = (unsigned)((threads + 255) / 256);
    if (y_diag_fits_lanes(s))
        y_diag_fwd_fast<T, M><<<grid, 256, 0, st>>>((const T *)V, (const T *)B, (const T *)C, g, (T *)y, s);
    else
        y_diag_fwd<T, M><<<grid, 256, 0, st>>>((const T *)V, (const T *)B, (const T *)C, g, (T *)y, s);
    return cudaGetLastError();
}
template <typename T, int M>
cudaError_t launch_y_bwd(const DShape &s, const void *dY, const void *V, const void *B, const void *C,
                         const float *g, void *dV, void *dB, void *dC, float *dg, cudaStream_t st) {
    const long long threads = s.T * s.H * 32;
    const unsigned grid = (unsigned)((threads + 255) / 256);
    if (y_diag_fits_lanes(s))
        y_diag_bwd_fast<T, M><<<grid, 256, 0, st>>>((const T *)dY, (const T *)V, (const T *)B, (const T *)C, g,
                                                    (T *)dV, (T *)dB, (T *)dC, dg, s);
    else
        y_diag_bwd<T, M><<<grid, 256, 0, st>>>((const T *)dY, (const T *)V, (const T *)B, (const T *)C, g,
                                               (T *)dV, (T *)dB, (T *)dC, dg, s);
    return cudaGetLastError();
}

ssd_status y_check(ssd_dtype dtype, const void *const *ptrs, int n, int64_t T, int64_t m, int64_t H, int64_t P,
                   int64_t N) {
    if (dtype != SSD_F32 && dtype != SSD_BF16) return m3_fail(SSD_ERR_INVALID_ARG, "unknown dtype");
    if (T < 1 || m < 1 || H < 1 || P < 1 || N < 1) return m3_fail(SSD_ERR_INVALID_ARG, "every dimension must be >= 1");
    if (m > 4) return m3_fail(SSD_ERR_UNSUPPORTED, "mimo rank above 4");
    if ((P & 1) || (N & 1)) return m3_fail(SSD_ERR_UNSUPPORTED, "headdim and dstate must be even");
    if (P > (1 << 20) || N > (1 << 20) || H > (1 << 20) || (double)T * H * 32 > 4.0e18)
        return m3_fail(SSD_ERR_UNSUPPORTED, "problem too large");
    for (int i = 0; i < n; ++i)
        if (!ptrs[i] || !al16(ptrs[i])) return m3_fail(SSD_ERR_INVALID_ARG, "a required pointer is NULL or not 16-byte aligned");
    return SSD_OK;
}

ssd_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return SSD_OK;
    char msg[256];
    snprintf(msg, sizeof(msg), "launch failed: %s", cudaGetErrorString(e));
    return m3_fail(SSD_ERR_CUDA, msg);
}

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" {

size_t m3_quat_workspace_bytes(int64_t b, int64_t L, int64_t H, int64_t J, int backward) {
    if (b < 1 || L < 1 || H < 1 || J < 1) return 0;
    const QShape s = qshape(b, L, H, J);
    return (size_t)(backward ? 3 : 1) * (size_t)(s.b * s.S * s.C * 4) * sizeof(float);
}

ssd_status m3_quat_cumprod(const float *q, const float *init, float *cum, int64_t b, int64_t L, int64_t H,
                           int64_t J, void *workspace, size_t workspace_bytes, void *stream) {
    record_error("");
    const void *req[] = {q, cum, workspace};
    ssd_status st = quat_check(req, 3, b, L, H, J);
    if (st != SSD_OK) return st;
    if (init && !al16(init)) return m3_fail(SSD_ERR_INVALID_ARG, "init is not 16-byte aligned");
    if (workspace_bytes < m3_quat_workspace_bytes(b, L, H, J, 0)) return m3_fail(SSD_ERR_WORKSPACE, "workspace too small");
    const QShape s = qshape(b, L, H, J);
    cudaStream_t cs = (cudaStream_t)stream;
    float *segp = (float *)workspace;
    quat_seg_product<<<qgrid(s), 256, 0, cs>>>(q, segp, s);
    quat_seg_carry<<<cgrid(s), 256, 0, cs>>>(segp, init, s);
    quat_seg_scan<<<qgrid(s), 256, 0, cs>>>(q, segp, cum, s);
    return cuda_status(cudaGetLastError());
}

ssd_status m3_quat_cumprod_backward(const float *q, const float *init, const float *d_cum, float *d_q,
                                    float *d_init, int64_t b, int64_t L, int64_t H, int64_t J, void *workspace,
                                    size_t workspace_bytes, void *stream) {
    record_error("");
    const void *req[] = {q, d_cum, d_q, workspace};
    ssd_status st = quat_check(req, 4, b, L, H, J);
    if (st != SSD_OK) return st;
    if ((init && !al16(init)) || (d_init && !al16(d_init)))
        return m3_fail(SSD_ERR_INVALID_ARG, "init / d_init is not 16-byte aligned");
    if (workspace_bytes < m3_quat_workspace_bytes(b, L, H, J, 1)) return m3_fail(SSD_ERR_WORKSPACE, "workspace too small");
    const QShape s = qshape(b, L, H, J);
    cudaStream_t cs = (cudaStream_t)stream;
    float *segp = (float *)workspace, *segT = segp + s.b * s.S * s.C * 4, *later = segT + s.b * s.S * s.C * 4;
    quat_bwd_segments<<<qgrid(s), 256, 0, cs>>>(q, d_cum, segp, segT, s);
    quat_bwd_carry<<<cgrid(s), 256, 0, cs>>>(segp, segT, later, s);
    quat_bwd_apply<<<qgrid(s), 256, 0, cs>>>(q, init, d_cum, segp, segT, later, d_q, d_init, s);
    return cuda_status(cudaGetLastError());
}

ssd_status m3_y_diag(ssd_dtype dtype, const void *V, const void *B, const void *C, const float *gamma, void *y,
                     int64_t T, int64_t m, int64_t H, int64_t P, int64_t N, void *stream) {
    record_error("");
    const void *req[] = {V, B, C, gamma, y};
    ssd_status st = y_check(dtype, req, 5, T, m, H, P, N);
    if (st != SSD_OK) return st;
    const DShape s{T, (int)H, (int)P, (int)N};
    cudaStream_t cs = (cudaStream_t)stream;
    cudaError_t e;
#define Y_FWD(TY)                                                              \
    switch (m) {                                                               \
        case 1: e = launch_y_fwd<TY, 1>(s, V, B, C, gamma, y, cs); break;      \
        case 2: e = launch_y_fwd<TY, 2>(s, V, B, C, gamma, y, cs); break;      \
        case 3: e = launch_y_fwd<TY, 3>(s, V, B, C, gamma, y, cs); break;      \
        default: e = launch_y_fwd<TY, 4>(s, V, B, C, gamma, y, cs); break;     \
    }
    if (dtype == SSD_F32) {
        Y_FWD(float)
    } else {
        Y_FWD(bf16)
    }
#undef Y_FWD
    return cuda_status(e);
}

ssd_status m3_y_diag_backward(ssd_dtype dtype, const void *dY, const void *V, const void *B, const void *C,
                              const float *gamma, void *dV, void *dB, void *dC, float *d_gamma, int64_t T,
                              int64_t m, int64_t H, int64_t P, int64_t N, void *stream) {
    record_error("");
    const void *req[] = {dY, V, B, C, gamma, dV, dB, dC, d_gamma};
    ssd_status st = y_check(dtype, req, 9, T, m, H, P, N);
    if (st != SSD_OK) return st;
    const DShape s{T, (int)H, (int)P, (int)N};
    cudaStream_t cs = (cudaStream_t)stream;
    cudaError_t e;
#define Y_BWD(TY)                                                                                \
    switch (m) {                                                                                 \
        case 1: e = launch_y_bwd<TY, 1>(s, dY, V, B, C, gamma, dV, dB, dC, d_gamma, cs); break;  \
        case 2: e = launch_y_bwd<TY, 2>(s, dY, V, B, C, gamma, dV, dB, dC, d_gamma, cs); break;  \
        case 3: e = launch_y_bwd<TY, 3>(s, dY, V, B, C, gamma, dV, dB, dC, d_gamma, cs); break;  \
        default: e = launch_y_bwd<TY, 4>(s, dY, V, B, C, gamma, dV, dB, dC, d_gamma, cs); break; \
    }
    if (dtype == SSD_F32) {
        Y_BWD(float)
    } else {
        Y_BWD(bf16)
    }
#undef Y_BWD
    return cuda_status(e);
}

}  // extern "C"
