// ssd_tc.cu -- tcgen05 tensor-core kernels of the bf16 path (sm_103a).
//
// The dense contractions of the chunked scan run as tcgen05.mma (kind::f16,
// bf16 operands, fp32 accumulators in TMEM) on operands staged in shared
// memory: raw tiles of x, dy, B, C and the bf16 chunk states arrive by TMA
// (cp.async.bulk.tensor, 128-byte swizzle); operands that carry a per-token
// factor (the causal decay matrix W, the K3 / BLUE scales) are formed by the
// CTA's threads in registers and written to shared memory in the same
// swizzled layout.  One elected thread issues the MMAs; the epilogues read
// TMEM with tcgen05.ld (warp w owns TMEM lanes 32w..32w+31).
//
// Formulas (burn-mamba, "combined_backward.rs"): K2 CB = C B^T; K3 intra =
// x^T (B * dt * exp(cumA_last - cumA)); K5 y = exp(cumA) (C s_in^T) +
// causal(CB * exp(cumA_t - cumA_s) * dt_s) x + D x; BLUE backward
// d_s_in = (dy * exp(cumA))^T C and d_da_blue; ORANGE backward dW = dy x^T,
// dx = W^T dy, ddt / d_da row and column sums, d_cb; K3 backward
// dx += bbs * (B d_intra^T), d_bbs; K2 backward dC = d_cb B, dB = d_cb^T C.
//
// Supported: headdim 64, dstate 128, chunk_len 128 or 256 (t-blocks of 128
// rows, MMA M = 128).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "ssd_tc.cuh"
#include "tc_ptx.cuh"

namespace ssd {

using namespace tc;

namespace {

constexpr int kP = 64;     // headdim
constexpr int kN = 128;    // dstate
constexpr int kThreads = 128;
constexpr int kTile = 16384;  // one [128 rows][64] bf16 SW128 tile
constexpr int kStatusTimeout = 5;

struct TcMaps {
    CUtensorMap x, dy, B, C, st, dst;
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return (uint8_t *)(((uintptr_t)p + 1023) & ~(uintptr_t)1023);
}

__device__ __forceinline__ void flag_timeout(const Params &p) { atomicExch(p.status, kStatusTimeout); }

// Bounded wait by every thread of the CTA; the result is made CTA-uniform so
// that no warp can diverge before a .sync.aligned tcgen05 instruction or a
// barrier inside a loop.
__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t parity, bool ok) {
    const bool r = ok ? mbar_wait(bar, parity) : false;
    return __syncthreads_and(r ? 1 : 0) != 0;
}

// Synchronise the CTA around tcgen05 work (orders TMEM accesses with the barrier).
__device__ __forceinline__ void tc_sync() {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// Scale every bf16 of `rows` consecutive 128-byte rows (any swizzle) by f[row];
// rows whose flag is off are zeroed (a select, so non-finite padding cannot leak).
__device__ __forceinline__ void scale_rows(uint8_t *tile, int rows, const float *f, int valid_rows) {
    const uint32_t base = smem_u32(tile);
    for (int i = threadIdx.x; i < rows * 8; i += blockDim.x) {
        const int row = i >> 3;
        const uint32_t a = base + (uint32_t)i * 16u;
        if (row >= valid_rows) {
            st_shared_v4(a, 0u, 0u, 0u, 0u);
            continue;
        }
        uint4 v = ld_shared_v4(a);
        const float s = f[row];
        v.x = pack_bf2(bf_lo(v.x) * s, bf_hi(v.x) * s);
        v.y = pack_bf2(bf_lo(v.y) * s, bf_hi(v.y) * s);
        v.z = pack_bf2(bf_lo(v.z) * s, bf_hi(v.z) * s);
        v.w = pack_bf2(bf_lo(v.w) * s, bf_hi(v.w) * s);
        st_shared_v4(a, v.x, v.y, v.z, v.w);
    }
}

// Zero rows [from, rows) of a tile of 128-byte rows.
__device__ __forceinline__ void zero_rows_from(uint8_t *tile, int rows, int from) {
    if (from >= rows) return;
    const uint32_t base = smem_u32(tile);
    for (int i = threadIdx.x + from * 8; i < rows * 8; i += blockDim.x)
        st_shared_v4(base + (uint32_t)i * 16u, 0u, 0u, 0u, 0u);
}

// Dot product of a swizzled bf16 row (64 values) with 64 floats.
__device__ __forceinline__ float dot_row64(const uint8_t *tile, int row, const float *v) {
    const uint32_t base = smem_u32(tile);
    float acc = 0.f;
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
        const uint4 u = ld_shared_v4(base + sw128_chunk(row, c8));
        const float *w = v + 8 * c8;
        acc += bf_lo(u.x) * w[0] + bf_hi(u.x) * w[1] + bf_lo(u.y) * w[2] + bf_hi(u.y) * w[3] +
               bf_lo(u.z) * w[4] + bf_hi(u.z) * w[5] + bf_lo(u.w) * w[6] + bf_hi(u.w) * w[7];
    }
    return acc;
}

// Unpack one swizzled bf16 row (64 values) into floats.
__device__ __forceinline__ void load_row64(const uint8_t *tile, int row, float *out) {
    const uint32_t base = smem_u32(tile);
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
        const uint4 u = ld_shared_v4(base + sw128_chunk(row, c8));
        float *o = out + 8 * c8;
        o[0] = bf_lo(u.x); o[1] = bf_hi(u.x); o[2] = bf_lo(u.y); o[3] = bf_hi(u.y);
        o[4] = bf_lo(u.z); o[5] = bf_hi(u.z); o[6] = bf_lo(u.w); o[7] = bf_hi(u.w);
    }
}

// Store 64 floats as a contiguous bf16 row in global memory.
__device__ __forceinline__ void store_row64_bf16(bf16 *dst, const float *v) {
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
        uint4 u;
        u.x = pack_bf2(v[8 * c8 + 0], v[8 * c8 + 1]);
        u.y = pack_bf2(v[8 * c8 + 2], v[8 * c8 + 3]);
        u.z = pack_bf2(v[8 * c8 + 4], v[8 * c8 + 5]);
        u.w = pack_bf2(v[8 * c8 + 6], v[8 * c8 + 7]);
        reinterpret_cast<uint4 *>(dst)[c8] = u;
    }
}

// ====================================================================== K2
// CTA per (b, chunk, group).  CB[t, s] = sum_r C[t, r] B[s, r] for the causal
// column range of each 128-row t-block (both operands K-major).
template <int Q>
__global__ void __launch_bounds__(kThreads) tc_k2_kernel(const Params p, const __grid_constant__ TcMaps maps) {
    constexpr int NT = Q / 128;
    constexpr uint32_t RB = Q * 128;  // one r-block ([Q rows][64])
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *Cs = sm, *Bs = sm + 2 * RB;
    __shared__ uint64_t bar_tma, bar_mma;
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.x % p.G, c = (blockIdx.x / p.G) % p.n, bi = blockIdx.x / (p.G * p.n);
    const int t0 = c * Q;
    const int vrows = min(Q, valid_len_of(p, bi) - t0);
    if (vrows <= 0) return;  // consumers never read CB of chunks past valid_len
    constexpr uint32_t NCOL = NT == 2 ? 512 : 128;
    if (tid == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&s_tmem, NCOL);
    tc_sync();
    const uint32_t tm = s_tmem;
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar_tma, 4 * RB);
        for (int rb = 0; rb < 2; ++rb)
            for (int j = 0; j < NT; ++j) {
                tma_load_4d(Cs + rb * RB + j * kTile, &maps.C, &bar_tma, 64 * rb, g, t0 + 128 * j, bi);
                tma_load_4d(Bs + rb * RB + j * kTile, &maps.B, &bar_tma, 64 * rb, g, t0 + 128 * j, bi);
            }
    }
    bool ok = wait_all(&bar_tma, 0, true);
    if (ok && vrows < Q) {
        for (int rb = 0; rb < 2; ++rb) {
            zero_rows_from(Cs + rb * RB, Q, vrows);
            zero_rows_from(Bs + rb * RB, Q, vrows);
        }
    }
    fence_async_smem();
    tc_sync();
    if (tid == 0 && ok) {
        for (int tb = 0; tb < NT; ++tb) {
            const uint32_t idesc = idesc_bf16(128, 128 * (tb + 1), false, false);
            const uint32_t col = tb == 0 ? 0u : 128u;
            for (int ks = 0; ks < kN / 16; ++ks)
                mma_bf16(tm + col, sdesc_kmajor(smem_u32(Cs + tb * kTile), ks, RB),
                         sdesc_kmajor(smem_u32(Bs), ks, RB), idesc, ks > 0);
        }
        mma_commit(&bar_mma);
    }
    ok = wait_all(&bar_mma, 0, ok);
    tc_fence_after();
    if (ok) {
        float *cb = p.CB + ix_cb(p, bi, c, g);
        for (int tb = 0; tb < NT; ++tb) {
            const int t = tb * 128 + 32 * warp + lane;
            const uint32_t col = tb == 0 ? 0u : 128u;
            for (int s0 = 0; s0 < 128 * (tb + 1); s0 += 32) {
                float v[32];
                tmem_ld32(tmem_addr(tm, 32 * warp, col + s0), v);
                float4 *dst = reinterpret_cast<float4 *>(cb + (size_t)t * Q + s0);
#pragma unroll
                for (int j = 0; j < 8; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            }
        }
    } else if (tid == 0) {
        flag_timeout(p);
    }
    tc_sync();
    if (warp == 0) tmem_dealloc(tm, NCOL);
}

// ====================================================================== K3
// CTA per (b, chunk, head).  intra[p, r] = sum_l x[l, p] * B[l, r] * bbs[l],
// bbs = dt * exp(cumA_last - cumA), computed as D[r, p] with M = dstate (A =
// scaled B, MN-major) and N = headdim (B operand = x, MN-major).
template <int Q>
__global__ void __launch_bounds__(kThreads) tc_k3_kernel(const Params p, const __grid_constant__ TcMaps maps) {
    constexpr int NT = Q / 128;
    constexpr uint32_t XB = Q * 128;  // [Q][64] bf16
    constexpr uint32_t RB = Q * 128;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *xs = sm, *bs = sm + XB;
    float *bbs = reinterpret_cast<float *>(bs + 2 * RB);
    __shared__ uint64_t bar_tma, bar_mma;
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x % p.H, c = (blockIdx.x / p.H) % p.n, bi = blockIdx.x / (p.H * p.n);
    const int g = h / p.hpg, t0 = c * Q;
    const int V = valid_len_of(p, bi);
    const int vrows = min(Q, V - t0);
    float *out = p.states + ix_state(p, bi, c, h);
    if (vrows <= 0) {
        for (int i = tid; i < kP * kN; i += kThreads) out[i] = 0.f;
        return;
    }
    if (tid == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&s_tmem, 64);
    tc_sync();
    const uint32_t tm = s_tmem;
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar_tma, XB + 2 * RB);
        for (int j = 0; j < NT; ++j) {
            tma_load_4d(xs + j * kTile, &maps.x, &bar_tma, 0, h, t0 + 128 * j, bi);
            for (int rb = 0; rb < 2; ++rb)
                tma_load_4d(bs + rb * RB + j * kTile, &maps.B, &bar_tma, 64 * rb, g, t0 + 128 * j, bi);
        }
    }
    const float *cum = p.cumA + ix_chunk(p, bi, h, c) * Q;
    const float cend = p.endA[ix_chunk(p, bi, h, c)];
    for (int l = tid; l < Q; l += kThreads)
        bbs[l] = l < vrows ? p.dt[ix_dt(p, bi, h, t0 + l)] * __expf(cend - cum[l]) : 0.f;
    bool ok = wait_all(&bar_tma, 0, true);
    if (ok) {
        scale_rows(bs, Q, bbs, vrows);
        scale_rows(bs + RB, Q, bbs, vrows);
        zero_rows_from(xs, Q, vrows);
    }
    fence_async_smem();
    tc_sync();
    if (tid == 0 && ok) {
        const uint32_t idesc = idesc_bf16(128, 64, true, true);
        for (int ks = 0; ks < Q / 16; ++ks)
            mma_bf16(tm, sdesc_mnmajor(smem_u32(bs), ks, RB), sdesc_mnmajor(smem_u32(xs), ks, XB), idesc, ks > 0);
        mma_commit(&bar_mma);
    }
    ok = wait_all(&bar_mma, 0, ok);
    tc_fence_after();
    if (ok) {
        const int r = 32 * warp + lane;
        for (int cc = 0; cc < kP; cc += 32) {
            float v[32];
            tmem_ld32(tmem_addr(tm, 32 * warp, cc), v);
#pragma unroll
            for (int j = 0; j < 32; ++j) out[(size_t)(cc + j) * kN + r] = v[j];
        }
    } else if (tid == 0) {
        flag_timeout(p);
    }
    tc_sync();
    if (warp == 0) tmem_dealloc(tm, 64);
}

// ====================================================================== K5
// CTA per (b, chunk, head).  Per 128-row t-block tb:
//   ORANGE (TMEM cols tb*64):        W[tb] (K-major, formed here) x  (x MN-major)
//   BLUE   (TMEM cols NT*64+tb*64):  C[tb] (K-major)             s_in (K-major)
// y = ORANGE + exp(cumA_t) * BLUE + D x;  W[t, s] = CB[t, s] exp(cumA_t - cumA_s) dt_s (s <= t).
template <int Q>
__global__ void __launch_bounds__(kThreads) tc_k5_kernel(const Params p, const __grid_constant__ TcMaps maps) {
    constexpr int NT = Q / 128;
    constexpr uint32_t XB = Q * 128, RB = Q * 128, SB = 64 * 128;
    constexpr uint32_t WB = kTile * 2 * (NT * (NT + 1) / 2);  // tb0: 2 tiles, tb1: 4 tiles
    constexpr uint32_t NCOL = NT == 2 ? 256 : 128;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *xs = sm, *Cs = xs + XB, *Ss = Cs + 2 * RB, *Ws = Ss + 2 * SB;
    float *cum = reinterpret_cast<float *>(Ws + WB);
    float *dts = cum + Q;
    __shared__ uint64_t bar_tma, bar_mma;
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x % p.H, c = (blockIdx.x / p.H) % p.n, bi = blockIdx.x / (p.H * p.n);
    const int g = h / p.hpg, t0 = c * Q;
    const int V = valid_len_of(p, bi);
    const int vrows = min(Q, V - t0);
    bf16 *Y = (bf16 *)p.y;
    if (vrows <= 0) {
        const int rows = min(Q, p.L - t0);
        for (int i = tid; i < rows * (kP / 8); i += kThreads)
            reinterpret_cast<uint4 *>(Y + ix_x(p, bi, t0 + i / 8, h, 0))[i % 8] = make_uint4(0, 0, 0, 0);
        return;
    }
    if (tid == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&s_tmem, NCOL);
    tc_sync();
    const uint32_t tm = s_tmem;
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar_tma, XB + 2 * RB + 2 * SB);
        const int sidx = (bi * p.n + c) * p.H + h;
        for (int j = 0; j < NT; ++j) {
            tma_load_4d(xs + j * kTile, &maps.x, &bar_tma, 0, h, t0 + 128 * j, bi);
            for (int rb = 0; rb < 2; ++rb)
                tma_load_4d(Cs + rb * RB + j * kTile, &maps.C, &bar_tma, 64 * rb, g, t0 + 128 * j, bi);
        }
        for (int rb = 0; rb < 2; ++rb) tma_load_3d(Ss + rb * SB, &maps.st, &bar_tma, 64 * rb, 0, sidx);
    }
    const float *cumg = p.cumA + ix_chunk(p, bi, h, c) * Q;
    for (int l = tid; l < Q; l += kThreads) {
        cum[l] = cumg[l];
        dts[l] = l < vrows ? p.dt[ix_dt(p, bi, h, t0 + l)] : 0.f;
    }
    __syncthreads();
    // ---- form W (bf16, K-major per t-block) while the TMA loads land
    const float *cb = p.CB + ix_cb(p, bi, c, g);
    for (int tb = 0; tb < NT; ++tb) {
        uint8_t *Wt = Ws + kTile * 2 * (tb * (tb + 1) / 2);
        const int nch = 16 * (tb + 1);  // 8-column chunks per row
        for (int i = tid; i < 128 * nch; i += kThreads) {
            const int row = i / nch, ch = i % nch;
            const int t = tb * 128 + row, s0 = 8 * ch;
            uint32_t u[4] = {0u, 0u, 0u, 0u};
            if (s0 <= t && t < vrows) {
                const float4 a = *reinterpret_cast<const float4 *>(cb + (size_t)t * Q + s0);
                const float4 b = *reinterpret_cast<const float4 *>(cb + (size_t)t * Q + s0 + 4);
                const float cv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                const float ct = cum[t];
                float w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int s = s0 + e;
                    w[e] = (s <= t && s < vrows) ? cv[e] * __expf(ct - cum[s]) * dts[s] : 0.f;
                }
                u[0] = pack_bf2(w[0], w[1]);
                u[1] = pack_bf2(w[2], w[3]);
                u[2] = pack_bf2(w[4], w[5]);
                u[3] = pack_bf2(w[6], w[7]);
            }
            st_shared_v4(smem_u32(Wt + (s0 / 64) * kTile) + sw128_chunk(row, (s0 % 64) / 8), u[0], u[1], u[2], u[3]);
        }
    }
    bool ok = wait_all(&bar_tma, 0, true);
    if (ok && vrows < Q) {
        zero_rows_from(xs, Q, vrows);
        zero_rows_from(Cs, Q, vrows);
        zero_rows_from(Cs + RB, Q, vrows);
    }
    fence_async_smem();
    tc_sync();
    if (tid == 0 && ok) {
        for (int tb = 0; tb < NT; ++tb) {
            uint8_t *Wt = Ws + kTile * 2 * (tb * (tb + 1) / 2);
            const uint32_t id = idesc_bf16(128, 64, false, true);
            for (int ks = 0; ks < 8 * (tb + 1); ++ks)
                mma_bf16(tm + tb * 64, sdesc_kmajor(smem_u32(Wt), ks, kTile), sdesc_mnmajor(smem_u32(xs), ks, XB), id,
                         ks > 0);
            const uint32_t ib = idesc_bf16(128, 64, false, false);
            for (int ks = 0; ks < kN / 16; ++ks)
                mma_bf16(tm + NT * 64 + tb * 64, sdesc_kmajor(smem_u32(Cs + tb * kTile), ks, RB),
                         sdesc_kmajor(smem_u32(Ss), ks, SB), ib, ks > 0);
        }
        mma_commit(&bar_mma);
    }
    ok = wait_all(&bar_mma, 0, ok);
    tc_fence_after();
    if (ok) {
        const float Dh = p.D[h];
        for (int tb = 0; tb < NT; ++tb) {
            const int t = tb * 128 + 32 * warp + lane;
            float o[64], bl[64], xv[64];
            tmem_ld32(tmem_addr(tm, 32 * warp, tb * 64), o);
            tmem_ld32(tmem_addr(tm, 32 * warp, tb * 64 + 32), o + 32);
            tmem_ld32(tmem_addr(tm, 32 * warp, NT * 64 + tb * 64), bl);
            tmem_ld32(tmem_addr(tm, 32 * warp, NT * 64 + tb * 64 + 32), bl + 32);
            if (t0 + t < p.L) {
                if (t < vrows) {
                    load_row64(xs, t, xv);
                    const float e = __expf(cum[t]);
#pragma unroll
                    for (int j = 0; j < 64; ++j) o[j] = o[j] + e * bl[j] + Dh * xv[j];
                } else {
#pragma unroll
                    for (int j = 0; j < 64; ++j) o[j] = 0.f;
                }
                store_row64_bf16(Y + ix_x(p, bi, t0 + t, h, 0), o);
            }
        }
    } else if (tid == 0) {
        flag_timeout(p);
    }
    tc_sync();
    if (warp == 0) tmem_dealloc(tm, NCOL);
}

// ====================================================================== BLUE backward
// CTA per (b, chunk, head).  d_ch = dy * exp(cumA) (formed in place over dy).
//   d_s_in[r, p] = sum_l C[l, r] d_ch[l, p]        (TMEM cols 0..63; A = C MN-major, B = d_ch MN-major)
//   u[l, p]      = sum_r C[l, r] s_in[p, r]        (TMEM cols 64 + tb*64; both K-major)
//   d_cumA_blue[l] = sum_p d_ch[l, p] u[l, p]
template <int Q>
__global__ void __launch_bounds__(kThreads) tc_bwd_blue_kernel(const Params p, const __grid_constant__ TcMaps maps) {
    constexpr int NT = Q / 128;
    constexpr uint32_t XB = Q * 128, RB = Q * 128, SB = 64 * 128;
    constexpr uint32_t NCOL = NT == 2 ? 256 : 128;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *Cs = sm, *Ds = Cs + 2 * RB, *Ss = Ds + XB;
    float *ecum = reinterpret_cast<float *>(Ss + 2 * SB);
    __shared__ uint64_t bar_tma, bar_mma;
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x % p.H, c = (blockIdx.x / p.H) % p.n, bi = blockIdx.x / (p.H * p.n);
    const int g = h / p.hpg, t0 = c * Q;
    const int V = valid_len_of(p, bi);
    const int vrows = min(Q, V - t0);
    float *dsin = p.dstates + ix_state(p, bi, c, h);
    float *dcb = p.dcum_blue + ix_chunk(p, bi, h, c) * Q;
    if (vrows <= 0) {
        for (int i = tid; i < kP * kN; i += kThreads) dsin[i] = 0.f;
        for (int i = tid; i < Q; i += kThreads) dcb[i] = 0.f;
        return;
    }
    if (tid == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&s_tmem, NCOL);
    tc_sync();
    const uint32_t tm = s_tmem;
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar_tma, XB + 2 * RB + 2 * SB);
        const int sidx = (bi * p.n + c) * p.H + h;
        for (int j = 0; j < NT; ++j) {
            tma_load_4d(Ds + j * kTile, &maps.dy, &bar_tma, 0, h, t0 + 128 * j, bi);
            for (int rb = 0; rb < 2; ++rb)
                tma_load_4d(Cs + rb * RB + j * kTile, &maps.C, &bar_tma, 64 * rb, g, t0 + 128 * j, bi);
        }
        for (int rb = 0; rb < 2; ++rb) tma_load_3d(Ss + rb * SB, &maps.st, &bar_tma, 64 * rb, 0, sidx);
    }
    const float *cum = p.cumA + ix_chunk(p, bi, h, c) * Q;
    for (int l = tid; l < Q; l += kThreads) ecum[l] = l < vrows ? __expf(cum[l]) : 0.f;
    bool ok = wait_all(&bar_tma, 0, true);
    if (ok) {
        scale_rows(Ds, Q, ecum, vrows);
        if (vrows < Q) {
            zero_rows_from(Cs, Q, vrows);
            zero_rows_from(Cs + RB, Q, vrows);
        }
    }
    fence_async_smem();
    tc_sync();
    if (tid == 0 && ok) {
        const uint32_t i1 = idesc_bf16(128, 64, true, true);
        for (int ks = 0; ks < Q / 16; ++ks)
            mma_bf16(tm, sdesc_mnmajor(smem_u32(Cs), ks, RB), sdesc_mnmajor(smem_u32(Ds), ks, XB), i1, ks > 0);
        const uint32_t i2 = idesc_bf16(128, 64, false, false);
        for (int tb = 0; tb < NT; ++tb)
            for (int ks = 0; ks < kN / 16; ++ks)
                mma_bf16(tm + 64 + tb * 64, sdesc_kmajor(smem_u32(Cs + tb * kTile), ks, RB),
                         sdesc_kmajor(smem_u32(Ss), ks, SB), i2, ks > 0);
        mma_commit(&bar_mma);
    }
    ok = wait_all(&bar_mma, 0, ok);
    tc_fence_after();
    if (ok) {
        const int r = 32 * warp + lane;
        for (int cc = 0; cc < kP; cc += 32) {
            float v[32];
            tmem_ld32(tmem_addr(tm, 32 * warp, cc), v);
#pragma unroll
            for (int j = 0; j < 32; ++j) dsin[(size_t)(cc + j) * kN + r] = v[j];
        }
        for (int tb = 0; tb < NT; ++tb) {
            const int l = tb * 128 + 32 * warp + lane;
            float u[64];
            tmem_ld32(tmem_addr(tm, 32 * warp, 64 + tb * 64), u);
            tmem_ld32(tmem_addr(tm, 32 * warp, 64 + tb * 64 + 32), u + 32);
            dcb[l] = l < vrows ? dot_row64(Ds, l, u) : 0.f;
        }
    } else if (tid == 0) {
        flag_timeout(p);
    }
    tc_sync();
    if (warp == 0) tmem_dealloc(tm, NCOL);
}

// ====================================================================== main backward
// CTA per (b, chunk, head).  TMEM (Q = 256): dW tb0 cols [0,128), tb1 [128,384);
// U = B d_intra^T per 128-row s-block at [384 + mb*64); dx accumulators reuse
// [mb*64) once dW has been read.
//   phase 1: dW = dy x^T (K-major, K = headdim), U (K-major, K = dstate)
//   phase 2: d_bbs[s] = sum_p x U, dD partial; then W, row/column sums from dW
//            (W written MN-major over the freed x / B tiles)
//   phase 3: dx = W^T dy  (A = W MN-major, B = dy MN-major)
//   phase 4: dx += bbs * U + D dy; per-token outputs.
template <int Q>
__global__ void __launch_bounds__(kThreads) tc_bwd_main_kernel(const Params p, const __grid_constant__ TcMaps maps) {
    constexpr int NT = Q / 128;
    constexpr uint32_t XB = Q * 128, RB = Q * 128, SB = 64 * 128;
    constexpr uint32_t NCOL = NT == 2 ? 512 : 256;
    constexpr uint32_t UCOL = NT == 2 ? 384 : 128;   // U accumulators
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *DYs = sm, *Xs = DYs + XB, *Bs = Xs + XB, *DIs = Bs + 2 * RB;
    uint8_t *Ws = Xs;  // reuses x + B (3 * Q * 128 bytes >= W bytes)
    float *cum = reinterpret_cast<float *>(DIs + 2 * SB);
    float *dts = cum + Q;              // dt (0 past valid_len)
    float *dec_end = dts + Q;          // exp(cumA_last - cumA)
    float *dbbs = dec_end + Q;         // d_bbs
    float *tgt = dbbs + Q;             // row sums of dW * W
    float *colp = tgt + Q;             // [NT][4][2][Q] column partials (ddt_orange, src)
    float *red = colp + NT * 4 * 2 * Q;  // [4] dD partials
    __shared__ uint64_t bar_tma, bar_mma1, bar_mma2;
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x % p.H, c = (blockIdx.x / p.H) % p.n, bi = blockIdx.x / (p.H * p.n);
    const int g = h / p.hpg, t0 = c * Q;
    const int V = valid_len_of(p, bi);
    const int vrows = min(Q, V - t0);
    const size_t cbase = ix_chunk(p, bi, h, c) * Q;
    bf16 *DX = (bf16 *)p.dx;
    if (vrows <= 0) {
        const int rows = min(Q, p.L - t0);
        for (int i = tid; i < rows * (kP / 8); i += kThreads)
            reinterpret_cast<uint4 *>(DX + ix_x(p, bi, t0 + i / 8, h, 0))[i % 8] = make_uint4(0, 0, 0, 0);
        for (int i = tid; i < Q; i += kThreads) {
            p.ddt_main[cbase + i] = 0.f;
            p.d_delta[cbase + i] = 0.f;
            p.dcum_main[cbase + i] = 0.f;
        }
        if (tid == 0) p.dD_part[((size_t)bi * p.n + c) * p.H + h] = 0.f;
        return;
    }
    if (tid == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma1, 1);
        mbar_init(&bar_mma2, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&s_tmem, NCOL);
    tc_sync();
    const uint32_t tm = s_tmem;
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar_tma, 2 * XB + 2 * RB + 2 * SB);
        const int sidx = (bi * p.n + c) * p.H + h;
        for (int j = 0; j < NT; ++j) {
            tma_load_4d(DYs + j * kTile, &maps.dy, &bar_tma, 0, h, t0 + 128 * j, bi);
            tma_load_4d(Xs + j * kTile, &maps.x, &bar_tma, 0, h, t0 + 128 * j, bi);
            for (int rb = 0; rb < 2; ++rb)
                tma_load_4d(Bs + rb * RB + j * kTile, &maps.B, &bar_tma, 64 * rb, g, t0 + 128 * j, bi);
        }
        for (int rb = 0; rb < 2; ++rb) tma_load_3d(DIs + rb * SB, &maps.dst, &bar_tma, 64 * rb, 0, sidx);
    }
    {
        const float *cumg = p.cumA + cbase;
        const float cend = p.endA[ix_chunk(p, bi, h, c)];
        for (int l = tid; l < Q; l += kThreads) {
            const float cl = cumg[l];
            cum[l] = cl;
            dts[l] = l < vrows ? p.dt[ix_dt(p, bi, h, t0 + l)] : 0.f;
            dec_end[l] = __expf(cend - cl);
        }
        for (int i = tid; i < NT * 4 * 2 * Q; i += kThreads) colp[i] = 0.f;
    }
    bool ok = wait_all(&bar_tma, 0, true);
    if (ok && vrows < Q) {
        zero_rows_from(DYs, Q, vrows);
        zero_rows_from(Xs, Q, vrows);
        zero_rows_from(Bs, Q, vrows);
        zero_rows_from(Bs + RB, Q, vrows);
    }
    fence_async_smem();
    tc_sync();
    // ---- phase 1 MMAs
    if (tid == 0 && ok) {
        for (int tb = 0; tb < NT; ++tb) {
            const uint32_t id = idesc_bf16(128, 128 * (tb + 1), false, false);
            const uint32_t col = tb == 0 ? 0u : 128u;
            for (int ks = 0; ks < kP / 16; ++ks)
                mma_bf16(tm + col, sdesc_kmajor(smem_u32(DYs + tb * kTile), ks, XB),
                         sdesc_kmajor(smem_u32(Xs), ks, XB), id, ks > 0);
        }
        const uint32_t iu = idesc_bf16(128, 64, false, false);
        for (int mb = 0; mb < NT; ++mb)
            for (int ks = 0; ks < kN / 16; ++ks)
                mma_bf16(tm + UCOL + mb * 64, sdesc_kmajor(smem_u32(Bs + mb * kTile), ks, RB),
                         sdesc_kmajor(smem_u32(DIs), ks, SB), iu, ks > 0);
        mma_commit(&bar_mma1);
    }
    ok = wait_all(&bar_mma1, 0, ok);
    tc_fence_after();
    // ---- phase 2a: x-dependent reductions (before x / B are overwritten by W)
    float dd = 0.f;
    if (ok) {
        for (int mb = 0; mb < NT; ++mb) {
            const int s = mb * 128 + 32 * warp + lane;
            float u[64];
            tmem_ld32(tmem_addr(tm, 32 * warp, UCOL + mb * 64), u);
            tmem_ld32(tmem_addr(tm, 32 * warp, UCOL + mb * 64 + 32), u + 32);
            dbbs[s] = dot_row64(Xs, s, u);
            float dyv[64];
            load_row64(DYs, s, dyv);
            dd += dot_row64(Xs, s, dyv);
        }
    }
    dd = warp_sum(dd);
    if (lane == 0) red[warp] = dd;
    tc_sync();
    // ---- phase 2b: W (bf16, MN-major per 128-row s-block, rows t >= 128*mb), sums
    if (ok) {
        const float *cbm = p.CB + ix_cb(p, bi, c, g);
        for (int tb = 0; tb < NT; ++tb) {
            const int t = tb * 128 + 32 * warp + lane;
            const bool tv = t < vrows;
            const float ct = cum[t];
            const uint32_t col0 = tb == 0 ? 0u : 128u;
            float rowsum = 0.f;
            for (int s0 = 0; s0 < 128 * (tb + 1); s0 += 32) {
                float dw[32];
                tmem_ld32(tmem_addr(tm, 32 * warp, col0 + s0), dw);
                float gsum[32], dsum[32];
                float wv[32];
                const float *cbrow = cbm + (size_t)t * Q + s0;
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    float4 cv = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (tv && s0 + 4 * j4 <= t) cv = *reinterpret_cast<const float4 *>(cbrow + 4 * j4);
                    const float cvv[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = 4 * j4 + e, s = s0 + j;
                        float gg = 0.f, w = 0.f;
                        if (tv && s <= t && s < vrows) {
                            const float cbd = cvv[e] * __expf(ct - cum[s]);
                            gg = dw[j] * cbd;
                            w = cbd * dts[s];
                        }
                        gsum[j] = gg;
                        dsum[j] = gg * dts[s];
                        wv[j] = w;
                        rowsum += gg * dts[s];
                    }
                }
                // column sums over the warp's 32 rows: butterfly transpose-reduce
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) {
#pragma unroll
                    for (int j = 0; j < off; ++j) {
                        const bool upper = (lane & off) != 0;
                        const float send_g = upper ? gsum[j] : gsum[j + off];
                        const float send_d = upper ? dsum[j] : dsum[j + off];
                        const float rg = __shfl_xor_sync(0xffffffffu, send_g, off);
                        const float rd = __shfl_xor_sync(0xffffffffu, send_d, off);
                        if (upper) {
                            gsum[j] = gsum[j + off] + rg;
                            dsum[j] = dsum[j + off] + rd;
                        } else {
                            gsum[j] = gsum[j] + rg;
                            dsum[j] = dsum[j] + rd;
                        }
                    }
                }
                // lane now holds column s0 + lane in gsum[0], dsum[0]
                colp[((tb * 4 + warp) * 2 + 0) * Q + s0 + lane] = gsum[0];
                colp[((tb * 4 + warp) * 2 + 1) * Q + s0 + lane] = dsum[0];
                // W values into the MN-major tile of s-block mb = s0 / 128
                const int mb = s0 / 128;
                const uint32_t mbase = (mb == 0) ? 0u : (uint32_t)(2 * Q * 128);
                const uint32_t blk = (uint32_t)((Q - 128 * mb) * 128);  // bytes per 64-column block
                const int wrow = t - 128 * mb;
                if (wrow >= 0) {
                    const int sb = (s0 % 128) / 64;       // which 64-column block of the pair
                    const int c8b = (s0 % 64) / 8;         // first chunk of the 32 columns
                    const uint32_t base = smem_u32(Ws) + mbase + sb * blk;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        st_shared_v4(base + sw128_chunk(wrow, c8b + q4), pack_bf2(wv[8 * q4], wv[8 * q4 + 1]),
                                     pack_bf2(wv[8 * q4 + 2], wv[8 * q4 + 3]), pack_bf2(wv[8 * q4 + 4], wv[8 * q4 + 5]),
                                     pack_bf2(wv[8 * q4 + 6], wv[8 * q4 + 7]));
                }
            }
            tgt[t] = rowsum;
        }
    }
    fence_async_smem();
    tc_sync();
    // ---- phase 3: dx = W^T dy into the freed dW columns
    if (tid == 0 && ok) {
        const uint32_t id = idesc_bf16(128, 64, true, true);
        for (int mb = 0; mb < NT; ++mb) {
            const uint32_t mbase = (mb == 0) ? 0u : (uint32_t)(2 * Q * 128);
            const uint32_t blk = (uint32_t)((Q - 128 * mb) * 128);
            const int nks = (Q - 128 * mb) / 16;
            for (int ks = 0; ks < nks; ++ks)
                mma_bf16(tm + mb * 64, sdesc_mnmajor(smem_u32(Ws) + mbase, ks, blk),
                         sdesc_mnmajor(smem_u32(DYs) + (uint32_t)(128 * mb * 128), ks, XB), id, ks > 0);
        }
        mma_commit(&bar_mma2);
    }
    ok = wait_all(&bar_mma2, 0, ok);
    tc_fence_after();
    // ---- phase 4: dx and per-token outputs
    if (ok) {
        const float Dh = p.D[h];
        for (int mb = 0; mb < NT; ++mb) {
            const int s = mb * 128 + 32 * warp + lane;
            float acc[64], u[64], dyv[64];
            tmem_ld32(tmem_addr(tm, 32 * warp, mb * 64), acc);
            tmem_ld32(tmem_addr(tm, 32 * warp, mb * 64 + 32), acc + 32);
            tmem_ld32(tmem_addr(tm, 32 * warp, UCOL + mb * 64), u);
            tmem_ld32(tmem_addr(tm, 32 * warp, UCOL + mb * 64 + 32), u + 32);
            if (t0 + s < p.L) {
                if (s < vrows) {
                    load_row64(DYs, s, dyv);
                    const float bbs = dts[s] * dec_end[s];
#pragma unroll
                    for (int j = 0; j < 64; ++j) acc[j] = acc[j] + bbs * u[j] + Dh * dyv[j];
                } else {
#pragma unroll
                    for (int j = 0; j < 64; ++j) acc[j] = 0.f;
                }
                store_row64_bf16(DX + ix_x(p, bi, t0 + s, h, 0), acc);
            }
        }
        for (int s = tid; s < Q; s += kThreads) {
            float ddo = 0.f, src = 0.f;
            for (int tb = 0; tb < NT; ++tb)
                for (int w = 0; w < 4; ++w) {
                    ddo += colp[((tb * 4 + w) * 2 + 0) * Q + s];
                    src += colp[((tb * 4 + w) * 2 + 1) * Q + s];
                }
            const float dbb = s < vrows ? dbbs[s] : 0.f;
            const float ddelta = dbb * dts[s] * dec_end[s];
            p.ddt_main[cbase + s] = ddo + dbb * dec_end[s];
            p.d_delta[cbase + s] = ddelta;
            p.dcum_main[cbase + s] = tgt[s] - src - ddelta;
        }
        if (tid == 0) p.dD_part[((size_t)bi * p.n + c) * p.H + h] = red[0] + red[1] + red[2] + red[3];
    } else if (tid == 0) {
        flag_timeout(p);
    }
    tc_sync();
    if (warp == 0) tmem_dealloc(tm, NCOL);
}

// ====================================================================== group backward
// G1: CTA per (b, chunk, group, head slice, t-block).  Accumulates, over the
// slice's heads, d_cb[t, s] = sum_h dt_h[s] exp(cumA_h[t] - cumA_h[s]) dW_h[t, s]
// (s <= t) in TMEM (dW_h = dy_h x_h^T by MMA each head), then writes the fp32
// partial to the workspace.
template <int Q>
__global__ void __launch_bounds__(kThreads) tc_bwd_dcb_kernel(const Params p, const __grid_constant__ TcMaps maps) {
    constexpr int NT = Q / 128;
    constexpr uint32_t STG = kTile * (1 + NT);  // dy rows (1 tile) + x rows (up to NT tiles)
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    float *cumv = reinterpret_cast<float *>(sm + 2 * STG);  // [2][Q]
    float *dtv = cumv + 2 * Q;                              // [2][Q]
    __shared__ uint64_t bar_tma[2], bar_mma;
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int idx = blockIdx.x;
    const int tb = idx % NT;
    idx /= NT;
    const int slice = idx % p.nslice_cb;
    idx /= p.nslice_cb;
    const int g = idx % p.G, c = (idx / p.G) % p.n, bi = idx / (p.G * p.n);
    const int t0 = c * Q;
    const int vrows = min(Q, valid_len_of(p, bi) - t0);
    const int ncols = 128 * (tb + 1);
    const int per = (p.hpg + p.nslice_cb - 1) / p.nslice_cb;
    const int h_begin = g * p.hpg + slice * per;
    const int h_end = min(g * p.hpg + p.hpg, h_begin + per);
    float *out = p.d_cb + ((size_t)slice * p.b * p.n * p.G + ((size_t)bi * p.n + c) * p.G + g) * (size_t)Q * Q;
    if (vrows <= 0 || h_begin >= h_end) {
        for (int i = tid; i < 128 * ncols; i += kThreads)
            out[(size_t)(tb * 128 + i / ncols) * Q + i % ncols] = 0.f;
        return;
    }
    const uint32_t NCOL = tb == 0 ? 256u : 512u;
    const uint32_t ACC = 0, DW = (uint32_t)ncols;
    if (tid == 0) {
        mbar_init(&bar_tma[0], 1);
        mbar_init(&bar_tma[1], 1);
        mbar_init(&bar_mma, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&s_tmem, NCOL);
    tc_sync();
    const uint32_t tm = s_tmem;
    const uint32_t stage_bytes = (uint32_t)(kTile * (1 + (tb + 1)));
    auto issue = [&](int k) {
        const int h = h_begin + k, st = k & 1;
        uint8_t *dys = sm + st * STG, *xs = dys + kTile;
        mbar_arrive_expect_tx(&bar_tma[st], stage_bytes);
        tma_load_4d(dys, &maps.dy, &bar_tma[st], 0, h, t0 + 128 * tb, bi);
        for (int j = 0; j <= tb; ++j) tma_load_4d(xs + j * kTile, &maps.x, &bar_tma[st], 0, h, t0 + 128 * j, bi);
    };
    const int nh = h_end - h_begin;
    if (tid == 0) {
        issue(0);
        if (nh > 1) issue(1);
    }
    bool ok = true;
    const int t = tb * 128 + 32 * warp + lane;
    const bool tv = t < vrows;
    for (int k = 0; k < nh && ok; ++k) {
        const int h = h_begin + k, st = k & 1;
        float *cv = cumv + st * Q, *dv = dtv + st * Q;
        const float *cumg = p.cumA + ix_chunk(p, bi, h, c) * Q;
        for (int l = tid; l < Q; l += kThreads) {
            cv[l] = cumg[l];
            dv[l] = l < vrows ? p.dt[ix_dt(p, bi, h, t0 + l)] : 0.f;
        }
        tc_fence_before();
        ok = wait_all(&bar_tma[st], (uint32_t)((k >> 1) & 1), ok);
        tc_fence_after();
        if (tid == 0 && ok) {
            uint8_t *dys = sm + st * STG, *xs = dys + kTile;
            const uint32_t id = idesc_bf16(128, ncols, false, false);
            for (int ks = 0; ks < kP / 16; ++ks)
                mma_bf16(tm + DW, sdesc_kmajor(smem_u32(dys), ks, kTile), sdesc_kmajor(smem_u32(xs), ks, kTile), id,
                         ks > 0);
            mma_commit(&bar_mma);
        }
        ok = wait_all(&bar_mma, (uint32_t)(k & 1), ok);
        tc_fence_after();
        // the stage just consumed can be refilled with head k + 2
        if (tid == 0 && ok && k + 2 < nh) issue(k + 2);
        if (ok) {
            const float ct = cv[t];
            for (int s0 = 0; s0 < ncols; s0 += 32) {
                float dw[32], acc[32];
                tmem_ld32(tmem_addr(tm, 32 * warp, DW + s0), dw);
                if (k > 0) tmem_ld32(tmem_addr(tm, 32 * warp, ACC + s0), acc);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int s = s0 + j;
                    const float v = (tv && s <= t && s < vrows) ? dw[j] * dv[s] * __expf(ct - cv[s]) : 0.f;
                    acc[j] = (k > 0 ? acc[j] : 0.f) + v;
                }
                tmem_st32(tmem_addr(tm, 32 * warp, ACC + s0), acc);
            }
        }
        tc_fence_before();
        ok = __syncthreads_and(ok ? 1 : 0) != 0;
        tc_fence_after();
    }
    if (ok) {
        float *orow = out + (size_t)t * Q;
        for (int s0 = 0; s0 < ncols; s0 += 32) {
            float v[32];
            tmem_ld32(tmem_addr(tm, 32 * warp, ACC + s0), v);
            float4 *dst = reinterpret_cast<float4 *>(orow + s0);
#pragma unroll
            for (int j = 0; j < 8; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
    } else if (tid == 0) {
        flag_timeout(p);
    }
    tc_sync();
    if (warp == 0) tmem_dealloc(tm, NCOL);
}

// G2: CTA per (b, chunk, group, head slice).  TMEM: dC accumulators at
// [tb*128), dB accumulators at [NT*128 + mb*128).
//   slice 0 only:  dC += d_cb B        (A = d_cb K-major, B = B MN-major)
//                  dB += d_cb^T C      (A = d_cb MN-major view, B = C MN-major)
//   every slice:   dC += sum_h (dy_h exp(cumA_h)) s_in_h      (long-K over heads)
//                  dB += sum_h (x_h bbs_h) d_intra_h
// and writes the fp32 partial sums of the slice.
template <int Q>
__global__ void __launch_bounds__(kThreads) tc_bwd_dbc_kernel(const Params p, const __grid_constant__ TcMaps maps) {
    constexpr int NT = Q / 128;
    constexpr uint32_t XB = Q * 128, RB = Q * 128, SB = 64 * 128;
    constexpr uint32_t STG = 2 * XB + 4 * SB;  // dy, x, s_in (2 r-blocks), d_intra (2 r-blocks)
    constexpr uint32_t NCOL = NT == 2 ? 512 : 256;
    constexpr uint32_t DBCOL = NT * 128;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    float *fv = reinterpret_cast<float *>(sm + 2 * STG);  // [2][2][Q]: exp(cumA), bbs per stage
    __shared__ uint64_t bar_tma[2], bar_mma[2], bar_a;
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int idx = blockIdx.x;
    const int slice = idx % p.nslice;
    idx /= p.nslice;
    const int g = idx % p.G, c = (idx / p.G) % p.n, bi = idx / (p.G * p.n);
    const int t0 = c * Q;
    const int vrows = min(Q, valid_len_of(p, bi) - t0);
    const int per = (p.hpg + p.nslice - 1) / p.nslice;
    const int h_begin = g * p.hpg + slice * per;
    const int h_end = min(g * p.hpg + p.hpg, h_begin + per);
    const size_t pstride = (size_t)p.b * p.n * p.G * Q * kN;
    float *outC = p.dBC_part + ((size_t)slice * 2 + 0) * pstride + (((size_t)bi * p.n + c) * p.G + g) * (size_t)Q * kN;
    float *outB = p.dBC_part + ((size_t)slice * 2 + 1) * pstride + (((size_t)bi * p.n + c) * p.G + g) * (size_t)Q * kN;
    const bool do_k2 = slice == 0;
    const int nh = max(0, h_end - h_begin);
    if (vrows <= 0 || (!do_k2 && nh == 0)) {
        for (int i = tid; i < Q * kN; i += kThreads) {
            outC[i] = 0.f;
            outB[i] = 0.f;
        }
        return;
    }
    if (tid == 0) {
        mbar_init(&bar_tma[0], 1);
        mbar_init(&bar_tma[1], 1);
        mbar_init(&bar_mma[0], 1);
        mbar_init(&bar_mma[1], 1);
        mbar_init(&bar_a, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&s_tmem, NCOL);
    tc_sync();
    const uint32_t tm = s_tmem;
    bool ok = true;
    uint32_t pa = 0;  // bar_a phase
    bool have_acc = false;
    if (do_k2) {
        // d_cb (bf16, K-major [t][s] in 64-column blocks of Q rows) from the G1 partials
        uint8_t *dcb = sm, *BCs = sm + (uint32_t)Q * Q * 2;
        if (tid == 0) {
            mbar_arrive_expect_tx(&bar_a, 2 * RB);
            for (int rb = 0; rb < 2; ++rb)
                for (int j = 0; j < NT; ++j)
                    tma_load_4d(BCs + rb * RB + j * kTile, &maps.B, &bar_a, 64 * rb, g, t0 + 128 * j, bi);
        }
        const size_t cstride = (size_t)p.b * p.n * p.G * Q * Q;
        const float *part = p.d_cb + (((size_t)bi * p.n + c) * p.G + g) * (size_t)Q * Q;
        for (int i = tid; i < Q * (Q / 8); i += kThreads) {
            const int t = i / (Q / 8), s0 = 8 * (i % (Q / 8));
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.f;
            if (s0 <= t) {
                for (int sl = 0; sl < p.nslice_cb; ++sl) {
                    const float4 a = *reinterpret_cast<const float4 *>(part + sl * cstride + (size_t)t * Q + s0);
                    const float4 b = *reinterpret_cast<const float4 *>(part + sl * cstride + (size_t)t * Q + s0 + 4);
                    v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w;
                    v[4] += b.x; v[5] += b.y; v[6] += b.z; v[7] += b.w;
                }
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (s0 + e > t) v[e] = 0.f;
            }
            st_shared_v4(smem_u32(dcb + (s0 / 64) * RB) + sw128_chunk(t, (s0 % 64) / 8), pack_bf2(v[0], v[1]),
                         pack_bf2(v[2], v[3]), pack_bf2(v[4], v[5]), pack_bf2(v[6], v[7]));
        }
        ok = wait_all(&bar_a, pa, ok);
        pa ^= 1;
        if (ok && vrows < Q) {
            zero_rows_from(BCs, Q, vrows);
            zero_rows_from(BCs + RB, Q, vrows);
        }
        fence_async_smem();
        tc_sync();
        if (tid == 0 && ok) {
            const uint32_t id = idesc_bf16(128, kN, false, true);
            for (int tb = 0; tb < NT; ++tb)
                for (int ks = 0; ks < 8 * (tb + 1); ++ks)
                    mma_bf16(tm + tb * 128, sdesc_kmajor(smem_u32(dcb + tb * kTile), ks, RB),
                             sdesc_mnmajor(smem_u32(BCs), ks, RB), id, ks > 0);
            mma_commit(&bar_a);
        }
        ok = wait_all(&bar_a, pa, ok);
        pa ^= 1;
        tc_sync();
        // C into the same buffer, then dB += d_cb^T C
        if (tid == 0 && ok) {
            mbar_arrive_expect_tx(&bar_a, 2 * RB);
            for (int rb = 0; rb < 2; ++rb)
                for (int j = 0; j < NT; ++j)
                    tma_load_4d(BCs + rb * RB + j * kTile, &maps.C, &bar_a, 64 * rb, g, t0 + 128 * j, bi);
        }
        ok = wait_all(&bar_a, pa, ok);
        pa ^= 1;
        if (ok && vrows < Q) {
            zero_rows_from(BCs, Q, vrows);
            zero_rows_from(BCs + RB, Q, vrows);
        }
        fence_async_smem();
        tc_sync();
        if (tid == 0 && ok) {
            const uint32_t id = idesc_bf16(128, kN, true, true);
            for (int mb = 0; mb < NT; ++mb) {
                const uint32_t abase = smem_u32(dcb) + (uint32_t)(2 * mb) * RB + (uint32_t)(128 * mb * 128);
                const uint32_t bbase = smem_u32(BCs) + (uint32_t)(128 * mb * 128);
                for (int ks = 0; ks < (Q - 128 * mb) / 16; ++ks)
                    mma_bf16(tm + DBCOL + mb * 128, sdesc_mnmajor(abase, ks, RB), sdesc_mnmajor(bbase, ks, RB), id,
                             ks > 0);
            }
            mma_commit(&bar_a);
        }
        ok = wait_all(&bar_a, pa, ok);
        pa ^= 1;
        tc_sync();
        have_acc = true;
    }
    // ---- long-K part over the slice's heads (2-stage TMA pipeline)
    auto issue = [&](int k) {
        const int h = h_begin + k, st = k & 1;
        uint8_t *base = sm + st * STG;
        uint8_t *dys = base, *xs = base + XB, *sis = base + 2 * XB, *dis = sis + 2 * SB;
        const int sidx = (bi * p.n + c) * p.H + h;
        mbar_arrive_expect_tx(&bar_tma[st], STG);
        for (int j = 0; j < NT; ++j) {
            tma_load_4d(dys + j * kTile, &maps.dy, &bar_tma[st], 0, h, t0 + 128 * j, bi);
            tma_load_4d(xs + j * kTile, &maps.x, &bar_tma[st], 0, h, t0 + 128 * j, bi);
        }
        for (int rb = 0; rb < 2; ++rb) {
            tma_load_3d(sis + rb * SB, &maps.st, &bar_tma[st], 64 * rb, 0, sidx);
            tma_load_3d(dis + rb * SB, &maps.dst, &bar_tma[st], 64 * rb, 0, sidx);
        }
    };
    ok = __syncthreads_and(ok ? 1 : 0) != 0;
    if (tid == 0 && ok && nh > 0) {
        issue(0);
        if (nh > 1) issue(1);
    }
    for (int k = 0; k < nh && ok; ++k) {
        const int h = h_begin + k, st = k & 1;
        uint8_t *base = sm + st * STG;
        uint8_t *dys = base, *xs = base + XB, *sis = base + 2 * XB, *dis = sis + 2 * SB;
        float *ec = fv + st * 2 * Q, *bb = ec + Q;
        const float *cumg = p.cumA + ix_chunk(p, bi, h, c) * Q;
        const float cend = p.endA[ix_chunk(p, bi, h, c)];
        for (int l = tid; l < Q; l += kThreads) {
            const float cl = cumg[l];
            const bool v = l < vrows;
            ec[l] = v ? __expf(cl) : 0.f;
            bb[l] = v ? p.dt[ix_dt(p, bi, h, t0 + l)] * __expf(cend - cl) : 0.f;
        }
        ok = wait_all(&bar_tma[st], (uint32_t)((k >> 1) & 1), ok);
        if (ok) {
            scale_rows(dys, Q, ec, vrows);
            scale_rows(xs, Q, bb, vrows);
        }
        fence_async_smem();
        tc_sync();
        if (tid == 0 && ok) {
            const uint32_t id = idesc_bf16(128, kN, false, true);
            for (int tb = 0; tb < NT; ++tb)
                for (int ks = 0; ks < kP / 16; ++ks) {
                    const bool acc = have_acc || k > 0 || ks > 0;
                    mma_bf16(tm + tb * 128, sdesc_kmajor(smem_u32(dys + tb * kTile), ks, XB),
                             sdesc_mnmajor(smem_u32(sis), ks, SB), id, acc);
                    mma_bf16(tm + DBCOL + tb * 128, sdesc_kmajor(smem_u32(xs + tb * kTile), ks, XB),
                             sdesc_mnmajor(smem_u32(dis), ks, SB), id, acc);
                }
            mma_commit(&bar_mma[st]);
            // refill this stage with head k + 2 once its MMAs are done
            if (k + 2 < nh) {
                if (mbar_wait(&bar_mma[st], (uint32_t)((k >> 1) & 1))) issue(k + 2);
                else ok = false;
            }
        }
        ok = __syncthreads_and(ok ? 1 : 0) != 0;
    }
    // wait for the last MMAs
    if (nh > 0) {
        const int k = nh - 1, st = k & 1;
        ok = wait_all(&bar_mma[st], (uint32_t)((k >> 1) & 1), ok);
        if (nh > 1) {
            // head nh-2's MMAs were waited for only when a refill followed them
            const int k2 = nh - 2, st2 = k2 & 1;
            ok = wait_all(&bar_mma[st2], (uint32_t)((k2 >> 1) & 1), ok);
        }
    }
    tc_fence_after();
    if (ok) {
        for (int tb = 0; tb < NT; ++tb) {
            const int t = tb * 128 + 32 * warp + lane;
            for (int r0 = 0; r0 < kN; r0 += 32) {
                float v[32];
                tmem_ld32(tmem_addr(tm, 32 * warp, tb * 128 + r0), v);
                float4 *dC = reinterpret_cast<float4 *>(outC + (size_t)t * kN + r0);
#pragma unroll
                for (int j = 0; j < 8; ++j) dC[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                tmem_ld32(tmem_addr(tm, 32 * warp, DBCOL + tb * 128 + r0), v);
                float4 *dB = reinterpret_cast<float4 *>(outB + (size_t)t * kN + r0);
#pragma unroll
                for (int j = 0; j < 8; ++j) dB[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            }
        }
    } else if (tid == 0) {
        flag_timeout(p);
    }
    tc_sync();
    if (warp == 0) tmem_dealloc(tm, NCOL);
}

// G3: dB, dC = sum over slices of the G2 partials (fixed order), 0 past
// valid_len, cast to bf16.  One thread per 4 consecutive dstate entries.
template <int Q>
__global__ void tc_bwd_dbc_reduce(const Params p) {
    const size_t nvec = (size_t)p.b * p.L * p.G * (kN / 4);
    const size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    if (i >= nvec) return;
    const int r4 = (int)(i % (kN / 4));
    size_t rest = i / (kN / 4);
    const int g = (int)(rest % p.G);
    rest /= p.G;
    const int t = (int)(rest % p.L), bi = (int)(rest / p.L);
    const int c = t / Q, q = t % Q;
    const bool valid = t < valid_len_of(p, bi);
    float4 sc = make_float4(0.f, 0.f, 0.f, 0.f), sb = sc;
    if (valid) {
        const size_t pstride = (size_t)p.b * p.n * p.G * Q * kN;
        const size_t off = ((((size_t)bi * p.n + c) * p.G + g) * Q + q) * kN + 4 * r4;
        for (int sl = 0; sl < p.nslice; ++sl) {
            const float4 a = *reinterpret_cast<const float4 *>(p.dBC_part + (sl * 2 + 0) * pstride + off);
            const float4 b = *reinterpret_cast<const float4 *>(p.dBC_part + (sl * 2 + 1) * pstride + off);
            sc.x += a.x; sc.y += a.y; sc.z += a.z; sc.w += a.w;
            sb.x += b.x; sb.y += b.y; sb.z += b.z; sb.w += b.w;
        }
    }
    const size_t o = ix_bc(p, bi, t, g, 4 * r4);
    uint2 uc, ub;
    uc.x = pack_bf2(sc.x, sc.y);
    uc.y = pack_bf2(sc.z, sc.w);
    ub.x = pack_bf2(sb.x, sb.y);
    ub.y = pack_bf2(sb.z, sb.w);
    *reinterpret_cast<uint2 *>((bf16 *)p.dC + o) = uc;
    *reinterpret_cast<uint2 *>((bf16 *)p.dB + o) = ub;
}

// ====================================================================== host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
    });
    return fn;
}

cudaError_t encode(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                   const cuuint32_t *box) {
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// [b, L, H or G, 64 or 128] bf16 activations: boxes of 64 columns x 128 tokens.
cudaError_t map_tokens(CUtensorMap *m, const void *base, int b, int L, int heads, int width) {
    cuuint64_t dims[4] = {(cuuint64_t)width, (cuuint64_t)heads, (cuuint64_t)L, (cuuint64_t)b};
    cuuint64_t strides[3] = {(cuuint64_t)width * 2, (cuuint64_t)heads * width * 2, (cuuint64_t)L * heads * width * 2};
    cuuint32_t box[4] = {64, 1, 128, 1};
    return encode(m, base, 4, dims, strides, box);
}

// [b*n*H, P, N] bf16 chunk states: boxes of 64 dstate columns x 64 headdim rows.
cudaError_t map_states(CUtensorMap *m, const void *base, long long count) {
    cuuint64_t dims[3] = {(cuuint64_t)kN, (cuuint64_t)kP, (cuuint64_t)count};
    cuuint64_t strides[2] = {(cuuint64_t)kN * 2, (cuuint64_t)kP * kN * 2};
    cuuint32_t box[3] = {64, 64, 1};
    return encode(m, base, 3, dims, strides, box);
}

cudaError_t make_maps(const Params &p, TcMaps *mp, bool backward) {
    memset(mp, 0, sizeof(*mp));
    cudaError_t e;
    if ((e = map_tokens(&mp->x, p.x, p.b, p.L, p.H, kP)) != cudaSuccess) return e;
    if ((e = map_tokens(&mp->B, p.B, p.b, p.L, p.G, kN)) != cudaSuccess) return e;
    if ((e = map_tokens(&mp->C, p.C, p.b, p.L, p.G, kN)) != cudaSuccess) return e;
    if (p.states_bf && (e = map_states(&mp->st, p.states_bf, (long long)p.b * p.n * p.H)) != cudaSuccess) return e;
    if (backward) {
        if ((e = map_tokens(&mp->dy, p.dy, p.b, p.L, p.H, kP)) != cudaSuccess) return e;
        if (p.dstates_bf && (e = map_states(&mp->dst, p.dstates_bf, (long long)p.b * p.n * p.H)) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

template <typename K>
cudaError_t launch(K kernel, unsigned grid, size_t smem, cudaStream_t s, const Params &p, const TcMaps &maps) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, kThreads, smem, s>>>(p, maps);
    return cudaGetLastError();
}

constexpr size_t smem_k2(int Q) { return 1024 + 4 * (size_t)Q * 128; }
constexpr size_t smem_k3(int Q) { return 1024 + 3 * (size_t)Q * 128 + 4 * Q; }
constexpr size_t smem_k5(int Q) {
    return 1024 + 3 * (size_t)Q * 128 + 2 * 64 * 128 + (size_t)kTile * 2 * ((Q / 128) * (Q / 128 + 1) / 2) + 8 * Q;
}
constexpr size_t smem_blue(int Q) { return 1024 + 3 * (size_t)Q * 128 + 2 * 64 * 128 + 4 * Q; }
constexpr size_t smem_main(int Q) {
    return 1024 + 4 * (size_t)Q * 128 + 2 * 64 * 128 + 4 * (5 * Q + (Q / 128) * 4 * 2 * Q + 4);
}
// Padded above half of the SM's shared memory: a CTA holding 512 TMEM columns
// must never share its SM with another CTA of the same kernel.
constexpr size_t smem_dcb(int Q) {
    return (1024 + 2 * (size_t)kTile * (1 + Q / 128) + 4 * 4 * Q) > 120 * 1024
               ? 1024 + 2 * (size_t)kTile * (1 + Q / 128) + 4 * 4 * Q
               : 120 * 1024;
}
constexpr size_t smem_dbc(int Q) {
    return 1024 + 2 * (2 * (size_t)Q * 128 + 4 * 64 * 128) + 4 * 4 * Q;
}
static_assert(smem_main(256) <= 232448 && smem_main(256) > 116 * 1024, "main backward: one CTA per SM");
static_assert(smem_k2(256) > 116 * 1024, "K2 (512 TMEM columns): one CTA per SM");
static_assert(smem_k5(256) <= 232448, "K5 shared memory");
static_assert(smem_dbc(256) <= 232448, "group backward shared memory");
static_assert(2 * (size_t)256 * 256 + 2 * 256 * 128 <= 2 * (2 * (size_t)256 * 128 + 4 * 64 * 128),
              "d_cb + B tile must fit the two long-K stages");

}  // namespace

bool tc_supported(int64_t P, int64_t N, int64_t Q) { return P == kP && N == kN && (Q == 128 || Q == 256); }
int tc_dD_per(int64_t) { return 1; }
int tc_dcb_slices(const ssd_dims &d) {
    const long long hpg = d.nheads / d.ngroups;
    const long long n = (d.seqlen + d.chunk_len - 1) / d.chunk_len;
    const long long ctas = d.batch * n * d.ngroups * (d.chunk_len / 128);
    long long s = (2 * 152 + ctas - 1) / ctas;
    if (s < 1) s = 1;
    if (s > hpg) s = hpg;
    return (int)s;
}
int tc_group_slices(const ssd_dims &d) {
    const long long hpg = d.nheads / d.ngroups;
    const long long n = (d.seqlen + d.chunk_len - 1) / d.chunk_len;
    const long long ctas = d.batch * n * d.ngroups;
    long long s = (2 * 152 + ctas - 1) / ctas;
    if (s < 1) s = 1;
    if (s > hpg) s = hpg;
    return (int)s;
}

#define SSD_TC_DISPATCH(Q_, call) ((Q_) == 256 ? call(256) : call(128))

cudaError_t launch_tc_k2(const Params &p, cudaStream_t s) {
    TcMaps m;
    cudaError_t e = make_maps(p, &m, false);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(p.b * p.n * p.G);
#define CALL(Q) launch(tc_k2_kernel<Q>, grid, smem_k2(Q), s, p, m)
    return SSD_TC_DISPATCH(p.Q, CALL);
#undef CALL
}

cudaError_t launch_tc_k3(const Params &p, cudaStream_t s) {
    TcMaps m;
    cudaError_t e = make_maps(p, &m, false);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(p.b * p.n * p.H);
#define CALL(Q) launch(tc_k3_kernel<Q>, grid, smem_k3(Q), s, p, m)
    return SSD_TC_DISPATCH(p.Q, CALL);
#undef CALL
}

cudaError_t launch_tc_k5(const Params &p, cudaStream_t s) {
    TcMaps m;
    cudaError_t e = make_maps(p, &m, false);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(p.b * p.n * p.H);
#define CALL(Q) launch(tc_k5_kernel<Q>, grid, smem_k5(Q), s, p, m)
    return SSD_TC_DISPATCH(p.Q, CALL);
#undef CALL
}

cudaError_t launch_tc_bwd_blue(const Params &p, cudaStream_t s) {
    TcMaps m;
    cudaError_t e = make_maps(p, &m, true);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(p.b * p.n * p.H);
#define CALL(Q) launch(tc_bwd_blue_kernel<Q>, grid, smem_blue(Q), s, p, m)
    return SSD_TC_DISPATCH(p.Q, CALL);
#undef CALL
}

cudaError_t launch_tc_bwd_main(const Params &p, cudaStream_t s) {
    TcMaps m;
    cudaError_t e = make_maps(p, &m, true);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(p.b * p.n * p.H);
#define CALL(Q) launch(tc_bwd_main_kernel<Q>, grid, smem_main(Q), s, p, m)
    return SSD_TC_DISPATCH(p.Q, CALL);
#undef CALL
}

cudaError_t launch_tc_bwd_group(const Params &p, cudaStream_t s) {
    TcMaps m;
    cudaError_t e = make_maps(p, &m, true);
    if (e != cudaSuccess) return e;
    const unsigned g1 = (unsigned)(p.b * p.n * p.G * p.nslice_cb * (p.Q / 128));
    const unsigned g2 = (unsigned)(p.b * p.n * p.G * p.nslice);
#define CALL1(Q) launch(tc_bwd_dcb_kernel<Q>, g1, smem_dcb(Q), s, p, m)
#define CALL2(Q) launch(tc_bwd_dbc_kernel<Q>, g2, smem_dbc(Q), s, p, m)
    if ((e = SSD_TC_DISPATCH(p.Q, CALL1)) != cudaSuccess) return e;
    if ((e = SSD_TC_DISPATCH(p.Q, CALL2)) != cudaSuccess) return e;
#undef CALL1
#undef CALL2
    const size_t nvec = (size_t)p.b * p.L * p.G * (kN / 4);
    const unsigned g3 = (unsigned)((nvec + 255) / 256);
    if (p.Q == 256) tc_bwd_dbc_reduce<256><<<g3, 256, 0, s>>>(p);
    else tc_bwd_dbc_reduce<128><<<g3, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace ssd
