// ssd_tc.cu -- tcgen05 tensor-core kernels of the bf16 path (sm_103a).
//
// The dense contractions of the chunked scan run as tcgen05.mma (kind::f16,
// bf16 operands, fp32 accumulators in TMEM) on operands staged in shared
// memory: raw tiles of x, dy, B, C and the bf16 chunk states arrive by TMA
// (cp.async.bulk.tensor, 128-byte swizzle); operands that carry a per-token
// factor (the causal decay matrix W, the K3 / BLUE scales) are formed by the
// CTA's threads in registers and written to shared memory in the same
// swizzled layout, or -- for the decay matrix W of K5 and the ORANGE
// backward -- into TMEM as packed bf16 pairs, the MMA's A operand.  One
// elected thread issues the MMAs; the epilogues read TMEM with tcgen05.ld
// (warp w owns TMEM lanes 32(w%4)..32(w%4)+31; with 256 threads, warps w and
// w+4 split the columns).  K5 and the backward's ORANGE / K3 kernels loop
// over the heads of a group with the group's operands resident.
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
constexpr int kThreadsWide = 256;
constexpr int kTile = 16384;  // one [128 rows][64] bf16 SW128 tile
constexpr int kStatusTimeout = 5;

struct TcMaps {
    CUtensorMap x, dy, B, C, st, dst, cb, cbt, dcb, part, dx, y, cb64;
    CUtensorMap xs, Bs;    // chunk-state scan: x of 1 or 2 heads, both halves of B, 128 tokens
};

constexpr int kScanConsumers = 512;  // consumer threads of the chunk-state scan
// tokens per sub-stage of the chunk-state scan: 64 with two heads per CTA, 128 with one
__host__ __device__ constexpr int scan_tok(int hpc) { return hpc == 2 ? 64 : 128; }

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

// AND of `v` over the `nthreads` threads (whole warps) that use named barrier `id`.
__device__ __forceinline__ bool bar_and(int id, int nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pv, pr;\n\t"
        "setp.ne.u32 pv, %1, 0;\n\t"
        "bar.red.and.pred pr, %2, %3, pv;\n\t"
        "selp.u32 %0, 1, 0, pr;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// Barrier among the `nthreads` threads (whole warps) that use named barrier `id`.
__device__ __forceinline__ void bar_sync_n(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
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

// Zero rows [from, rows) of a tile of 128-byte rows, using the first `nthreads` threads.
__device__ __forceinline__ void zero_rows_from_n(uint8_t *tile, int rows, int from, int nthreads) {
    if (from >= rows) return;
    const uint32_t base = smem_u32(tile);
    for (int i = threadIdx.x + from * 8; i < rows * 8; i += nthreads)
        st_shared_v4(base + (uint32_t)i * 16u, 0u, 0u, 0u, 0u);
}

// Scale the 64 bf16 of row `row` (SW128 tile) in place by f; zero it when
// !valid (a select, so non-finite padding cannot leak).
__device__ __forceinline__ void scale_row_bf16(uint8_t *tile, int row, float f, bool valid) {
    const uint32_t base = smem_u32(tile);
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
        const uint32_t a = base + sw128_chunk(row, c8);
        if (!valid) {
            st_shared_v4(a, 0u, 0u, 0u, 0u);
            continue;
        }
        uint4 v = ld_shared_v4(a);
        v.x = pack_bf2(bf_lo(v.x) * f, bf_hi(v.x) * f);
        v.y = pack_bf2(bf_lo(v.y) * f, bf_hi(v.y) * f);
        v.z = pack_bf2(bf_lo(v.z) * f, bf_hi(v.z) * f);
        v.w = pack_bf2(bf_lo(v.w) * f, bf_hi(v.w) * f);
        st_shared_v4(a, v.x, v.y, v.z, v.w);
    }
}

// Same in packed bf16 pairs (the factor rounded to bf16 first): half the
// instructions, for operands whose bf16 rounding dominates anyway.
__device__ __forceinline__ void scale_row_bf16x2(uint8_t *tile, int row, float f, bool valid) {
    const uint32_t base = smem_u32(tile);
    const uint32_t f2 = pack_bf2(f, f);
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
        const uint32_t a = base + sw128_chunk(row, c8);
        if (!valid) {
            st_shared_v4(a, 0u, 0u, 0u, 0u);
            continue;
        }
        const uint4 v = ld_shared_v4(a);
        st_shared_v4(a, bmul2(v.x, f2), bmul2(v.y, f2), bmul2(v.z, f2), bmul2(v.w, f2));
    }
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

// Store 32 floats as 32 contiguous bf16 in global memory (64-byte aligned).
__device__ __forceinline__ void store_row32_bf16(bf16 *dst, const float *v) {
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
        uint4 u;
        u.x = pack_bf2(v[8 * c8 + 0], v[8 * c8 + 1]);
        u.y = pack_bf2(v[8 * c8 + 2], v[8 * c8 + 3]);
        u.z = pack_bf2(v[8 * c8 + 4], v[8 * c8 + 5]);
        u.w = pack_bf2(v[8 * c8 + 6], v[8 * c8 + 7]);
        reinterpret_cast<uint4 *>(dst)[c8] = u;
    }
}

// ====================================================================== K2
// CTA per (b, chunk, group, 128-row block tb), 256 threads.  Both products of
// the block are issued together and committed once, both operands K-major:
//   CB[t, s]   = sum_r C[t, r] B[s, r],  t in block tb, s < 128 (tb + 1)   (TMEM cols [0, N1))
//   CB^T[s, t] = sum_r B[s, r] C[t, r],  s in block tb, t >= 128 tb         (TMEM cols [N1, N1 + N2))
// stored in bf16 (they only ever feed bf16 MMA operands); CB^T serves the
// backward, whose ORANGE term works on rows s.  The block needs C blocks
// tb .. and B blocks .. tb, nothing else.  Epilogue: the two warps of a TMEM
// lane quadrant take alternate 64-column pieces.
template <int Q>
__global__ void __launch_bounds__(kThreadsWide) tc_k2_kernel(const Params p, const __grid_constant__ TcMaps maps) {
    constexpr int NT = Q / 128;
    constexpr uint32_t RB = Q * 128;  // one r-block ([Q rows][64])
    constexpr uint32_t NCOL = NT == 2 ? 512 : 256;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *Cs = sm, *Bs = sm + 2 * RB;
    __shared__ uint64_t bar_tma, bar_mma;
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, hf = warp >> 2;
    int idx = blockIdx.x;
    const int tb = idx % NT;
    idx /= NT;
    const int g = idx % p.G, c = (idx / p.G) % p.n, bi = idx / (p.G * p.n);
    const int t0 = c * Q;
    const int vrows = min(Q, valid_len_of(p, bi) - t0);
    if (vrows <= 0) return;  // consumers never read CB of chunks past valid_len
    const int N1 = 128 * (tb + 1), N2 = Q - 128 * tb;
    if (tid == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&s_tmem, NCOL);
    tc_sync();
    const uint32_t tm = s_tmem;
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar_tma, 2u * (uint32_t)(NT - tb) * kTile + 2u * (uint32_t)(tb + 1) * kTile);
        for (int rb = 0; rb < 2; ++rb) {
            for (int j = tb; j < NT; ++j)
                tma_load_4d(Cs + rb * RB + j * kTile, &maps.C, &bar_tma, 64 * rb, g, t0 + 128 * j, bi);
            for (int j = 0; j <= tb; ++j)
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
        const uint32_t i1 = idesc_bf16(128, N1, false, false), i2 = idesc_bf16(128, N2, false, false);
        for (int ks = 0; ks < kN / 16; ++ks)
            mma_bf16(tm, sdesc_kmajor(smem_u32(Cs + tb * kTile), ks, RB), sdesc_kmajor(smem_u32(Bs), ks, RB), i1,
                     ks > 0);
        for (int ks = 0; ks < kN / 16; ++ks)
            mma_bf16(tm + (uint32_t)N1, sdesc_kmajor(smem_u32(Bs + tb * kTile), ks, RB),
                     sdesc_kmajor(smem_u32(Cs + tb * kTile), ks, RB), i2, ks > 0);
        mma_commit(&bar_mma);
    }
    ok = wait_all(&bar_mma, 0, ok);
    tc_fence_after();
    if (ok) {
        // 64-column pieces, bf16, staged over the (now dead) operand tiles in the
        // 128-byte swizzled layout of the CB / CB^T maps and written by TMA
        const int row = 32 * q4 + lane;
        const int npc = (N1 + N2) / 64;
#pragma unroll 1
        for (int j = hf; j < npc; j += 2) {
            float v[64];
            tmem_ld64(tmem_addr(tm, 32 * q4, 64 * j), v);
            const uint32_t base = smem_u32(sm + j * kTile) + (uint32_t)row * 128u;
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
                st_shared_v4(base + (uint32_t)((c8 ^ (row & 7)) * 16), pack_bf2(v[8 * c8], v[8 * c8 + 1]),
                             pack_bf2(v[8 * c8 + 2], v[8 * c8 + 3]), pack_bf2(v[8 * c8 + 4], v[8 * c8 + 5]),
                             pack_bf2(v[8 * c8 + 6], v[8 * c8 + 7]));
        }
        fence_async_smem();
    } else if (tid == 0) {
        flag_timeout(p);
    }
    tc_sync();
    if (ok && tid == 0) {
        const int row0 = ((bi * p.n + c) * p.G + g) * Q + 128 * tb;
        for (int j = 0; j < (N1 + N2) / 64; ++j) {
            if (64 * j < N1) tma_store_2d(&maps.cb, sm + j * kTile, 64 * j, row0);
            else tma_store_2d(&maps.cbt, sm + j * kTile, 128 * tb + 64 * j - N1, row0);
        }
        bulk_commit();
        bulk_wait_all();
    }
    if (warp == 0) tmem_dealloc(tm, NCOL);
}

// ====================================================================== K3
// CTA per (b, chunk, group, head slice): 8 consumer warps and one TMA producer
// warp; B stays resident, x streams through a ring of NST stages.  Per head
//   intra[p, r] = sum_l B[l, r] (bbs[l] x[l, p]),   bbs = dt exp(cumA_last - cumA)
// as D[r, p] (M = dstate; A = B, MN-major; B operand = scaled x, MN-major)
// into one of two TMEM buffers, so the MMA of head k overlaps the epilogue of
// head k - 1.  Consumer thread t scales row t of x (scalars fetched into
// registers two heads ahead).  The producer refills a stage once the MMA that
// read it completes and issues head k's MMA once every consumer warp has
// scaled its rows and left the epilogue of head k - 2 (mbarriers the warps
// arrive on).  The scale sits on x, not B, so B is shared by all heads.  The
// bf16 state of a head is staged in one of two swizzled shared tiles and
// written by TMA tile stores (a row-per-thread epilogue would store 2 bytes
// per lane per column).
template <int Q>
__global__ void __launch_bounds__(kThreadsWide + 32, 1) tc_k3_kernel(const Params p, const __grid_constant__ TcMaps maps) {
    constexpr int NT = Q / 128;
    constexpr uint32_t XB = Q * 128, RB = Q * 128;
    constexpr int NST = 4;
    constexpr int NCONS = kThreadsWide;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *Bs = sm, *xst = sm + 2 * RB;  // B: 2 r-blocks of Q rows; x: NST stages
    uint8_t *stg = xst + NST * XB;         // two [P][N] bf16 state tiles (two 64 x 64 boxes each)
    constexpr uint32_t STT = kP * kN * 2;
    __shared__ uint64_t bar_res, bar_x[NST], bar_free[NST], bar_scaled[NST], bar_mma[2], bar_tfree[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_issued, s_landed, s_perr;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int idx = blockIdx.x;
    const int slice = idx % p.nslice_k3;
    idx /= p.nslice_k3;
    const int g = idx % p.G, c = (idx / p.G) % p.n, bi = idx / (p.G * p.n);
    const int t0 = c * Q;
    const int vrows = min(Q, valid_len_of(p, bi) - t0);
    const int per = (p.hpg + p.nslice_k3 - 1) / p.nslice_k3;
    const int h_begin = g * p.hpg + slice * per;
    const int nh = max(0, min(g * p.hpg + p.hpg, h_begin + per) - h_begin);
    if (nh == 0) return;
    if (vrows <= 0) {  // a chunk wholly past valid_len: zero intra-chunk states
        for (int k = 0; k < nh; ++k) {
            bf16 *out = p.states_bf + ix_state(p, bi, c, h_begin + k);
            for (int i = tid; i < kP * kN / 8; i += blockDim.x) reinterpret_cast<uint4 *>(out)[i] = make_uint4(0, 0, 0, 0);
        }
        return;
    }
    if (tid == 0) {
        mbar_init(&bar_res, 1);
        for (int i = 0; i < NST; ++i) {
            mbar_init(&bar_x[i], 1);
            mbar_init(&bar_free[i], 1);
            mbar_init(&bar_scaled[i], NCONS / 32);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_mma[i], 1);
            mbar_init(&bar_tfree[i], NCONS / 32);
        }
        mbar_fence_init();
        s_issued = 0;
        s_landed = 0;
        s_perr = 0;
    }
    if (warp == 0) tmem_alloc(&s_tmem, 128);
    tc_sync();
    const uint32_t tm = s_tmem;
    bool ok = true;
    if (warp == NCONS / 32) {
        // ---- producer: B once; x_k into stage k % NST once head k - NST's MMA is
        // done; head k's MMA once it is scaled and TMEM buffer k & 1 is free
        if (lane == 0) {
            auto load = [&](int k) {
                const int st = k % NST;
                mbar_arrive_expect_tx(&bar_x[st], XB);
                for (int j = 0; j < NT; ++j)
                    tma_load_4d(xst + st * XB + j * kTile, &maps.x, &bar_x[st], 0, h_begin + k, t0 + 128 * j, bi);
                s_issued = k + 1;
            };
            mbar_arrive_expect_tx(&bar_res, 2 * RB);
            for (int rb = 0; rb < 2; ++rb)
                for (int j = 0; j < NT; ++j)
                    tma_load_4d(Bs + rb * RB + j * kTile, &maps.B, &bar_res, 64 * rb, g, t0 + 128 * j, bi);
            for (int k = 0; k < NST && k < nh; ++k) load(k);
            for (int k = 0; k < nh; ++k) {
                const int st = k % NST;
                if (!mbar_wait(&bar_scaled[st], (uint32_t)((k / NST) & 1)) || s_perr) {
                    s_perr = 1;
                    break;
                }
                s_landed = k + 1;
                // the stage of head k - 1 is free once its MMA is done: head k - 1 + NST goes there
                if (k >= 1 && k - 1 + NST < nh) {
                    if (!mbar_wait(&bar_free[(k - 1) % NST], (uint32_t)(((k - 1) / NST) & 1))) {
                        s_perr = 1;
                        break;
                    }
                    load(k - 1 + NST);
                }
                if (k >= 2 && !mbar_wait(&bar_tfree[k & 1], (uint32_t)(((k - 2) >> 1) & 1))) {
                    s_perr = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t idesc = idesc_bf16(128, 64, true, true);
                for (int ks = 0; ks < Q / 16; ++ks)
                    mma_bf16(tm + 64 * (k & 1), sdesc_mnmajor(smem_u32(Bs), ks, RB),
                             sdesc_mnmajor(smem_u32(xst + st * XB), ks, XB), idesc, ks > 0);
                mma_commit(&bar_mma[k & 1]);
                mma_commit(&bar_free[st]);
            }
        }
    } else {
        // ---- consumers
        const int t = tid;
        const bool valid = t < vrows;
        float c_cur = 0.f, d_cur = 0.f, e_cur = 0.f, c_nx = 0.f, d_nx = 0.f, e_nx = 0.f;
        auto fetch = [&](int k, float &cc, float &dd, float &ce) {
            const size_t ck = ix_chunk(p, bi, h_begin + k, c);
            ce = p.endA[ck];
            cc = t < Q ? p.cumA[ck * Q + t] : 0.f;
            dd = valid ? p.dt[ix_dt(p, bi, h_begin + k, t0 + t)] : 0.f;
        };
        fetch(0, c_cur, d_cur, e_cur);
        if (nh > 1) fetch(1, c_nx, d_nx, e_nx);
        ok = mbar_wait(&bar_res, 0);
        if (ok && vrows < Q) {
            zero_rows_from_n(Bs, Q, vrows, NCONS);
            zero_rows_from_n(Bs + RB, Q, vrows, NCONS);
        }
        // epilogue mapping: TMEM lane = dstate r, columns = headdim p
        const int q4 = warp & 3, hf = warp >> 2;
        const int r = 32 * q4 + lane;
        // the loop ends only on a CTA-uniform status (the named barriers below
        // need every consumer warp), so no warp leaves early
        for (int k = 0; k <= nh; ++k) {
            if (k < nh) {
                const int st = k % NST;
                uint8_t *xs = xst + st * XB;
                const float b_row = d_cur * __expf(e_cur - c_cur);
                c_cur = c_nx;
                d_cur = d_nx;
                e_cur = e_nx;
                if (k + 2 < nh) fetch(k + 2, c_nx, d_nx, e_nx);
                ok = __all_sync(0xffffffffu, mbar_wait(&bar_x[st], (uint32_t)((k / NST) & 1)) && ok);  // warp-uniform
                if (ok && t < Q) scale_row_bf16(xs, t, b_row, valid);
                if (!ok) s_perr = 1;
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_scaled[st]);  // the producer issues head k's MMA
            }
            if (k > 0) {
                // ---- epilogue of head k - 1
                const int kk = k - 1;
                ok = __all_sync(0xffffffffu, mbar_wait(&bar_mma[kk & 1], (uint32_t)((kk >> 1) & 1)) && ok);
                tc_fence_after();
                float v[32];
                tmem_ld32(tmem_addr(tm, 32 * q4, 64 * (kk & 1) + 32 * hf), v);
                // TMEM buffer kk & 1 read: the MMA of head k + 1 may overwrite it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_tfree[kk & 1]);
                // state tile kk & 1 is free once the store of head kk - 2 has read it
                uint8_t *stile = stg + (kk & 1) * STT;
                if (tid == 0 && kk >= 2) bulk_wait_read_1();
                ok = bar_and(2, NCONS, ok);
                if (ok) {  // element (p, r): box r / 64, row p, 16-byte chunk (r % 64) / 8 swizzled by p
                    const uint32_t base = smem_u32(stile) + (uint32_t)(r >> 6) * (STT / 2);
                    const int rc = r & 63;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int pp = 32 * hf + j;
                        const uint32_t a = base + (uint32_t)pp * 128u + (uint32_t)((((rc >> 3) ^ (pp & 7)) << 4) + (rc & 7) * 2);
                        st_shared_u16(a, __bfloat16_as_ushort(__float2bfloat16_rn(v[j])));
                    }
                    fence_async_smem();
                }
                ok = bar_and(2, NCONS, ok);
                if (!ok) {
                    s_perr = 1;
                    break;
                }
                if (tid == 0) {
                    const int sidx = (bi * p.n + c) * p.H + h_begin + kk;
                    tma_store_3d(&maps.st, stile, 0, 0, sidx);
                    tma_store_3d(&maps.st, stile + STT / 2, 64, 0, sidx);
                    bulk_commit();
                }
            }
        }
    }
    tc_fence_before();
    ok = __syncthreads_and(ok && s_perr == 0 ? 1 : 0) != 0;
    tc_fence_after();
    if (!ok && tid == 0) flag_timeout(p);
    // loads issued for heads that were never consumed have to land before exit,
    // and the last MMA (its commit covers the producer's earlier ones)
    if (tid == 0)
        for (int k = s_landed; k < s_issued; ++k) mbar_wait(&bar_x[k % NST], (uint32_t)((k / NST) & 1));
    if (tid == 0 && s_landed > 0) mbar_wait(&bar_free[(s_landed - 1) % NST], (uint32_t)(((s_landed - 1) / NST) & 1));
    if (tid == 0) bulk_wait_all();
    tc_sync();
    if (warp == 0) tmem_dealloc(tm, 128);
}

// ====================================================================== fused K1 + K3 + K4
// The chunk-state scan: CTA per (b, pair of heads of one group) -- or per
// (b, head) when the problem has few heads -- looping over the chunks in
// order with the running states in registers, so that the intra-chunk states
// never leave the SM (burn-mamba, "combined_backward.rs": the K1 recompute of
// dA = dt * A and its inclusive cumsum, k3_ssd_chunk_state_extended, and the
// K4 recurrence s_{i+1} = exp(dA_end_i) s_i + intra_i).  Per chunk c and head e:
//   cumA   inclusive cumsum of dt * A over the chunk (each lane sums Q / 32
//          consecutive tokens, a warp scan adds the lanes' sums), written to
//          the workspace with endA = cumA[Q - 1], and bbs = dt exp(endA - cumA)
//          into a table;
//   intra  intra[r, p] = sum_l B[l, r] (bbs[l] x[l, p]): one MMA accumulation
//          over sub-stages of 64 or 128 tokens (M = dstate, A = B, B = the scaled x of
//          the CTA's heads side by side, N = 64 per head, both MN-major) into
//          one of two TMEM buffers, so the MMAs of chunk c overlap the
//          epilogue of chunk c - 1;
//   carry  s_in_c = s goes to the workspace in bf16 for K5 and the backward,
//          then s <- exp(endA_c) s + intra_c in fp32 registers: consumer thread
//          (warp w, lane quadrant q4 = w % 4, column quarter cq = w / 4) keeps the
//          16 entries (p = 16 cq + j, r = 32 q4 + lane) of each head.
// Roles, handing over through mbarriers only (no CTA-wide barrier in the loop):
// 16 consumer warps scale the x rows of each sub-stage and run the carry; one
// thread issues the MMAs, one issues the TMA loads (one box for the x of both
// heads, one for both 64-column halves of B) into a ring of NSS stages, and
// one warp per head runs the scans up to NTAB chunks ahead.  The chain over chunks is
// serial, so the kernel lives on the depth of its ring: one CTA per SM, and
// two heads per CTA when there are enough heads to fill the SMs that way,
// which halves the B traffic; then 64-token sub-stages (a ring six deep),
// else 128-token ones (four deep), the faster of the two in each case on GB300.  Chunks wholly past valid_len load nothing:
// their cumA and endA are 0 and the states pass through them unchanged.
template <int HPC>
struct ScanGeom {
    static constexpr int TOK = scan_tok(HPC);              // tokens per sub-stage
    static constexpr uint32_t XS = TOK * 128;              // x of one head, one sub-stage: [TOK tokens][64]
    static constexpr uint32_t BS = TOK * 128;              // one 64-column half of B of a sub-stage
    static constexpr uint32_t SST = HPC * XS + 2 * BS;    // one stage
    static constexpr int NSS = HPC == 2 ? 6 : 4;          // ring depth (192 KB)
    static constexpr int NTAB = 4;                        // chunks of scan tables
    static constexpr size_t smem = 1024 + (size_t)NSS * SST;
};

template <int Q, int HPC>
__global__ void __launch_bounds__(kScanConsumers + 128, 1)
    tc_state_scan_kernel(const Params p, const __grid_constant__ TcMaps maps, int write_final) {
    using Gm = ScanGeom<HPC>;
    constexpr int TOK = Gm::TOK;
    constexpr int SPC = Q / TOK;  // sub-stages per chunk
    constexpr int NSS = Gm::NSS, NTAB = Gm::NTAB;
    constexpr uint32_t XS = Gm::XS, BS = Gm::BS, SST = Gm::SST;
    constexpr uint32_t BOFF = HPC * XS;   // B within a stage
    constexpr int NCW = kScanConsumers / 32;  // consumer warps
    constexpr int W_MMA = NCW, W_LOAD = NCW + 1, W_SCAN = NCW + 2;
    constexpr int NPX = HPC * TOK * 8, NPB = 2 * TOK * 8;  // 16-byte pieces of x, of B per sub-stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = align1024(smem_raw);
    __shared__ uint64_t bar_full[NSS], bar_scaled[NSS], bar_free[NSS], bar_mma[2], bar_tfree[2];
    __shared__ uint64_t bar_tab[NTAB], bar_tabfree[NTAB];
    __shared__ uint32_t s_tmem;
    __shared__ int s_issued, s_mma, s_perr;
    __shared__ float s_bbs[NTAB][HPC][Q];
    __shared__ float s_ea[NTAB][HPC];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // CTA -> (b, group, first head); a group with an odd head count ends in a one-head CTA
    const int cpg = (p.hpg + HPC - 1) / HPC;  // CTAs per (b, group)
    const int bg = blockIdx.x / cpg, g = bg % p.G, bi = bg / p.G;
    const int h0 = g * p.hpg + (blockIdx.x % cpg) * HPC;
    const int nh = min(HPC, g * p.hpg + p.hpg - h0);
    const int V = valid_len_of(p, bi);
    const int nv = (V + Q - 1) / Q;  // chunks holding a valid token (a prefix)
    const int U = nv * SPC;          // sub-stages loaded and multiplied
    // the backward's first kernel also clears the arrival counters (unless K1 ran first:
    // then K1 did that, reported valid_len, and wrote cumA / endA, which the scan reads)
    if (!p.cumA_given) {
        const int gs = gridDim.x * blockDim.x, i0 = blockIdx.x * blockDim.x + tid;
        if (p.cb_count)
            for (int i = i0; i < p.n_count; i += gs) p.cb_count[i] = 0;
        if (p.fin_count)
            for (int i = i0; i < p.H; i += gs) p.fin_count[i] = 0;
        // one CTA per sample reports a valid_len entry outside [0, L] (it is clamped)
        if (h0 == 0 && tid == 0 && valid_len_out_of_range(p, bi)) atomicAdd(p.status + kStatusValidLen, 1);
    }
    if (tid == 0) {
        for (int i = 0; i < NSS; ++i) {
            mbar_init(&bar_full[i], 1);
            mbar_init(&bar_scaled[i], NCW);
            mbar_init(&bar_free[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_mma[i], 1);
            mbar_init(&bar_tfree[i], NCW);
        }
        for (int i = 0; i < NTAB; ++i) {
            mbar_init(&bar_tab[i], 32 * HPC);
            mbar_init(&bar_tabfree[i], NCW);
        }
        mbar_fence_init();
        s_issued = 0;
        s_mma = 0;
        s_perr = 0;
    }
    // TMEM: buffer k & 1 at columns 64 HPC (k & 1), head e at + 64 e
    constexpr uint32_t NCOL = HPC == 2 ? 256 : 128;
    if (warp == 0) tmem_alloc(&s_tmem, NCOL);
    tc_sync();
    const uint32_t tm = s_tmem;
    bool ok = true;
    if (warp == W_MMA) {
        // ---- MMA issuer: sub-stage u once every consumer warp has scaled it
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(128, 64 * nh, true, true);
            for (int u = 0; u < U; ++u) {
                const int st = u % NSS, k = u / SPC, j = u % SPC;
                if (!mbar_wait(&bar_scaled[st], (uint32_t)((u / NSS) & 1)) || s_perr) {
                    s_perr = 1;
                    break;
                }
                // TMEM buffer k & 1 is free once the epilogue of chunk k - 2 has read it
                if (j == 0 && k >= 2 && !mbar_wait(&bar_tfree[k & 1], (uint32_t)(((k - 2) >> 1) & 1))) {
                    s_perr = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t base = smem_u32(ring + st * SST);
                for (int ks = 0; ks < TOK / 16; ++ks)
                    mma_bf16(tm + 64 * HPC * (k & 1), sdesc_mnmajor(base + BOFF, ks, BS), sdesc_mnmajor(base, ks, XS),
                             idesc, j > 0 || ks > 0);
                mma_commit(&bar_free[st]);
                if (j == SPC - 1) mma_commit(&bar_mma[k & 1]);
                s_mma = u + 1;
            }
        }
    } else if (warp == W_LOAD) {
        // ---- TMA loader: stage u % NSS once the MMAs of sub-stage u - NSS are done
        if (lane == 0) {
            for (int u = 0; u < U; ++u) {
                const int st = u % NSS, t = (u / SPC) * Q + TOK * (u % SPC);
                if (u >= NSS && !mbar_wait(&bar_free[st], (uint32_t)((u / NSS - 1) & 1))) {
                    s_perr = 1;
                    break;
                }
                uint8_t *dst = ring + st * SST;
                mbar_arrive_expect_tx(&bar_full[st], SST);
                tma_load_4d(dst, &maps.xs, &bar_full[st], 0, t, h0, bi);
                tma_load_5d(dst + BOFF, &maps.Bs, &bar_full[st], 0, t, 0, g, bi);
                s_issued = u + 1;
            }
        }
    } else if (warp >= W_SCAN) {
        // ---- scans: warp W_SCAN + e scans head e of chunk c into table c % NTAB, up to
        // NTAB chunks ahead.  Lane l holds tokens 32 i + l (i < TPL), so that the dt
        // loads (a chunk ahead), the cumA stores and the table stores are whole
        // 128-byte rows: one warp scan per 32 tokens, carried across the chunk.
        constexpr int TPL = Q / 32;
        const int e = warp - W_SCAN;
        const bool live = e < nh;
        const float Ah = live ? p.A[h0 + e] : 0.f;
        const float *dtrow = p.dt + ix_dt(p, bi, live ? h0 + e : h0, 0);
        auto fetch = [&](int c, float *v) {
            const int vr = min(Q, V - c * Q);
#pragma unroll
            for (int i = 0; i < TPL; ++i) {
                const int q = 32 * i + lane;
                v[i] = (live && q < vr) ? dtrow[c * Q + q] : 0.f;
            }
        };
        float vn[TPL];
        fetch(0, vn);
        for (int c = 0; c < p.n; ++c) {
            const int slot = c % NTAB;
            float v[TPL];
#pragma unroll
            for (int i = 0; i < TPL; ++i) v[i] = vn[i];
            if (c + 1 < p.n) fetch(c + 1, vn);
            if (c >= NTAB && !__all_sync(0xffffffffu, mbar_wait(&bar_tabfree[slot], (uint32_t)((c / NTAB - 1) & 1)))) {
                s_perr = 1;
                break;
            }
            if (live && p.cumA_given) {  // K1 has written cumA and endA: read them
                const int vr = min(Q, V - c * Q);
                const size_t ck = ix_chunk(p, bi, h0 + e, c);
                const float endA = p.endA[ck];
#pragma unroll
                for (int i = 0; i < TPL; ++i) {
                    const int q = 32 * i + lane;
                    s_bbs[slot][e][q] = q < vr ? v[i] * __expf(endA - p.cumA[ck * Q + q]) : 0.f;
                }
                if (lane == 0) s_ea[slot][e] = __expf(endA);
            } else if (live) {
                const int vr = min(Q, V - c * Q);
                float cum[TPL], run = 0.f;
#pragma unroll
                for (int i = 0; i < TPL; ++i) {
                    float incl = v[i] * Ah;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float w = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl += w;
                    }
                    cum[i] = run + incl;
                    run += __shfl_sync(0xffffffffu, incl, 31);
                }
                const float endA = run;
                const size_t ck = ix_chunk(p, bi, h0 + e, c);
#pragma unroll
                for (int i = 0; i < TPL; ++i) {
                    const int q = 32 * i + lane;
                    p.cumA[ck * Q + q] = cum[i];
                    s_bbs[slot][e][q] = q < vr ? v[i] * __expf(endA - cum[i]) : 0.f;
                }
                if (lane == 0) {
                    p.endA[ck] = endA;
                    s_ea[slot][e] = __expf(endA);
                }
            }
            mbar_arrive(&bar_tab[slot]);
        }
    } else if (warp < NCW) {
        // ---- consumers
        const int q4 = warp & 3, cq = warp >> 2;
        const int r = 32 * q4 + lane;
        float s[HPC][16];
#pragma unroll
        for (int e = 0; e < HPC; ++e) {
            const size_t bh = (size_t)bi * p.H + h0 + e;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                s[e][j] = (p.init && e < nh) ? p.init[(bh * kP + 16 * cq + j) * kN + r] : 0.f;
        }
        for (int c = 0; c <= p.n && ok; ++c) {
            if (c < p.n) {
                const int slot = c % NTAB, vr = min(Q, V - c * Q);
                ok = __all_sync(0xffffffffu, mbar_wait(&bar_tab[slot], (uint32_t)((c / NTAB) & 1)));
                // ---- K3 operands: scale x rows by bbs (packed bf16 pairs), zero rows past valid_len.
                // Thread i takes the 16-byte pieces i, i + 512, ... (32 consecutive pieces:
                // four whole 128-byte rows, no bank conflict; the 128-byte swizzle permutes
                // pieces within a row, so one scale per row).
                for (int j = 0; j < SPC && c < nv && ok; ++j) {
                    const int u = c * SPC + j, st = u % NSS;
                    const uint32_t sb = smem_u32(ring + st * SST);
                    ok = __all_sync(0xffffffffu, mbar_wait(&bar_full[st], (uint32_t)((u / NSS) & 1)));
                    if (!ok) break;
#pragma unroll
                    for (int pi = tid; pi < NPX; pi += kScanConsumers) {
                        const int e = pi / (TOK * 8), row = (pi >> 3) % TOK, tl = TOK * j + row;
                        if (e >= nh) continue;
                        const uint32_t a = sb + e * XS + (uint32_t)row * 128u + (uint32_t)(pi & 7) * 16u;
                        if (tl >= vr) {
                            st_shared_v4(a, 0u, 0u, 0u, 0u);
                            continue;
                        }
                        const float f = s_bbs[slot][e][tl];
                        const uint32_t f2 = pack_bf2(f, f);
                        const uint4 v0 = ld_shared_v4(a);
                        st_shared_v4(a, bmul2(v0.x, f2), bmul2(v0.y, f2), bmul2(v0.z, f2), bmul2(v0.w, f2));
                    }
                    if (TOK * j + TOK > vr) {  // B rows past valid_len (both halves)
#pragma unroll
                        for (int pi = tid; pi < NPB; pi += kScanConsumers) {
                            const int row = (pi >> 3) % TOK;
                            if (TOK * j + row >= vr)
                                st_shared_v4(sb + BOFF + (uint32_t)(pi / (TOK * 8)) * BS + (uint32_t)row * 128u +
                                                 (uint32_t)(pi & 7) * 16u,
                                             0u, 0u, 0u, 0u);
                        }
                    }
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar_scaled[st]);  // the MMA thread issues the sub-stage
                }
                if (!ok) break;
            }
            if (c > 0) {
                // ---- K4 step of chunk k = c - 1: s_in_k = s out, s <- exp(endA_k) s + intra_k,
                // one head at a time (16 accumulator values live at once)
                const int k = c - 1, kslot = k % NTAB;
                const bool live = k < nv;
                if (live) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&bar_mma[k & 1], (uint32_t)((k >> 1) & 1)));
                    if (!ok) break;
                    tc_fence_after();
                }
#pragma unroll
                for (int e = 0; e < HPC; ++e) {
                    float v[16];
                    if (live && e < nh) {
                        tmem_ld16(tmem_addr(tm, 32 * q4, 64 * (HPC * (k & 1) + e) + 16 * cq), v);
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] = 0.f;
                    }
                    if (e < nh) {
                        // s_in_k: for each p the warp's lanes write 32 consecutive r (64 bytes)
                        bf16 *dst = p.states_bf + ix_state(p, bi, k, h0 + e) + (size_t)(16 * cq) * kN + r;
#pragma unroll
                        for (int j = 0; j < 16; ++j) dst[(size_t)j * kN] = __float2bfloat16_rn(s[e][j]);
                        const float a = s_ea[kslot][e];
#pragma unroll
                        for (int j = 0; j < 16; ++j) s[e][j] = fmaf(a, s[e][j], v[j]);
                    }
                }
                if (live) {
                    // TMEM buffer k & 1 read: the MMAs of chunk k + 2 may overwrite it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar_tfree[k & 1]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_tabfree[kslot]);  // table of chunk k no longer read
            }
        }
        if (!ok) s_perr = 1;
        if (ok && write_final && p.final_state) {
#pragma unroll
            for (int e = 0; e < HPC; ++e) {
                if (e >= nh) break;
                const size_t bh = (size_t)bi * p.H + h0 + e;
#pragma unroll
                for (int j = 0; j < 16; ++j) p.final_state[(bh * kP + 16 * cq + j) * kN + r] = s[e][j];
            }
        }
    }
    tc_fence_before();
    ok = __syncthreads_and(ok && s_perr == 0 ? 1 : 0) != 0;
    tc_fence_after();
    if (!ok && tid == 0) flag_timeout(p);
    if (tid == 0) {
        // the latest load of every stage has to land before exit (one not consumed
        // after an error), and the last MMAs have to complete (they complete in order)
        for (int u = max(0, s_issued - NSS); u < s_issued; ++u) mbar_wait(&bar_full[u % NSS], (uint32_t)((u / NSS) & 1));
        if (s_mma > 0) mbar_wait(&bar_free[(s_mma - 1) % NSS], (uint32_t)(((s_mma - 1) / NSS) & 1));
    }
    tc_sync();
    if (warp == 0) tmem_dealloc(tm, NCOL);
}

// ====================================================================== K5
// CTA per (b, chunk, group, head slice), 256 threads, looping over the slice's
// heads with one CTA barrier per head.  C (BLUE's A operand) and the bf16 CB
// tiles stay resident in shared memory.  One thread issues the ORANGE MMAs and
// another the BLUE MMAs of a head, each committing to its own mbarrier.  W of
// t-block 0 has two TMEM buffers, so the next head's t-block-0 units (and its
// scalar tables) are built while this head's ORANGE MMAs run.  x of this head
// is requested as soon as the previous head's ORANGE MMAs are done; once its
// BLUE MMAs are done too, the previous head's epilogue writes y into a staging
// tile and the (now dead) s_in buffer, from which TMA tile stores take it, and
// s_in of this head follows.  The CB tiles whose upper 64 rows are zero (the
// upper 64-column group of each diagonal 128-block) are kept as 64-row tiles,
// which makes room for the staging tile.
// Per-head scalars are prefetched two heads ahead.  Per 128-row t-block tb:
//   ORANGE (TMEM cols tb*64):        W[tb] (A operand in TMEM) x  (x MN-major)
//   BLUE   (TMEM cols NT*64+tb*64):  C[tb] (K-major)            s_in (K-major)
// y = ORANGE + exp(cumA_t) * BLUE + D x, W[t, s] = CB[t, s] exp(cumA_t - cumA_s) dt_s
// (s <= t), stored to TMEM as packed bf16 pairs.  The decay is factored
// through pivots (both factors <= 1): cumA[64 sb + 63] for a 64 x 64 block
// strictly below the diagonal, cumA[16 v + 15] for a 16-wide sub-block left of
// the row's own inside a diagonal block.  The row's own 16-wide sub-block is
// factored through its first position when the sub-block's whole decay span
// stays below e^64 (a row factor <= 1 times a column factor <= e^64, both
// finite in bf16); a sub-block with a larger span takes direct exponentials.
template <int Q>
__global__ void __launch_bounds__(kThreadsWide, 1) tc_k5_kernel(const Params p, const __grid_constant__ TcMaps maps) {
    constexpr int NT = Q / 128;
    constexpr uint32_t XB = Q * 128, RB = Q * 128, SB = 64 * 128;
    constexpr int NWT = NT * (NT + 1);  // CB tiles: tb0 2, tb1 4
    constexpr uint32_t NCOL = NT == 2 ? 512 : 256;
    // TMEM: ORANGE | BLUE accumulators, W of t-block 1 (4 units), two buffers of
    // W of t-block 0 (2 units each; head k builds into one while the MMAs of
    // head k - 1 read the other)
    constexpr uint32_t OCOL = 0, BCOL = NT * 64, W1COL = 2 * NT * 64, W0COL = W1COL + (NT - 1) * 128;
    static_assert(W0COL + 128 == NCOL, "K5 TMEM columns");
    constexpr int NSC = 3;              // scalar buffers: staged two heads ahead
    // per-head tables (32-bit words): cum Q | dt Q | gcol pairs Q/2 | T16 pairs (Q/64) x 4 x 32 | piv 8 |
    // own-sub-block pairs Q/2 | own-sub-block fast flags Q/16
    constexpr int GOFF = 2 * Q, TOFF = GOFF + Q / 2, POFF = TOFF + (Q / 64) * 128;
    constexpr int OOFF = POFF + 8, FLOFF = OOFF + Q / 2;
    constexpr int FST = FLOFF + Q / 16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    // C | CB tiles (NWT - NT full, NT lower halves) | x | s_in | y staging tile | scalar tables
    uint8_t *Cs = sm, *CBf = Cs + 2 * RB, *CBh = CBf + (NWT - NT) * kTile, *xs = CBh + NT * (kTile / 2);
    uint8_t *Ss = xs + XB, *Ys = Ss + 2 * SB;
    float *fbuf = reinterpret_cast<float *>(Ys + kTile);  // [NSC][FST]
    // CB tile (t-block tb, 64-column group sb): its upper 64 rows are zero when sb = 2 tb + 1, and
    // only its lower half is stored, addressed as if the whole tile were there (rows >= 64 read)
    auto cb_tile = [&](int tb, int sb) -> uint8_t * {
        return sb == 2 * tb + 1 ? CBh + tb * (kTile / 2) - kTile / 2 : CBf + (tb * (tb + 1) + sb - tb) * kTile;
    };
    __shared__ uint64_t bar_res, bar_x, bar_s, bar_o, bar_b, bar_cb;
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, hf = warp >> 2;
    int idx = blockIdx.x;
    const int slice = idx % p.nslice_k5;
    idx /= p.nslice_k5;
    const int g = idx % p.G, c = (idx / p.G) % p.n, bi = idx / (p.G * p.n);
    const int t0 = c * Q;
    const int vrows = min(Q, valid_len_of(p, bi) - t0);
    const int per = (p.hpg + p.nslice_k5 - 1) / p.nslice_k5;
    const int h_begin = g * p.hpg + slice * per;
    const int h_end = min(g * p.hpg + p.hpg, h_begin + per);
    const int nh = h_end - h_begin;
    bf16 *Y = (bf16 *)p.y;
    if (nh <= 0) return;
    if (vrows <= 0) {
        const int rows = min(Q, p.L - t0);
        for (int hh = h_begin; hh < h_end; ++hh)
            for (int i = tid; i < rows * (kP / 8); i += kThreadsWide)
                reinterpret_cast<uint4 *>(Y + ix_x(p, bi, t0 + i / 8, hh, 0))[i % 8] = make_uint4(0, 0, 0, 0);
        return;
    }
    // raw per-head scalars cumA, dt (0 past valid_len): fetched into registers
    // (thread l holds token l) one head before they are staged in buffer `b`,
    // so the global load latency is hidden behind a whole head's work
    float r_cum = 0.f, r_dt = 0.f;
    auto fetch = [&](int k) {
        const int h = h_begin + k;
        if (tid < Q) {
            r_cum = p.cumA[ix_chunk(p, bi, h, c) * Q + tid];
            r_dt = tid < vrows ? p.dt[ix_dt(p, bi, h, t0 + tid)] : 0.f;
        }
    };
    auto stash = [&](int b) {
        float *f = fbuf + b * FST;
        if (tid < Q) {
            f[tid] = r_cum;
            f[Q + tid] = r_dt;
        }
    };
    // column tables from the raw values (visible after a barrier), as bf16 pairs:
    //   gcol[s]       = dt_s exp(piv_g - cumA_s), piv_g = cumA[64 g + 63] of s's 64-group g
    //   T16[g][u][s'] = dt_s exp(P_u - cumA_s) for s' = s - 64 g < 16 u, else 0, where
    //                   P_u = cumA[64 g + 16 u - 1] ends the 16-wide sub-blocks left of u
    auto derive = [&](int b) {
        float *f = fbuf + b * FST;
        uint32_t *f2 = reinterpret_cast<uint32_t *>(f);
        for (int e = tid; e < Q / 2; e += kThreadsWide) {
            const int s = 2 * e;
            const float pv = f[s | 63];
            f2[GOFF + e] = pack_bf2(f[Q + s] * __expf(pv - f[s]), f[Q + s + 1] * __expf(pv - f[s + 1]));
        }
        for (int e = tid; e < (Q / 64) * 128; e += kThreadsWide) {
            const int gb = e >> 7, u = (e >> 5) & 3, s = 64 * gb + 2 * (e & 31);
            float lo = 0.f, hi = 0.f;
            if (2 * (e & 31) < 16 * u) {
                const float pv = f[64 * gb + 16 * u - 1];
                lo = f[Q + s] * __expf(pv - f[s]);
                hi = f[Q + s + 1] * __expf(pv - f[s + 1]);
            }
            f2[TOFF + e] = pack_bf2(lo, hi);
        }
        for (int j = tid; j < Q / 64; j += kThreadsWide) f[POFF + j] = f[64 * j + 63];
        //   own[s] = dt_s exp(cumA[16 v] - cumA_s) for s in sub-block v (>= 1, <= e^64 where used)
        for (int e = tid; e < Q / 2; e += kThreadsWide) {
            const int s = 2 * e;
            const float pv = f[s & ~15];
            f2[OOFF + e] = pack_bf2(f[Q + s] * __expf(pv - f[s]), f[Q + s + 1] * __expf(pv - f[s + 1]));
        }
        for (int v = tid; v < Q / 16; v += kThreadsWide) f[FLOFF + v] = f[16 * v] - f[16 * v + 15] < 64.f ? 1.f : 0.f;
    };
    auto issue_x = [&](int h) {
        mbar_arrive_expect_tx(&bar_x, XB);
        for (int j = 0; j < NT; ++j) tma_load_4d(xs + j * kTile, &maps.x, &bar_x, 0, h, t0 + 128 * j, bi);
    };
    auto issue_s = [&](int h) {
        const int sidx = (bi * p.n + c) * p.H + h;
        mbar_arrive_expect_tx(&bar_s, 2 * SB);
        for (int rb = 0; rb < 2; ++rb) tma_load_3d(Ss + rb * SB, &maps.st, &bar_s, 64 * rb, 0, sidx);
    };
    if (tid == 0) {
        mbar_init(&bar_res, 1);
        mbar_init(&bar_x, 1);
        mbar_init(&bar_s, 1);
        mbar_init(&bar_o, 1);
        mbar_init(&bar_b, 1);
        mbar_init(&bar_cb, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&s_tmem, NCOL);
    tc_sync();
    const uint32_t tm = s_tmem;
    // ---- K2 prologue: CB = C B^T of the chunk and group (burn-mamba "K2 -- CB
    // matrix used in K5 ORANGE"), once per CTA for all of its heads.  C and B
    // come in by TMA (B into the CB tile region when it fits there, else into
    // the x / s_in / staging region, and then the first head's x and s_in wait
    // until CB is out of TMEM); per t-block tb one MMA accumulation (both
    // operands K-major) gives CB[t, s] for s < 128 (tb + 1) in TMEM columns
    // [64 tb (tb + 1), 64 (tb + 1) (tb + 2)), which the threads round to bf16
    // into the swizzled CB tiles the W build reads.
    constexpr bool B_IN_CB = (NWT - NT) * kTile + NT * (kTile / 2) >= 2 * RB;
    uint8_t *Bsm = B_IN_CB ? CBf : xs;
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar_res, 4 * RB);
        for (int j = 0; j < NT; ++j)
            for (int rb = 0; rb < 2; ++rb) {
                tma_load_4d(Cs + rb * RB + j * kTile, &maps.C, &bar_res, 64 * rb, g, t0 + 128 * j, bi);
                tma_load_4d(Bsm + rb * RB + j * kTile, &maps.B, &bar_res, 64 * rb, g, t0 + 128 * j, bi);
            }
        if (B_IN_CB) {
            issue_x(h_begin);
            issue_s(h_begin);
        }
    }
    fetch(0);
    stash(0);
    if (nh > 1) {
        fetch(1);
        stash(1);
    }
    if (nh > 2) fetch(2);
    bool ok = wait_all(&bar_res, 0, true);  // publishes the raw scalars of heads 0 and 1
    if (ok && vrows < Q) {
        for (int rb = 0; rb < 2; ++rb) {
            zero_rows_from(Cs + rb * RB, Q, vrows);
            zero_rows_from(Bsm + rb * RB, Q, vrows);
        }
    }
    fence_async_smem();
    tc_sync();
    if (tid == 0 && ok) {
        for (int tb = 0; tb < NT; ++tb) {
            const uint32_t id = idesc_bf16(128, 128 * (tb + 1), false, false);
            for (int ks = 0; ks < kN / 16; ++ks)
                mma_bf16(tm + (uint32_t)(64 * tb * (tb + 1)), sdesc_kmajor(smem_u32(Cs + tb * kTile), ks, RB),
                         sdesc_kmajor(smem_u32(Bsm), ks, RB), id, ks > 0);
        }
        mma_commit(&bar_cb);
    }
    ok = wait_all(&bar_cb, 0, ok);
    tc_fence_after();
    if (ok) {
        // warps of a lane quadrant take alternate 64-column pieces; the upper 64
        // rows of the half tiles are zero and not stored
        const int row = 32 * q4 + lane;
#pragma unroll
        for (int tb = 0; tb < NT; ++tb)
            for (int sb = hf; sb < 2 * (tb + 1); sb += 2) {
                if (sb == 2 * tb + 1 && q4 < 2) continue;
                float v[64];
                tmem_ld64(tmem_addr(tm, 32 * q4, 64 * tb * (tb + 1) + 64 * sb), v);
                const uint32_t base = smem_u32(cb_tile(tb, sb)) + (uint32_t)row * 128u;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8)
                    st_shared_v4(base + (uint32_t)((c8 ^ (row & 7)) << 4), pack_bf2(v[8 * c8], v[8 * c8 + 1]),
                                 pack_bf2(v[8 * c8 + 2], v[8 * c8 + 3]), pack_bf2(v[8 * c8 + 4], v[8 * c8 + 5]),
                                 pack_bf2(v[8 * c8 + 6], v[8 * c8 + 7]));
            }
    }
    // CB tiles visible, CB out of TMEM, B dead
    tc_fence_before();
    ok = __syncthreads_and(ok ? 1 : 0) != 0;
    tc_fence_after();
    if (!B_IN_CB && tid == 0 && ok) {
        issue_x(h_begin);
        issue_s(h_begin);
    }
    int x_issued = B_IN_CB || ok ? 1 : 0, x_landed = 0, s_issued = x_issued, s_landed = 0;
    derive(0);
    __syncthreads();
    uint4 xr[NT][4];  // this thread's D x slices of the head whose epilogue comes next
    float D_ep = 0.f;  // D of the head whose epilogue comes next
    float ep_ep[NT], ep_k[NT];  // exp(cumA_t) of this thread's epilogue rows: next epilogue's, this head's
#pragma unroll
    for (int tb = 0; tb < NT; ++tb) ep_ep[tb] = ep_k[tb] = 0.f;
    for (int k = 0; k <= nh && ok; ++k) {
        const int h = h_begin + k, cur = k % NSC;
        const float D_k = k < nh ? p.D[h] : 0.f;  // used one iteration later
        const float *f = fbuf + cur * FST;
        const float *cum = f, *dts = f + Q, *piv = f + POFF;
        const uint32_t *f2 = reinterpret_cast<const uint32_t *>(f);
        // ---- W_k into TMEM (packed bf16 pairs, lane = t).  Units (t-block tb,
        // 64-column group sb) of rows t = 128 tb + 32 q4 + lane: every thread gets
        // one per t-block, exactly one of its three on the diagonal 64-group.
        auto build = [&](int tb, int sb, uint32_t col) {
            const int t = tb * 128 + 32 * q4 + lane, tr = t >> 6, row = t - 128 * tb;
            uint32_t pk[32];
            if (sb > tr) {
#pragma unroll
                for (int j = 0; j < 32; ++j) pk[j] = 0u;
            } else {
                const uint32_t cbb = smem_u32(cb_tile(tb, sb));
                const bool diag = sb == tr;
                const int u = (t & 63) >> 4, t16 = t & ~15;
                const float ct = cum[t];
                // row factor: exp(cumA_t - pivot); on the diagonal group the pivot ends the
                // sub-blocks left of the row's own (none when u = 0: the table is all 0)
                const float er = diag ? (u > 0 ? __expf(ct - cum[t16 - 1]) : 0.f) : __expf(ct - piv[sb]);
                const uint32_t er2 = pack_bf2(er, er);
                const uint32_t *tab = diag ? f2 + TOFF + 128 * sb + 32 * u : f2 + GOFF + 32 * sb;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    const uint4 cv = ld_shared_v4(cbb + sw128_chunk(row, c8));
                    const uint4 gv = *reinterpret_cast<const uint4 *>(tab + 4 * c8);
                    pk[4 * c8] = bmul2(bmul2(cv.x, gv.x), er2);
                    pk[4 * c8 + 1] = bmul2(bmul2(cv.y, gv.y), er2);
                    pk[4 * c8 + 2] = bmul2(bmul2(cv.z, gv.z), er2);
                    pk[4 * c8 + 3] = bmul2(bmul2(cv.w, gv.w), er2);
                }
                if (diag) {  // the row's own 16-wide sub-block, 0 for s > t
                    const uint4 c0 = ld_shared_v4(cbb + sw128_chunk(row, 2 * u));
                    const uint4 c1 = ld_shared_v4(cbb + sw128_chunk(row, 2 * u + 1));
                    const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                    uint32_t own[8];
                    if (f[FLOFF + (t >> 4)] != 0.f) {  // factored through cumA[t16]
                        const float ro = __expf(ct - cum[t16]);
                        const uint32_t ro2 = pack_bf2(ro, ro);
                        const uint4 o0 = *reinterpret_cast<const uint4 *>(f2 + OOFF + (t16 >> 1));
                        const uint4 o1 = *reinterpret_cast<const uint4 *>(f2 + OOFF + (t16 >> 1) + 4);
                        const uint32_t ow[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
                        const int tt = t & 15;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const uint32_t m = (2 * j <= tt ? 0x0000FFFFu : 0u) | (2 * j + 1 <= tt ? 0xFFFF0000u : 0u);
                            own[j] = bmul2(bmul2(cw[j], ow[j]), ro2) & m;
                        }
                    } else {  // direct exponentials
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int s0 = t16 + 2 * j;
                            const float w0 = s0 <= t ? bf_lo(cw[j]) * __expf(ct - cum[s0]) * dts[s0] : 0.f;
                            const float w1 = s0 + 1 <= t ? bf_hi(cw[j]) * __expf(ct - cum[s0 + 1]) * dts[s0 + 1] : 0.f;
                            own[j] = pack_bf2(w0, w1);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) pk[j] = (j >> 3) == u ? own[j & 7] : pk[j];
                }
            }
            tmem_st32u(tmem_addr(tm, 32 * q4, col + 32 * sb), pk);
        };
        const int dq = q4 >> 1;  // the rows' 64-group inside their t-block
        if (k < nh) {
#pragma unroll
            for (int tb = 0; tb < NT; ++tb) ep_k[tb] = __expf(cum[tb * 128 + 32 * q4 + lane]);
            // t-block 0 into its spare buffer: the ORANGE MMAs of head k - 2 read it last
            build(0, hf == 0 ? dq : 1 - dq, W0COL + 64 * (k & 1));
        }
        if (k > 0) {
            // ORANGE MMAs of head k-1 done: W of t-block 1 and the x buffer are free
            ok = mbar_wait(&bar_o, (uint32_t)((k - 1) & 1)) && ok;
            if (k < nh) {
                if (tid == 0 && ok) issue_x(h);
                if (ok) x_issued = k + 1;
            }
            // BLUE MMAs done too: the accumulators are final, the s_in buffer is free
            ok = mbar_wait(&bar_b, (uint32_t)((k - 1) & 1)) && ok;
            tc_fence_after();
            // ---- epilogue of head k - 1: y rows of t-block 0 into the staging tile, of t-block 1
            // into the s_in buffer
            const float Dh = D_ep;
#pragma unroll
            for (int tb = 0; tb < NT; ++tb) {
                const int t = tb * 128 + 32 * q4 + lane;
                float o[32], bl[32];
                tmem_ld32(tmem_addr(tm, 32 * q4, OCOL + tb * 64 + hf * 32), o);
                tmem_ld32(tmem_addr(tm, 32 * q4, BCOL + tb * 64 + hf * 32), bl);
                const float e = ep_ep[tb];
                const bool valid = t < vrows;
                const uint32_t yb = smem_u32(tb == 0 ? Ys : Ss) - (uint32_t)(tb * kTile);  // row t of the tile
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    const uint4 u = xr[tb][c8];
                    const uint32_t xw[4] = {u.x, u.y, u.z, u.w};
                    uint32_t yw[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float y0 = o[8 * c8 + 2 * j] + e * bl[8 * c8 + 2 * j] + Dh * bf_lo(xw[j]);
                        const float y1 = o[8 * c8 + 2 * j + 1] + e * bl[8 * c8 + 2 * j + 1] + Dh * bf_hi(xw[j]);
                        yw[j] = valid ? pack_bf2(y0, y1) : 0u;
                    }
                    st_shared_v4(yb + sw128_chunk(t, 4 * hf + c8), yw[0], yw[1], yw[2], yw[3]);
                }
            }
            fence_async_smem();
            tc_fence_before();
            ok = __syncthreads_and(ok ? 1 : 0) != 0;
            tc_fence_after();
            if (tid == 0 && ok) {  // y of head k - 1 out (rows past the sequence end are clipped); s_in of head k in
                for (int j = 0; j < NT; ++j) tma_store_4d(&maps.y, j == 0 ? Ys : Ss, 0, h - 1, t0 + 128 * j, bi);
                bulk_commit();
                if (k < nh) {
                    bulk_wait_read_all();
                    issue_s(h);
                }
            }
            if (ok && k < nh) s_issued = k + 1;
            if (!ok) break;
        }
        if (k < nh) {
            // prefetch raw scalars of head k + 2, derive those of head k + 1 (raw visible
            // since the last barrier), after x of head k has been requested
            if (k + 2 < nh) {
                stash((k + 2) % NSC);
                if (k + 3 < nh) fetch(k + 3);
            }
            if (k + 1 < nh) derive((k + 1) % NSC);
        }
        if (NT == 2 && k < nh) {
            if (hf == 0) {
                build(1, 0, W1COL);
                build(1, 1, W1COL);
            } else {
                build(1, dq == 0 ? 3 : 2, W1COL);
                build(1, 2 + dq, W1COL);
            }
        }
        if (k == nh) break;
        D_ep = D_k;
#pragma unroll
        for (int tb = 0; tb < NT; ++tb) ep_ep[tb] = ep_k[tb];
        // ---- x_k landed: keep this thread's D x slices, zero padded rows
        ok = mbar_wait(&bar_x, (uint32_t)(k & 1)) && ok;
        if (ok) x_landed = k + 1;
        ok = mbar_wait(&bar_s, (uint32_t)(k & 1)) && ok;
        if (ok) s_landed = k + 1;
#pragma unroll
        for (int tb = 0; tb < NT; ++tb) {
            const int t = tb * 128 + 32 * q4 + lane;
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) xr[tb][c8] = ld_shared_v4(smem_u32(xs) + sw128_chunk(t, 4 * hf + c8));
        }
        if (vrows < Q) {
            __syncthreads();
            zero_rows_from(xs, Q, vrows);
            fence_async_smem();
        }
        // ---- one barrier: W_k stored, accumulators of k-1 read, x_k in place.  The
        // two issuing threads sit in warps 4 and 5, whose rows carry the fewest
        // W entries (two of their three units lie above the diagonal when q4 < 2).
        tc_fence_before();
        ok = __syncthreads_and(ok ? 1 : 0) != 0;
        tc_fence_after();
        if (tid == 128 && ok) {
            const uint32_t id = idesc_bf16(128, 64, false, true);
            if (NT == 2)
                for (int ks = 0; ks < 16; ++ks)
                    mma_bf16_tmem_a(tm + OCOL + 64, tm + W1COL + 8 * ks, sdesc_mnmajor(smem_u32(xs), ks, XB), id,
                                    ks > 0);
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16_tmem_a(tm + OCOL, tm + W0COL + 64 * (k & 1) + 8 * ks, sdesc_mnmajor(smem_u32(xs), ks, XB),
                                id, ks > 0);
            mma_commit(&bar_o);
        }
        if (tid == 160 && ok) {
            const uint32_t ib = idesc_bf16(128, 64, false, false);
            for (int tb = 0; tb < NT; ++tb)
                for (int ks = 0; ks < kN / 16; ++ks)
                    mma_bf16(tm + BCOL + tb * 64, sdesc_kmajor(smem_u32(Cs + tb * kTile), ks, RB),
                             sdesc_kmajor(smem_u32(Ss), ks, SB), ib, ks > 0);
            mma_commit(&bar_b);
        }
    }
    if (!ok && tid == 0) flag_timeout(p);
    // a load issued for a head that was never waited for has to land before exit
    if (x_issued > x_landed) mbar_wait(&bar_x, (uint32_t)((x_issued - 1) & 1));
    if (s_issued > s_landed) mbar_wait(&bar_s, (uint32_t)((s_issued - 1) & 1));
    if (tid == 0) bulk_wait_all();
    tc_sync();
    if (warp == 0) tmem_dealloc(tm, NCOL);
}

// ====================================================================== BLUE backward
// CTA per (b, chunk, group, head slice): 8 consumer warps and one producer
// warp; C stays resident, (dy, s_in) stream through a ring of NST stages.  Per head
//   d_ch[l, p]     = dy[l, p] exp(cumA_l)   (row l scaled in place by consumer thread l,
//                                            which keeps it in registers for the dot below)
//   d_s_in[r, p]   = sum_l C[l, r] d_ch[l, p]   (A = C MN-major, B = d_ch MN-major)
//   u[l, p]        = sum_r C[l, r] s_in[p, r]   (A = C K-major,  B = s_in K-major)
//   d_cumA_blue[l] = sum_p d_ch[l, p] u[l, p]
// into one of two TMEM buffers.  The producer issues the TMA refills and the
// MMAs: head k's once every consumer warp has scaled its rows and left the
// epilogue of head k - 2 (two mbarriers the warps arrive on), so no CTA-wide
// barrier sits in the loop and the MMAs of head k overlap the epilogue of k - 1.
template <int Q>
__global__ void __launch_bounds__(kThreadsWide + 32, 1) tc_bwd_blue_kernel(const Params p, const __grid_constant__ TcMaps maps) {
    constexpr int NT = Q / 128;
    constexpr uint32_t XB = Q * 128, RB = Q * 128, SB = 64 * 128;
    constexpr uint32_t STG = XB + 2 * SB;
    constexpr int NST = 3;
    constexpr uint32_t BUF = 256;  // TMEM columns per buffer: d_s_in 64 | u NT * 64
    constexpr int NCONS = kThreadsWide;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *Cs = sm, *stg = sm + 2 * RB;
    __shared__ uint64_t bar_res, bar_x[NST], bar_free[NST], bar_scaled[NST], bar_mma[2], bar_tfree[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_issued, s_landed, s_perr;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int idx = blockIdx.x;
    const int slice = idx % p.nslice_k3;
    idx /= p.nslice_k3;
    const int g = idx % p.G, c = (idx / p.G) % p.n, bi = idx / (p.G * p.n);
    const int t0 = c * Q;
    const int vrows = min(Q, valid_len_of(p, bi) - t0);
    const int per = (p.hpg + p.nslice_k3 - 1) / p.nslice_k3;
    const int h_begin = g * p.hpg + slice * per;
    const int nh = max(0, min(g * p.hpg + p.hpg, h_begin + per) - h_begin);
    if (nh == 0) return;
    if (vrows <= 0) {
        for (int k = 0; k < nh; ++k) {
            bf16 *dsin = p.dstates_bf + ix_state(p, bi, c, h_begin + k);
            for (int i = tid; i < kP * kN / 8; i += blockDim.x) reinterpret_cast<uint4 *>(dsin)[i] = make_uint4(0, 0, 0, 0);
            float *dcb = p.dcum_blue + ix_chunk(p, bi, h_begin + k, c) * Q;
            for (int i = tid; i < Q; i += blockDim.x) dcb[i] = 0.f;
        }
        return;
    }
    if (tid == 0) {
        mbar_init(&bar_res, 1);
        for (int i = 0; i < NST; ++i) {
            mbar_init(&bar_x[i], 1);
            mbar_init(&bar_free[i], 1);
            mbar_init(&bar_scaled[i], NCONS / 32);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_mma[i], 1);
            mbar_init(&bar_tfree[i], NCONS / 32);
        }
        mbar_fence_init();
        s_issued = 0;
        s_landed = 0;
        s_perr = 0;
    }
    if (warp == 0) tmem_alloc(&s_tmem, 512);
    tc_sync();
    const uint32_t tm = s_tmem;
    bool ok = true;
    if (warp == NCONS / 32) {
        // ---- producer: C once; (dy_k, s_in_k) into stage k % NST once head k - NST's
        // MMAs are done; head k's MMAs once it is scaled and TMEM buffer k & 1 is free
        if (lane == 0) {
            auto load = [&](int k) {
                const int st = k % NST, h = h_begin + k;
                uint8_t *dys = stg + st * STG, *sis = dys + XB;
                const int sidx = (bi * p.n + c) * p.H + h;
                mbar_arrive_expect_tx(&bar_x[st], STG);
                for (int j = 0; j < NT; ++j) tma_load_4d(dys + j * kTile, &maps.dy, &bar_x[st], 0, h, t0 + 128 * j, bi);
                for (int rb = 0; rb < 2; ++rb) tma_load_3d(sis + rb * SB, &maps.st, &bar_x[st], 64 * rb, 0, sidx);
                s_issued = k + 1;
            };
            mbar_arrive_expect_tx(&bar_res, 2 * RB);
            for (int rb = 0; rb < 2; ++rb)
                for (int j = 0; j < NT; ++j)
                    tma_load_4d(Cs + rb * RB + j * kTile, &maps.C, &bar_res, 64 * rb, g, t0 + 128 * j, bi);
            for (int k = 0; k < NST && k < nh; ++k) load(k);
            for (int k = 0; k < nh; ++k) {
                const int st = k % NST;
                if (!mbar_wait(&bar_scaled[st], (uint32_t)((k / NST) & 1)) || s_perr) {
                    s_perr = 1;
                    break;
                }
                s_landed = k + 1;
                // the stage of head k - 1 is free once its MMAs are done: head k - 1 + NST goes there
                if (k >= 1 && k - 1 + NST < nh) {
                    if (!mbar_wait(&bar_free[(k - 1) % NST], (uint32_t)(((k - 1) / NST) & 1))) {
                        s_perr = 1;
                        break;
                    }
                    load(k - 1 + NST);
                }
                if (k >= 2 && !mbar_wait(&bar_tfree[k & 1], (uint32_t)(((k - 2) >> 1) & 1))) {
                    s_perr = 1;
                    break;
                }
                tc_fence_after();
                uint8_t *dys = stg + st * STG, *sis = dys + XB;
                const uint32_t buf = BUF * (k & 1);
                const uint32_t i1 = idesc_bf16(128, 64, true, true);
                for (int ks = 0; ks < Q / 16; ++ks)
                    mma_bf16(tm + buf, sdesc_mnmajor(smem_u32(Cs), ks, RB), sdesc_mnmajor(smem_u32(dys), ks, XB), i1,
                             ks > 0);
                const uint32_t i2 = idesc_bf16(128, 64, false, false);
                for (int tb = 0; tb < NT; ++tb)
                    for (int ks = 0; ks < kN / 16; ++ks)
                        mma_bf16(tm + buf + 64 + tb * 64, sdesc_kmajor(smem_u32(Cs + tb * kTile), ks, RB),
                                 sdesc_kmajor(smem_u32(sis), ks, SB), i2, ks > 0);
                mma_commit(&bar_mma[k & 1]);
                mma_commit(&bar_free[st]);
            }
        }
    } else {
        // ---- consumers: thread t owns token row t; for the d_s_in epilogue,
        // TMEM lane r = 32 (warp % 4) + lane and headdim half warp / 4
        const int t = tid;
        const bool valid = t < vrows;
        const int q4 = warp & 3, hf = warp >> 2;
        const int r = 32 * q4 + lane;
        float c_cur = 0.f, c_nx = 0.f;
        auto fetch = [&](int k) { return t < Q ? p.cumA[ix_chunk(p, bi, h_begin + k, c) * Q + t] : 0.f; };
        c_cur = fetch(0);
        if (nh > 1) c_nx = fetch(1);
        ok = mbar_wait(&bar_res, 0);
        if (ok && vrows < Q) {
            zero_rows_from_n(Cs, Q, vrows, NCONS);
            zero_rows_from_n(Cs + RB, Q, vrows, NCONS);
        }
        uint4 dch[8], dch_prev[8];  // scaled dy row t of the current / previous head
#pragma unroll
        for (int i = 0; i < 8; ++i) dch_prev[i] = dch[i] = make_uint4(0, 0, 0, 0);
        for (int k = 0; k <= nh && ok; ++k) {
            if (k < nh) {
                const int st = k % NST;
                uint8_t *dys = stg + st * STG;
                const float e_row = __expf(c_cur);
                c_cur = c_nx;
                if (k + 2 < nh) c_nx = fetch(k + 2);
                ok = __all_sync(0xffffffffu, mbar_wait(&bar_x[st], (uint32_t)((k / NST) & 1)) && ok);  // warp-uniform
                if (ok && t < Q) {
                    const uint32_t base = smem_u32(dys);
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        const uint32_t a = base + sw128_chunk(t, c8);
                        uint4 v = make_uint4(0, 0, 0, 0);
                        if (valid) {
                            v = ld_shared_v4(a);
                            v.x = pack_bf2(bf_lo(v.x) * e_row, bf_hi(v.x) * e_row);
                            v.y = pack_bf2(bf_lo(v.y) * e_row, bf_hi(v.y) * e_row);
                            v.z = pack_bf2(bf_lo(v.z) * e_row, bf_hi(v.z) * e_row);
                            v.w = pack_bf2(bf_lo(v.w) * e_row, bf_hi(v.w) * e_row);
                        }
                        st_shared_v4(a, v.x, v.y, v.z, v.w);
                        dch[c8] = v;
                    }
                }
                if (!ok) s_perr = 1;
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_scaled[st]);  // the producer issues head k's MMAs
            }
            if (k > 0) {
                // ---- epilogue of head k - 1
                const int kk = k - 1, h = h_begin + kk;
                const uint32_t buf = BUF * (kk & 1);
                ok = __all_sync(0xffffffffu, mbar_wait(&bar_mma[kk & 1], (uint32_t)((kk >> 1) & 1)) && ok);
                if (!ok) {
                    s_perr = 1;
                    break;
                }
                tc_fence_after();
                float v[32];
                tmem_ld32(tmem_addr(tm, 32 * q4, buf + 32 * hf), v);
                float u[64];
                if (t < Q) {  // warp w holds rows 128 (w / 4) + 32 (w % 4) + lane of u: its own t
                    tmem_ld32(tmem_addr(tm, 32 * q4, buf + 64 + 64 * hf), u);
                    tmem_ld32(tmem_addr(tm, 32 * q4, buf + 64 + 64 * hf + 32), u + 32);
                }
                // TMEM buffer kk & 1 read: the MMAs of head k + 1 may overwrite it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_tfree[kk & 1]);
                bf16 *dsin = p.dstates_bf + ix_state(p, bi, c, h);
#pragma unroll
                for (int j = 0; j < 32; ++j) dsin[(size_t)(32 * hf + j) * kN + r] = __float2bfloat16_rn(v[j]);
                if (t < Q) {
                    float acc = 0.f;
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        const uint4 d = dch_prev[c8];
                        const float *uu = u + 8 * c8;
                        acc += bf_lo(d.x) * uu[0] + bf_hi(d.x) * uu[1] + bf_lo(d.y) * uu[2] + bf_hi(d.y) * uu[3] +
                               bf_lo(d.z) * uu[4] + bf_hi(d.z) * uu[5] + bf_lo(d.w) * uu[6] + bf_hi(d.w) * uu[7];
                    }
                    p.dcum_blue[ix_chunk(p, bi, h, c) * Q + t] = valid ? acc : 0.f;
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) dch_prev[i] = dch[i];
        }
    }
    tc_fence_before();
    ok = __syncthreads_and(ok && s_perr == 0 ? 1 : 0) != 0;
    tc_fence_after();
    if (!ok && tid == 0) flag_timeout(p);
    if (tid == 0)
        for (int k = s_landed; k < s_issued; ++k) mbar_wait(&bar_x[k % NST], (uint32_t)((k / NST) & 1));
    // the last heads' MMAs (each commit covers the producer's earlier ones)
    if (tid == 0 && s_landed > 0) mbar_wait(&bar_free[(s_landed - 1) % NST], (uint32_t)(((s_landed - 1) / NST) & 1));
    tc_sync();
    if (warp == 0) tmem_dealloc(tm, 512);
}

// ====================================================================== K3 backward
// CTA per (b, chunk, group, head slice), 256 threads, looping over the slice's
// heads with a two-stage TMA ring (x, d_intra); B stays resident.  Per head
// (the K3 BACKWARD block, with the per-head d_b_scaled folded away):
//   U[s, p]   = sum_r B[s, r] d_intra[p, r]           (TMEM, A = B K-major, B = d_intra K-major)
//   d_bbs[s]  = sum_p x[s, p] U[s, p]
//   dx       += bbs[s] U[s, p]                        (dx holds the ORANGE and skip terms)
//   ddt_main += d_bbs exp(cumA_last - cumA)           (the K3 part of ddt)
//   d_delta   = d_bbs dt exp(cumA_last - cumA),  dcum_main -= d_delta   (the K3 part of d cumA)
// Runs after the ORANGE kernel.  The dx tile of a head (which holds the ORANGE
// and skip terms) comes in by TMA, is updated in place in shared memory and
// goes back out by a TMA tile store; the next head's tile is fetched once that
// store has read the buffer.  The per-token sums are read-modify-written
// directly (coalesced), prefetched at the top of each head.
template <int Q>
__global__ void __launch_bounds__(kThreadsWide, 1) tc_bwd_k3_kernel(const Params p, const __grid_constant__ TcMaps maps) {
    constexpr int NT = Q / 128;
    constexpr uint32_t XB = Q * 128, RB = Q * 128, SB = 64 * 128;
    constexpr uint32_t STG = XB + 2 * SB;
    constexpr uint32_t NCOL = NT == 2 ? 256 : 128;  // U, two buffers of NT * 64 columns
    constexpr int NSC = 3;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *Bs = sm, *stg = Bs + 2 * RB, *dxs = stg + 2 * STG;
    float *fbuf = reinterpret_cast<float *>(dxs + XB);  // [NSC][3Q]: dts, dec_end, (spare)
    float *dbbp = fbuf + NSC * 3 * Q;                        // [2][Q]
    __shared__ uint64_t bar_res, bar_x[2], bar_mma[2], bar_dx;
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, hf = warp >> 2;
    int idx = blockIdx.x;
    const int slice = idx % p.nslice_k5;
    idx /= p.nslice_k5;
    const int g = idx % p.G, c = (idx / p.G) % p.n, bi = idx / (p.G * p.n);
    const int t0 = c * Q;
    const int vrows = min(Q, valid_len_of(p, bi) - t0);
    const int per = (p.hpg + p.nslice_k5 - 1) / p.nslice_k5;
    const int h_begin = g * p.hpg + slice * per;
    const int h_end = min(g * p.hpg + p.hpg, h_begin + per);
    const int nh = h_end - h_begin;
    bf16 *DX = (bf16 *)p.dx;
    if (nh <= 0) return;
    if (vrows <= 0) {  // dx, ddt_main, dcum_main already zero (ORANGE kernel)
        for (int hh = h_begin; hh < h_end; ++hh) {
            const size_t cb = ix_chunk(p, bi, hh, c) * Q;
            for (int i = tid; i < Q; i += kThreadsWide) p.d_delta[cb + i] = 0.f;
        }
        return;
    }
    // per-head scalars fetched into registers (thread l holds token l) a head
    // before they are staged: dt, and the decay to the chunk end
    float r_dt = 0.f, r_cum = 0.f, r_end = 0.f;
    auto fetch = [&](int k) {
        const int h = h_begin + k;
        if (tid < Q) {
            r_cum = p.cumA[ix_chunk(p, bi, h, c) * Q + tid];
            r_end = p.endA[ix_chunk(p, bi, h, c)];
            r_dt = tid < vrows ? p.dt[ix_dt(p, bi, h, t0 + tid)] : 0.f;
        }
    };
    auto stash = [&](int b) {
        float *f = fbuf + b * 3 * Q;
        if (tid < Q) {
            f[tid] = r_dt;
            f[Q + tid] = __expf(r_end - r_cum);
        }
    };
    auto issue_dx = [&](int k) {  // thread 0: the dx tile of head k
        mbar_arrive_expect_tx(&bar_dx, XB);
        for (int j = 0; j < NT; ++j) tma_load_4d(dxs + j * kTile, &maps.dx, &bar_dx, 0, h_begin + k, t0 + 128 * j, bi);
    };
    auto issue = [&](int k) {
        const int h = h_begin + k, st = k & 1;
        uint8_t *xs = stg + st * STG, *dis = xs + XB;
        const int sidx = (bi * p.n + c) * p.H + h;
        mbar_arrive_expect_tx(&bar_x[st], STG);
        for (int j = 0; j < NT; ++j) tma_load_4d(xs + j * kTile, &maps.x, &bar_x[st], 0, h, t0 + 128 * j, bi);
        for (int rb = 0; rb < 2; ++rb) tma_load_3d(dis + rb * SB, &maps.dst, &bar_x[st], 64 * rb, 0, sidx);
    };
    if (tid == 0) {
        mbar_init(&bar_res, 1);
        mbar_init(&bar_x[0], 1);
        mbar_init(&bar_x[1], 1);
        mbar_init(&bar_mma[0], 1);
        mbar_init(&bar_mma[1], 1);
        mbar_init(&bar_dx, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&s_tmem, NCOL);
    tc_sync();
    const uint32_t tm = s_tmem;
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar_res, 2 * RB);
        for (int j = 0; j < NT; ++j)
            for (int rb = 0; rb < 2; ++rb)
                tma_load_4d(Bs + rb * RB + j * kTile, &maps.B, &bar_res, 64 * rb, g, t0 + 128 * j, bi);
        issue(0);
        if (nh > 1) issue(1);
        issue_dx(0);
    }
    fetch(0);
    stash(0);
    if (nh > 1) {
        fetch(1);
        stash(1);
    }
    if (nh > 2) fetch(2);
    int issued = nh > 1 ? 2 : 1, landed = 0, dx_issued = 1, dx_landed = 0;
    bool ok = wait_all(&bar_res, 0, true);
    if (ok && vrows < Q) {
        zero_rows_from(Bs, Q, vrows);
        zero_rows_from(Bs + RB, Q, vrows);
        fence_async_smem();
    }
    for (int k = 0; k < nh && ok; ++k) {
        const int h = h_begin + k, st = k & 1;
        uint8_t *xs = stg + st * STG, *dis = xs + XB;
        const float *f = fbuf + (k % NSC) * 3 * Q;
        const float *dts = f, *dec = f + Q;
        const size_t cbase = ix_chunk(p, bi, h, c) * Q;
        if (tid == 0 && k > 0) {  // the store of head k - 1's tile has read the buffer: fetch head k's
            bulk_wait_read_all();
            issue_dx(k);
        }
        if (k > 0) dx_issued = k + 1;
        // prefetch this head's per-token sums
        float ddt_pre[(Q + kThreadsWide - 1) / kThreadsWide], dcum_pre[(Q + kThreadsWide - 1) / kThreadsWide];
#pragma unroll
        for (int i = 0; i < (Q + kThreadsWide - 1) / kThreadsWide; ++i) {
            const int s = tid + i * kThreadsWide;
            if (s < Q) {
                ddt_pre[i] = p.ddt_main[cbase + s];
                dcum_pre[i] = p.dcum_main[cbase + s];
            }
        }
        ok = mbar_wait(&bar_x[st], (uint32_t)((k >> 1) & 1)) && ok;
        if (ok) landed = k + 1;
        if (vrows < Q) {
            __syncthreads();
            zero_rows_from(xs, Q, vrows);
        }
        fence_async_smem();
        tc_fence_before();
        ok = __syncthreads_and(ok ? 1 : 0) != 0;
        tc_fence_after();
        if (!ok) break;
        const uint32_t ucol = (uint32_t)(st * NT * 64);
        if (tid == 0) {
            const uint32_t iu = idesc_bf16(128, 64, false, false);
            for (int mb = 0; mb < NT; ++mb)
                for (int ks = 0; ks < kN / 16; ++ks)
                    mma_bf16(tm + ucol + mb * 64, sdesc_kmajor(smem_u32(Bs + mb * kTile), ks, RB),
                             sdesc_kmajor(smem_u32(dis), ks, SB), iu, ks > 0);
            mma_commit(&bar_mma[st]);
        }
        if (k + 2 < nh) {  // buffer (k + 2) % NSC was last read by head k - 1
            stash((k + 2) % NSC);
            if (k + 3 < nh) fetch(k + 3);
        }
        ok = mbar_wait(&bar_mma[st], (uint32_t)((k >> 1) & 1)) && ok;
        tc_fence_after();
        ok = mbar_wait(&bar_dx, (uint32_t)(k & 1)) && ok;
        if (ok) dx_landed = k + 1;
        for (int mb = 0; mb < NT; ++mb) {
            const int s = mb * 128 + 32 * q4 + lane;
            float u[32];
            tmem_ld32(tmem_addr(tm, 32 * q4, ucol + mb * 64 + 32 * hf), u);
            float part = 0.f;
            const uint32_t xb = smem_u32(xs);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                const uint4 xv = ld_shared_v4(xb + sw128_chunk(s, 4 * hf + c8));
                const float *uu = u + 8 * c8;
                part += bf_lo(xv.x) * uu[0] + bf_hi(xv.x) * uu[1] + bf_lo(xv.y) * uu[2] + bf_hi(xv.y) * uu[3] +
                        bf_lo(xv.z) * uu[4] + bf_hi(xv.z) * uu[5] + bf_lo(xv.w) * uu[6] + bf_hi(xv.w) * uu[7];
            }
            dbbp[hf * Q + s] = part;
            if (s < vrows) {  // rows past valid_len keep the ORANGE kernel's zeros
                const float bbs = dts[s] * dec[s];
                const uint32_t db = smem_u32(dxs + mb * kTile);
                const int row = s & 127;
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    const uint32_t ad = db + sw128_chunk(row, 4 * hf + c8);
                    const uint4 pv = ld_shared_v4(ad);
                    const float *a = u + 8 * c8;
                    st_shared_v4(ad, pack_bf2(a[0] * bbs + bf_lo(pv.x), a[1] * bbs + bf_hi(pv.x)),
                                 pack_bf2(a[2] * bbs + bf_lo(pv.y), a[3] * bbs + bf_hi(pv.y)),
                                 pack_bf2(a[4] * bbs + bf_lo(pv.z), a[5] * bbs + bf_hi(pv.z)),
                                 pack_bf2(a[6] * bbs + bf_lo(pv.w), a[7] * bbs + bf_hi(pv.w)));
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        ok = __syncthreads_and(ok ? 1 : 0) != 0;  // d_bbs halves complete; stage st no longer read
        tc_fence_after();
        if (tid == 0 && ok) {  // the updated dx tile goes out (rows past the sequence end are clipped)
            for (int j = 0; j < NT; ++j) tma_store_4d(&maps.dx, dxs + j * kTile, 0, h, t0 + 128 * j, bi);
            bulk_commit();
        }
        if (tid == 0 && k + 2 < nh) issue(k + 2);
        if (k + 2 < nh) issued = k + 3;
#pragma unroll
        for (int i = 0; i < (Q + kThreadsWide - 1) / kThreadsWide; ++i) {
            const int s = tid + i * kThreadsWide;
            if (s < Q) {
                const float dbb = s < vrows ? dbbp[s] + dbbp[Q + s] : 0.f;
                const float ddelta = dbb * dts[s] * dec[s];
                p.ddt_main[cbase + s] = ddt_pre[i] + dbb * dec[s];
                p.d_delta[cbase + s] = ddelta;
                p.dcum_main[cbase + s] = dcum_pre[i] - ddelta;
            }
        }
    }
    if (!ok && tid == 0) flag_timeout(p);
    // loads issued for heads that were never waited for have to land before exit
    for (int k = landed; k < issued; ++k) mbar_wait(&bar_x[k & 1], (uint32_t)((k >> 1) & 1));
    if (dx_issued > dx_landed) mbar_wait(&bar_dx, (uint32_t)((dx_issued - 1) & 1));
    if (tid == 0) bulk_wait_all();
    tc_sync();
    if (warp == 0) tmem_dealloc(tm, NCOL);
}

// ====================================================================== ORANGE backward
// CTA per (b, chunk, group, head slice), 256 threads, looping over the slice's
// heads.  x arrives in two 128-row halves: the lower half (read by the last
// MMAs of a head) has two buffers and is fetched a head ahead; the upper half
// (read only by the first MMAs) has one, refilled as soon as those complete.
// dy has two buffers and is fetched a head ahead.  A head's dx rows are
// staged in its dy buffer once the epilogue has read dy, and leave by TMA tile
// stores at the next head's first barrier.  The ORANGE block of the backward is
// restated so that every reduction becomes a per-row dot product of two MMA
// outputs (thread = row of the chunk):
//   W^T[s, t]   = dt_s CB^T[s, t] exp(cumA_t - cumA_s)   (t >= s, 0 above): built
//                 per head in shared memory from a copy of CB^T kept in TMEM
//   z[s, p]     = sum_t W^T[s, t] dy[t, p]          (A = W^T K-major,  B = dy MN-major)
//   yo[t, p]    = sum_s W^T[s, t] x[s, p]           (A = W^T MN-major, B = x MN-major)
//   dx[s, p]    = z[s, p] + D dy[s, p]              (= sum_t W[t, s] dy[t, p] + D dy[s, p])
//   src[s]      = sum_p x[s, p] z[s, p]             (= sum_t dW[t, s] W[t, s])
//   tgt[t]      = sum_p dy[t, p] yo[t, p]           (= sum_s dW[t, s] W[t, s])
//   ddt_orange[s] = src[s] / dt_s                   (= sum_t dW[t, s] CB[t, s] decay[t, s])
// with dW = dy x^T; the page's column sums over targets and the row sums over
// sources reduce to these because dW is a product.  tgt and src are sums of the
// same bf16 products (W^T, x and dy as the MMAs saw them), so their sums over
// the chunk cancel to fp32 rounding as the page's do.  A valid token whose
// |dt| is below 2^-30 (an exact 0 included) scales its row by 2^-30 instead,
// and ddt_orange divides by the same: the row factors of the factored decay
// reach e^-64, and with the scale e^-64 * 2^-30 is still a normal bf16, where
// a smaller scale would flush the row's near-diagonal entries to zero; the
// row's entries stay 1e-6 below those of an ordinary dt, far under bf16
// rounding of the others.  Rows past valid_len are zero.  W^T is
// built in two halves (s-block 1, then s-block 0) so the first half's MMAs run
// while the second half is built.  The decay is factored through 64-group
// pivots off the diagonal groups and 16-wide sub-block pivots inside them (all
// factors <= 1).  The row's own 16-wide sub-block is factored through its last
// position (a row factor <= 1, a column factor <= e^64) when its decay span is
// below e^64, one exponential per element otherwise.  This kernel writes dx, ddt_main, dcum_main and the dD
// partials first; the K3 backward kernel runs after it and adds its terms.
template <int Q>
__global__ void __launch_bounds__(kThreadsWide, 1) tc_bwd_orange_kernel(const Params p, const __grid_constant__ TcMaps maps) {
    constexpr int NT = Q / 128;
    constexpr uint32_t XB = Q * 128;
    constexpr int NCBT = NT == 2 ? 6 : 2;  // W^T tiles: s-block 0 Q/64, s-block 1 Q/64 - 2
    constexpr int NCONS = kThreadsWide;
    constexpr int NSC = 3;                 // scalar buffers: staged two heads ahead
    // per-head tables (32-bit words): cum Q | dt Q | E pairs 192 | E16 pairs 16 x 32 | piv 8 | piv16 16 | D 4 |
    // own-sub-block column pairs Q/2 | own-sub-block fast flags Q/16
    constexpr int E2OFF = 2 * Q, E16OFF = E2OFF + 192, POFF = E16OFF + 512, P16OFF = POFF + 8;
    constexpr int DOFF = P16OFF + 16;
    constexpr int OOFF = DOFF + 4, FLOFF = OOFF + Q / 2;
    constexpr int FST = FLOFF + Q / 16;
    constexpr uint32_t CBCOL0 = 256, CBCOL1 = 384;  // CB^T resident in TMEM (packed bf16 pairs)
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    constexpr int XSL = NT == 2 ? 3 : 2;  // x half tiles: lower half x 2, upper half
    uint8_t *Mt = sm, *xs = Mt + NCBT * kTile, *dys = xs + XSL * kTile;  // dys: 2 buffers
    uint8_t *xhi = xs + 2 * kTile;                                        // upper half of x (Q = 256)
    float *fbuf = reinterpret_cast<float *>(dys + 2 * XB);       // [NSC][FST]
    __shared__ uint64_t bar_cb, bar_xlo[2], bar_xhi, bar_a, bar_dy[2], bar_mma;
    __shared__ uint32_t s_tmem;
    __shared__ int s_lo_issued, s_hi_issued, s_dy_issued, s_landed;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int idx = blockIdx.x;
    const int slice = idx % p.nslice_k5;
    idx /= p.nslice_k5;
    const int g = idx % p.G, c = (idx / p.G) % p.n, bi = idx / (p.G * p.n);
    const int t0 = c * Q;
    const int vrows = min(Q, valid_len_of(p, bi) - t0);
    const int per = (p.hpg + p.nslice_k5 - 1) / p.nslice_k5;
    const int h_begin = g * p.hpg + slice * per;
    const int nh = max(0, min(g * p.hpg + p.hpg, h_begin + per) - h_begin);
    bf16 *DX = (bf16 *)p.dx;
    if (nh == 0) return;
    if (vrows <= 0) {  // a chunk wholly past valid_len contributes nothing
        const int rows = min(Q, p.L - t0);
        for (int hh = h_begin; hh < h_begin + nh; ++hh) {
            for (int i = tid; i < rows * (kP / 8); i += blockDim.x)
                reinterpret_cast<uint4 *>(DX + ix_x(p, bi, t0 + i / 8, hh, 0))[i % 8] = make_uint4(0, 0, 0, 0);
            const size_t cb = ix_chunk(p, bi, hh, c) * Q;
            for (int i = tid; i < Q; i += blockDim.x) {
                p.dcum_main[cb + i] = 0.f;
                p.ddt_main[cb + i] = 0.f;
            }
            for (int i = tid; i < p.dD_per; i += blockDim.x)
                p.dD_part[(((size_t)bi * p.n + c) * p.H + hh) * p.dD_per + i] = 0.f;
        }
        return;
    }
    auto tile_of = [&](int mb, int tj) -> uint8_t * {  // W^T tile of s-block mb, t-tile tj (tj >= 2 mb)
        return Mt + (mb == 0 ? tj : (Q / 64) + tj - 2) * kTile;
    };
    if (tid == 0) {
        mbar_init(&bar_cb, 1);
        mbar_init(&bar_xlo[0], 1);
        mbar_init(&bar_xlo[1], 1);
        mbar_init(&bar_xhi, 1);
        mbar_init(&bar_a, 1);
        mbar_init(&bar_dy[0], 1);
        mbar_init(&bar_dy[1], 1);
        mbar_init(&bar_mma, 2);
        mbar_fence_init();
        s_lo_issued = 0;
        s_hi_issued = 0;
        s_dy_issued = 0;
        s_landed = 0;
    }
    if (warp == 0) tmem_alloc(&s_tmem, 512);
    tc_sync();
    const uint32_t tm = s_tmem;  // z[mb] at 64 mb, yo[tb] at 128 + 64 tb, CB^T at 256
    bool ok = true;
    const int cbrow = ((bi * p.n + c) * p.G + g) * Q;
    auto issue_xlo = [&](int k) {  // rows 0..127 of x of head k into buffer k & 1
        mbar_arrive_expect_tx(&bar_xlo[k & 1], kTile);
        tma_load_4d(xs + (k & 1) * kTile, &maps.x, &bar_xlo[k & 1], 0, h_begin + k, t0, bi);
        s_lo_issued = k + 1;
    };
    auto issue_xhi = [&](int k) {  // rows 128..255 of x of head k
        mbar_arrive_expect_tx(&bar_xhi, kTile);
        tma_load_4d(xhi, &maps.x, &bar_xhi, 0, h_begin + k, t0 + 128, bi);
        s_hi_issued = k + 1;
    };
    auto issue_dy = [&](int k) {  // thread 0: dy of head k into buffer k & 1
        const int b = k & 1;
        mbar_arrive_expect_tx(&bar_dy[b], XB);
        for (int j = 0; j < NT; ++j)
            tma_load_4d(dys + b * XB + j * kTile, &maps.dy, &bar_dy[b], 0, h_begin + k, t0 + 128 * j, bi);
        s_dy_issued = k + 1;
    };
    if (tid == 0) {  // CB^T once (staged through the W^T buffer into TMEM), then the head ring
        mbar_arrive_expect_tx(&bar_cb, NCBT * kTile);
        for (int mb = 0; mb < NT; ++mb)
            for (int tj = 2 * mb; tj < Q / 64; ++tj)
                tma_load_2d(tile_of(mb, tj), &maps.cbt, &bar_cb, 64 * tj, cbrow + 128 * mb);
        issue_xlo(0);
        if (NT == 2) issue_xhi(0);
        if (nh > 1) issue_xlo(1);
        issue_dy(0);
    }
    {
        const int i = tid;  // chunk row of this thread (token for the row outputs)
        const bool valid = i < vrows;
        float r_cum = 0.f, r_dt = 0.f, r_D = 0.f;
        auto fetch = [&](int k) {
            const int h = h_begin + k;
            if (i < Q) {
                r_cum = p.cumA[ix_chunk(p, bi, h, c) * Q + i];
                r_dt = valid ? p.dt[ix_dt(p, bi, h, t0 + i)] : 0.f;
            }
            if (i == 0) r_D = p.D[h];
        };
        auto stash = [&](int k) {
            float *f = fbuf + (k % NSC) * FST;
            if (i < Q) {
                f[i] = r_cum;
                f[Q + i] = r_dt;
            }
            if (i == 0) f[DOFF] = r_D;
        };
        // pivot tables from the raw cumA (visible after a barrier), as bf16 pairs
        auto derive = [&](int k) {
            float *f = fbuf + (k % NSC) * FST;
            uint32_t *f2 = reinterpret_cast<uint32_t *>(f);
            // E[sg][t] = exp(cumA_t - cumA[64 sg + 63]) for t >= 64 (sg + 1); pair rows at 0, 96, 160
            for (int e = i; e < 192; e += NCONS) {
                const int sg = e < 96 ? 0 : (e < 160 ? 1 : 2);
                const int t = 64 * (sg + 1) + 2 * (e - (sg == 0 ? 0 : (sg == 1 ? 96 : 160)));
                const float pv = f[64 * sg + 63];
                f2[E2OFF + e] = (sg < Q / 64 - 1 && t < Q) ? pack_bf2(__expf(f[t] - pv), __expf(f[t + 1] - pv)) : 0u;
            }
            // E16[v][tt] = exp(cumA_t - cumA[16 v + 15]) for t = 64 (v / 4) + tt past v's sub-block
            for (int e = i; e < 512; e += NCONS) {
                const int v = e >> 5, t = 64 * (v >> 2) + 2 * (e & 31);
                float lo = 0.f, hi = 0.f;
                if (16 * v < Q && t < Q) {
                    const float pv = f[16 * v + 15];
                    if (t > 16 * v + 15) lo = __expf(f[t] - pv);
                    if (t + 1 > 16 * v + 15) hi = __expf(f[t + 1] - pv);
                }
                f2[E16OFF + e] = pack_bf2(lo, hi);
            }
            if (i < Q / 64) f[POFF + i] = f[64 * i + 63];
            if (i < Q / 16) f[P16OFF + i] = f[16 * i + 15];
            // own sub-block: O[t] = exp(cumA_t - cumA[t | 15]) (>= 1, <= e^64 where used)
            for (int e = i; e < Q / 2; e += NCONS) {
                const int t = 2 * e;
                const float pv = f[t | 15];
                f2[OOFF + e] = pack_bf2(__expf(f[t] - pv), __expf(f[t + 1] - pv));
            }
            if (i < Q / 16) f[FLOFF + i] = f[16 * i] - f[16 * i + 15] < 64.f ? 1.f : 0.f;
        };
        // W^T[s, t] for row s of t-tile tj: CB^T from TMEM, scaled as packed bf16 pairs
        // (off the row's own 16-wide sub-block), written to the shared-memory tile
        const int q4 = warp & 3;  // this warp's TMEM lane quarter (= row s % 128 / 32)
        auto cb_col = [&](int mb, int tj) -> uint32_t { return (mb == 0 ? CBCOL0 : CBCOL1) + 32 * (tj - 2 * mb); };
        // Each thread owns exactly one row-tile on the diagonal 64-group (see the unit
        // mapping below); the CB^T values of that row's own 16-wide sub-block are kept
        // in registers, so the sub-block's direct exponentials need no lane-dependent
        // TMEM column.
        uint32_t cbown[8];
        // the scale of row s of W^T: dt_s on valid tokens (+-2^-30 where |dt_s| < 2^-30), 0 past valid_len
        auto row_dt = [&](const float *f, int s) -> float {
            const float d = f[Q + s];
            return s < vrows ? (fabsf(d) >= 0x1p-30f ? d : (d < 0.f ? -0x1p-30f : 0x1p-30f)) : 0.f;
        };
        auto transform = [&](const float *f, int s, int tj) {
            const int sg = s >> 6, row = s & 127, mb = s >> 7;
            const uint32_t base = smem_u32(tile_of(mb, tj));
            uint32_t cb[32];
            tmem_ld32u(tmem_addr(tm, 32 * q4, cb_col(mb, tj)), cb);
            if (tj < sg) {  // wholly above the diagonal (never read by an MMA; kept finite)
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) st_shared_v4(base + sw128_chunk(row, c8), 0u, 0u, 0u, 0u);
                return;
            }
            const uint32_t *f2 = reinterpret_cast<const uint32_t *>(f);
            const float cs = f[s];
            // off the diagonal group: column table of the 64-group pivot; on it: column table
            // of the row's 16-wide sub-block pivot (0 up to and including that sub-block)
            const bool diag = tj == sg;
            const float dsc = row_dt(f, s);
            const float fr = __expf((diag ? f[P16OFF + (s >> 4)] : f[POFF + sg]) - cs) * dsc;
            const uint32_t fr2 = pack_bf2(fr, fr);
            const uint32_t *Erow = diag ? f2 + E16OFF + 32 * (s >> 4) - 32 * sg
                                        : f2 + E2OFF + (sg == 0 ? 0 : (sg == 1 ? 96 : 160)) - 32 * (sg + 1);
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                const uint4 e = *reinterpret_cast<const uint4 *>(Erow + 32 * tj + 4 * c8);
                st_shared_v4(base + sw128_chunk(row, c8), bmul2(bmul2(cb[4 * c8], e.x), fr2),
                             bmul2(bmul2(cb[4 * c8 + 1], e.y), fr2), bmul2(bmul2(cb[4 * c8 + 2], e.z), fr2),
                             bmul2(bmul2(cb[4 * c8 + 3], e.w), fr2));
            }
            if (diag) {  // the row's own 16-wide sub-block, 0 for t < s
                const int t16 = s & ~15, us = (s & 63) >> 4;
                uint32_t w2[8];
                if (f[FLOFF + (s >> 4)] != 0.f) {
                    // span below e^64: factored through cumA[t16 + 15], row factor (<= 1) x column table
                    const float ro = __expf(f[t16 + 15] - cs) * dsc;
                    const uint32_t ro2 = pack_bf2(ro, ro);
                    const uint4 o0 = *reinterpret_cast<const uint4 *>(f2 + OOFF + (t16 >> 1));
                    const uint4 o1 = *reinterpret_cast<const uint4 *>(f2 + OOFF + (t16 >> 1) + 4);
                    const uint32_t ow[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
                    const int ss = s & 15;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t m = (2 * j >= ss ? 0x0000FFFFu : 0u) | (2 * j + 1 >= ss ? 0xFFFF0000u : 0u);
                        w2[j] = bmul2(bmul2(cbown[j], ow[j]), ro2) & m;
                    }
                } else {  // direct exponentials
                    float w[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const uint32_t pr = cbown[j >> 1];
                        const float cv = (j & 1) ? bf_hi(pr) : bf_lo(pr);
                        w[j] = t16 + j >= s ? cv * __expf(f[t16 + j] - cs) * dsc : 0.f;
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) w2[j] = pack_bf2(w[2 * j], w[2 * j + 1]);
                }
                st_shared_v4(base + sw128_chunk(row, 2 * us), w2[0], w2[1], w2[2], w2[3]);
                st_shared_v4(base + sw128_chunk(row, 2 * us + 1), w2[4], w2[5], w2[6], w2[7]);
            }
        };
        // CB^T: shared-memory tiles (TMA) -> TMEM, by the threads that later transform each row
        auto cb_to_tmem = [&](int s, int tj) {
            const int row = s & 127, mb = s >> 7;
            const uint32_t base = smem_u32(tile_of(mb, tj));
            uint32_t v[32];
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                const uint4 u = ld_shared_v4(base + sw128_chunk(row, c8));
                v[4 * c8] = u.x;
                v[4 * c8 + 1] = u.y;
                v[4 * c8 + 2] = u.z;
                v[4 * c8 + 3] = u.w;
            }
            tmem_st32u(tmem_addr(tm, 32 * q4, cb_col(mb, tj)), v);
            if (tj == (s >> 6)) {  // this thread's diagonal row-tile: keep its own sub-block
                const int us = (s & 63) >> 4;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    cbown[j] = us == 0 ? v[j] : (us == 1 ? v[8 + j] : (us == 2 ? v[16 + j] : v[24 + j]));
            }
        };
        // row-tile units: s-block 1 (phase A) row 128 + r, t-tile 2 + (i / 128); s-block 0
        // (phase B) row r, t-tiles 1 - (i / 128) and 3 - (i / 128).  Every thread gets
        // exactly one unit on the diagonal 64-group and TMEM lane quarter r / 32.
        const int r = i & 127, hi = i >> 7;
        ok = mbar_wait(&bar_cb, 0);
        if (NT == 2) cb_to_tmem(128 + r, 2 + hi);
        cb_to_tmem(r, 1 - hi);
        if (NT == 2) cb_to_tmem(r, 3 - hi);
        tc_fence_before();
        ok = bar_and(1, NCONS, ok);
        tc_fence_after();
        fetch(0);
        stash(0);
        if (nh > 1) {
            fetch(1);
            stash(1);
        }
        if (nh > 2) fetch(2);
        bar_sync_n(1, NCONS);
        derive(0);
        bar_sync_n(1, NCONS);
        // epilogue mapping: warp w holds TMEM lanes 32 (w % 4) .. of block w / 4 = row i's block
        const int blk = warp >> 2;
        for (int k = 0; k < nh; ++k) {
            const int h = h_begin + k, db = k & 1;
            const float *f = fbuf + (k % NSC) * FST;
            uint8_t *dyb = dys + db * XB;
            // ---- head k's tiles landed: keep row i of x, zero padded rows of x and dy
            bool okk = ok && mbar_wait(&bar_xlo[db], (uint32_t)((k >> 1) & 1));
            if (NT == 2) okk = okk && mbar_wait(&bar_xhi, (uint32_t)(k & 1));
            uint8_t *xlo = xs + db * kTile;
            okk = okk && mbar_wait(&bar_dy[db], (uint32_t)((k >> 1) & 1));
            uint4 xr[8];  // row i of x; dy row i stays in shared memory until the epilogue
            if (i < Q) {
                const uint32_t xb = smem_u32(i < 128 ? xlo : xhi), yb = smem_u32(dyb);
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    const uint32_t ax = xb + sw128_chunk(i & 127, c8), ay = yb + sw128_chunk(i, c8);
                    uint4 xv = make_uint4(0, 0, 0, 0);
                    if (valid && okk) xv = ld_shared_v4(ax);
                    xr[c8] = xv;
                    if (!valid) {  // padding never reaches an MMA (non-finite values included)
                        st_shared_v4(ax, 0u, 0u, 0u, 0u);
                        st_shared_v4(ay, 0u, 0u, 0u, 0u);
                    }
                }
            }
            // ---- W^T, s-block 1 first (its MMAs run while s-block 0 is built)
            if (NT == 2 && okk) transform(f, 128 + r, 2 + hi);
            fence_async_smem();
            tc_fence_before();
            okk = bar_and(1, NCONS, okk);
            tc_fence_after();
            if (!okk) {
                ok = false;
                break;
            }
            if (tid == 0) {
                s_landed = k + 1;
                if (k > 0) {  // head k - 1's dx, staged in dy buffer (k - 1) & 1 by its epilogue
                    for (int j = 0; j < NT; ++j)
                        tma_store_4d(&maps.dx, dys + (db ^ 1) * XB + j * kTile, 0, h - 1, t0 + 128 * j, bi);
                    bulk_commit();
                }
            }
            if (NT == 2 && tid == 192) {  // warp 6's phase-B units are the lightest
                // z[1] = W^T[s-block 1] dy[t >= 128];  yo[1] = (s-block 1 part)
                const uint32_t ia = idesc_bf16(128, 64, false, true), ib = idesc_bf16(128, 64, true, true);
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16(tm + 64, sdesc_kmajor(smem_u32(tile_of(1, 2)), ks, kTile),
                             sdesc_mnmajor(smem_u32(dyb) + 128 * 128, ks, XB), ia, ks > 0);
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16(tm + 128 + 64, sdesc_mnmajor(smem_u32(tile_of(1, 2)), ks, kTile),
                             sdesc_mnmajor(smem_u32(xhi), ks, kTile), ib, ks > 0);
                mma_commit(&bar_a);  // the upper half of x is free once these complete
            }
            if (k + 2 < nh) {  // buffer (k + 2) % NSC was last read by head k - 1
                stash(k + 2);
                if (k + 3 < nh) fetch(k + 3);
            }
            // ---- W^T, s-block 0
            transform(f, r, 1 - hi);
            if (NT == 2) transform(f, r, 3 - hi);
            fence_async_smem();
            tc_fence_before();
            okk = bar_and(1, NCONS, true);
            tc_fence_after();
            // The s-block 0 MMAs, split between two issuing threads in warps 6 and 7 (the
            // lightest in this phase), each committing to bar_mma (two arrivals): the
            // commit of thread 192 also covers its s-block 1 MMAs issued above.
            if (tid == 224) {  // z[0] = W^T[s-block 0] dy
                const uint32_t ia = idesc_bf16(128, 64, false, true);
                for (int ks = 0; ks < Q / 16; ++ks)
                    mma_bf16(tm, sdesc_kmajor(smem_u32(tile_of(0, 0)), ks, kTile), sdesc_mnmajor(smem_u32(dyb), ks, XB),
                             ia, ks > 0);
                mma_commit(&bar_mma);
            }
            if (tid == 192) {  // yo[0] = W[t-block 0, s-block 0] x;  yo[1] += s-block 0 part
                const uint32_t ib = idesc_bf16(128, 64, true, true);
                for (int tb = 0; tb < NT; ++tb)
                    for (int ks = 0; ks < 8; ++ks)
                        mma_bf16(tm + 128 + 64 * tb, sdesc_mnmajor(smem_u32(tile_of(0, 2 * tb)), ks, kTile),
                                 sdesc_mnmajor(smem_u32(xlo), ks, kTile), ib, tb == 1 || ks > 0);
                mma_commit(&bar_mma);
                if (NT == 2 && k + 1 < nh) {  // the s-block 1 MMAs (issued a phase ago) are done: next upper half
                    if (mbar_wait(&bar_a, (uint32_t)(k & 1))) issue_xhi(k + 1);
                    else ok = false;
                }
            }
            if (tid == 0) {
                // the store of head k - 1's dx has read its buffer: dy of head k + 1 goes there
                if (k > 0) bulk_wait_read_all();
                if (k + 1 < nh) issue_dy(k + 1);
            }
            if (k + 1 < nh) derive(k + 1);  // while the MMAs run (raw scalars visible since barrier 1)
            // ---- epilogue of head k (row i): every MMA of the head is done, so dy may be overwritten
            okk = mbar_wait(&bar_mma, (uint32_t)(k & 1));
            tc_fence_after();
            if (!okk) ok = false;
            if (tid == 0 && okk && k + 2 < nh) issue_xlo(k + 2);  // the lower-half buffer of head k is free
            const float Dh = f[DOFF];
            const float2 Dh2 = make_float2(Dh, Dh);
            float2 src2 = make_float2(0.f, 0.f), dd2 = src2, tgt2 = src2;
            if (i < Q) {
                // z[i]: TMEM block blk (= i / 128), lanes 32 q4 + lane
                const uint32_t yb = smem_u32(dyb);
                uint4 dyr[8];
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) dyr[c8] = ld_shared_v4(yb + sw128_chunk(i, c8));
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float z[32];
                    tmem_ld32(tmem_addr(tm, 32 * q4, 64 * blk + 32 * hh), z);
                    uint32_t o[16];
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        const uint4 xv = xr[4 * hh + c8], yv = dyr[4 * hh + c8];
                        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, yw[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float2 x2 = bf2_to_f2(xw[j]), y2 = bf2_to_f2(yw[j]);
                            const float2 z2 = make_float2(z[8 * c8 + 2 * j], z[8 * c8 + 2 * j + 1]);
                            src2 = ffma2(x2, z2, src2);
                            dd2 = ffma2(x2, y2, dd2);
                            const float2 o2 = ffma2(Dh2, y2, z2);
                            o[4 * c8 + j] = valid ? pack_bf2(o2.x, o2.y) : 0u;
                        }
                    }
                    // dx row i over dy row i (read into registers above, by this thread only)
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
                        st_shared_v4(yb + sw128_chunk(i, 4 * hh + c4), o[4 * c4], o[4 * c4 + 1], o[4 * c4 + 2],
                                     o[4 * c4 + 3]);
                }
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float y[32];
                    tmem_ld32(tmem_addr(tm, 32 * q4, 128 + 64 * blk + 32 * hh), y);
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        const uint4 yv = dyr[4 * hh + c8];
                        const uint32_t yw[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            tgt2 = ffma2(bf2_to_f2(yw[j]), make_float2(y[8 * c8 + 2 * j], y[8 * c8 + 2 * j + 1]), tgt2);
                    }
                }
                const size_t cbase = ix_chunk(p, bi, h, c) * Q;
                const float src = src2.x + src2.y;
                p.ddt_main[cbase + i] = valid ? src / row_dt(f, i) : 0.f;  // the K3 backward adds its terms
                p.dcum_main[cbase + i] = valid ? (tgt2.x + tgt2.y) - src : 0.f;
            }
            fence_async_smem();  // the staged dx rows are read by the next head's TMA store
            float dd = dd2.x + dd2.y;
            dd = warp_sum(dd);
            if (lane == 0) p.dD_part[(((size_t)bi * p.n + c) * p.H + h) * p.dD_per + warp] = dd;
        }
    }
    tc_fence_before();
    ok = __syncthreads_and(ok ? 1 : 0) != 0;
    tc_fence_after();
    if (!ok && tid == 0) flag_timeout(p);
    if (ok && tid == 0) {  // the last head's dx
        for (int j = 0; j < NT; ++j)
            tma_store_4d(&maps.dx, dys + ((nh - 1) & 1) * XB + j * kTile, 0, h_begin + nh - 1, t0 + 128 * j, bi);
        bulk_commit();
    }
    if (tid == 0) bulk_wait_all();
    // loads issued for heads that were never consumed have to land before exit
    if (tid == 0) {
        mbar_wait(&bar_cb, 0);  // landed long ago unless the kernel gave up early
        for (int k = s_landed; k < s_lo_issued; ++k) mbar_wait(&bar_xlo[k & 1], (uint32_t)((k >> 1) & 1));
        if (s_hi_issued > s_landed) mbar_wait(&bar_xhi, (uint32_t)((s_hi_issued - 1) & 1));
        if (NT == 2 && s_landed > 0) mbar_wait(&bar_a, (uint32_t)((s_landed - 1) & 1));
        for (int k = s_landed; k < s_dy_issued; ++k) mbar_wait(&bar_dy[k & 1], (uint32_t)((k >> 1) & 1));
    }
    tc_sync();
    if (warp == 0) tmem_dealloc(tm, 512);
}

// ====================================================================== group backward
// G1: CTA per (b, chunk, group, head slice, 128 x 128 block of d_cb on or below
// the diagonal), 256 threads: thread = one row t of the block (its TMEM lane)
// and 64 of its columns.  Accumulates, over the slice's heads and in registers,
//   d_cb[t, s] = sum_h dt_h[s] exp(cumA_h[t] - cumA_h[s]) dW_h[t, s]     (s <= t)
// where dW_h = dy_h x_h^T is one MMA per head into one of two TMEM buffers, so
// the MMA of head k + 1 runs during the epilogue of head k.  dy / x tiles come
// through a three-stage TMA ring (head k + 3 is requested once MMA k is done, so
// a load has two heads' work to land in); per-head scalars are fetched into registers
// three heads ahead and staged in shared memory.  The slices' fp32 partials
// are summed, in slice order, by the last CTA of the block to finish, which
// writes d_cb in bf16 (the operand type of the next kernel).  The decay is factored through pivots, both factors <= 1:
// cumA at the last row of the column block for the block below the diagonal;
// inside a diagonal block cumA[64 j + 63] for 64-wide column blocks left of
// the row's own, cumA[16 v + 15] for 16-wide sub-blocks left of the row's own;
// only the row's own 16-wide sub-block takes one exponential per element.
template <int Q>
__global__ void __launch_bounds__(kThreadsWide, 2) tc_bwd_dcb_kernel(const Params p, const __grid_constant__ TcMaps maps) {
    constexpr int NT = Q / 128;
    constexpr int NBLK = NT * (NT + 1) / 2;
    constexpr uint32_t STG = 2 * kTile;  // dy rows of the t-block, x rows of the s-block
    constexpr int NST = 3;               // TMA stages: head k + 3 is requested once MMA k is done
    constexpr int NSC = 3;               // scalar buffers
    // own-sub-block column table and fast flags after the pivots (16-byte aligned)
    constexpr int OWNOFF = (4 * Q + Q / 64 + Q / 16 + 3) & ~3, FLOFF = OWNOFF + Q;
    constexpr int FST = (FLOFF + Q / 16 + 3) & ~3;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    float *fbuf = reinterpret_cast<float *>(sm + NST * STG);  // [NSC][cum | dt | g64 | g16 | piv64 | piv16 | own | flags]
    __shared__ uint64_t bar_tma[NST], bar_mma[NST];
    __shared__ uint32_t s_tmem;
    __shared__ int s_last;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, hf = warp >> 2;
    int idx = blockIdx.x;
    const int blk = idx % NBLK;
    idx /= NBLK;
    const int tb = blk == 0 ? 0 : 1, sk = blk == 2 ? 1 : 0;
    const int slice = idx % p.nslice_cb;
    idx /= p.nslice_cb;
    const int g = idx % p.G, c = (idx / p.G) % p.n, bi = idx / (p.G * p.n);
    const int t0 = c * Q;
    const int vrows = min(Q, valid_len_of(p, bi) - t0);
    const int per = (p.hpg + p.nslice_cb - 1) / p.nslice_cb;
    const int h_begin = g * p.hpg + slice * per;
    const int nh = max(0, min(g * p.hpg + p.hpg, h_begin + per) - h_begin);
    const int tl = 32 * q4 + lane, t = 128 * tb + tl;  // this thread's row
    // and its columns: two 32-wide pieces, 32 hf + 64 j (j = 0, 1) inside the block,
    // so that on a diagonal block every warp has at most one piece on the diagonal
    auto colp = [&](int j) { return 32 * hf + 64 * j; };
    const size_t cbase = ((size_t)bi * p.n + c) * p.G + g;  // (b, chunk, group)
    const size_t pstride = (size_t)p.b * p.n * p.G * Q * Q;   // between slices' partials
    const size_t rbase = cbase * Q * Q + (size_t)t * Q + 128 * sk;  // this thread's row of the block
    float acc[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) acc[i] = 0.f;
    auto write_bf16 = [&](const float *v) {
#pragma unroll
        for (int j = 0; j < 2; ++j) store_row32_bf16(p.d_cb_bf + rbase + colp(j), v + 32 * j);
    };
    if (vrows <= 128 * tb) {  // the whole block lies past valid_len: zeros, written once
        if (slice == 0) write_bf16(acc);
        return;
    }
    const bool diag = tb == sk;
    // --- per-head scalars: registers -> shared buffer k % NSC -> derived tables
    // two register sets (head k in set k & 1), so a head's global loads are
    // issued two heads before they are staged
    float r_cum[2] = {0.f, 0.f}, r_dt[2] = {0.f, 0.f};
    auto fetch = [&](int k) {
        if (tid < Q) {
            const int h = h_begin + k;
            r_cum[k & 1] = p.cumA[ix_chunk(p, bi, h, c) * Q + tid];
            r_dt[k & 1] = tid < vrows ? p.dt[ix_dt(p, bi, h, t0 + tid)] : 0.f;
        }
    };
    auto stash = [&](int k) {
        float *f = fbuf + (k % NSC) * FST;
        if (tid < Q) {
            f[tid] = r_cum[k & 1];
            f[Q + tid] = r_dt[k & 1];
        }
    };
    auto derive = [&](int k) {  // diagonal blocks only
        float *f = fbuf + (k % NSC) * FST;
        const int l = 128 * sk + (tid & 127);  // a column of this block
        if (tid < 128) {
            const float cl = f[l], d = f[Q + l];
            f[2 * Q + l] = d * __expf(f[l | 63] - cl);
            f[3 * Q + l] = d * __expf(f[l | 15] - cl);
            if ((l & 63) == 63) f[4 * Q + (l >> 6)] = cl;
            if ((l & 15) == 15) f[4 * Q + Q / 64 + (l >> 4)] = cl;
            // own sub-block: dt_s exp(cumA[16 v] - cumA_s) (>= 0, <= e^64 dt_s where used)
            f[OWNOFF + l] = d * __expf(f[l & ~15] - cl);
            if ((l & 15) == 0) f[FLOFF + (l >> 4)] = f[l] - f[l + 15] < 64.f ? 1.f : 0.f;
        }
    };
    const int xrow = vrows - 128 * sk;  // valid rows of the x tile (> 0)
    auto issue = [&](int k) {
        const int h = h_begin + k, st = k % NST;
        uint8_t *dys = sm + st * STG, *xs = dys + kTile;
        mbar_arrive_expect_tx(&bar_tma[st], STG);
        tma_load_4d(dys, &maps.dy, &bar_tma[st], 0, h, t0 + 128 * tb, bi);
        tma_load_4d(xs, &maps.x, &bar_tma[st], 0, h, t0 + 128 * sk, bi);
    };
    if (tid == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&bar_tma[i], 1);
            mbar_init(&bar_mma[i], 1);
        }
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&s_tmem, 256);
    tc_sync();
    const uint32_t tm = s_tmem;
    int issued = 0, landed = 0;  // TMA bookkeeping of thread 0
    if (tid == 0)
        for (; issued < min(nh, NST); ++issued) issue(issued);
    bool ok = true, okt = true;
    if (!diag) {
        // ---- the block below the diagonal: its pivot P = cumA[128 sk + 127] (the last
        // column) lies between every s and t of the block, so the decay factors into a
        // dy row scale and an x row scale (both <= 1), and the sum over heads is one
        // long-K accumulation in TMEM with no per-head epilogue:
        //   d_cb[t, s] = sum_h sum_p (dy_h[t, p] exp(cumA_t - P)) (x_h[s, p] dt_s exp(P - cumA_s))
        // Thread r < 128 scales dy row 128 tb + r, thread 128 + r scales x row 128 sk + r.
        const int r = tid & 127;
        const bool on_dy = tid < 128;
        const int row = on_dy ? 128 * tb + r : 128 * sk + r;  // chunk row
        const bool rv = row < vrows;
        float cr = 0.f, dr = 0.f, pr = 0.f, cn = 0.f, dn = 0.f, pn = 0.f;
        auto fetch_o = [&](int k, float &cc, float &dd, float &pp) {
            const size_t ck = ix_chunk(p, bi, h_begin + k, c) * Q;
            pp = p.cumA[ck + 128 * sk + 127];
            cc = p.cumA[ck + row];
            dd = (!on_dy && rv) ? p.dt[ix_dt(p, bi, h_begin + k, t0 + row)] : 0.f;
        };
        if (nh > 0) fetch_o(0, cr, dr, pr);
        if (nh > 1) fetch_o(1, cn, dn, pn);
        for (int k = 0; k < nh && ok; ++k) {
            const int st = k % NST;
            const float fct = on_dy ? __expf(cr - pr) : dr * __expf(pr - cr);
            cr = cn;
            dr = dn;
            pr = pn;
            if (k + 2 < nh) fetch_o(k + 2, cn, dn, pn);
            const bool okk = mbar_wait(&bar_tma[st], (uint32_t)((k / NST) & 1));
            if (tid == 0 && okk) landed = k + 1;
            if (okk) scale_row_bf16x2(sm + st * STG + (on_dy ? 0 : kTile), r, fct, rv);
            fence_async_smem();
            tc_fence_before();
            ok = __syncthreads_and(okk ? 1 : 0) != 0;
            tc_fence_after();
            if (ok && tid == 0) {
                const uint32_t dys = smem_u32(sm + st * STG), xs = dys + kTile;
                const uint32_t id = idesc_bf16(128, 128, false, false);
#pragma unroll
                for (int ks = 0; ks < kP / 16; ++ks)
                    mma_bf16(tm, sdesc_kmajor(dys, ks, kTile), sdesc_kmajor(xs, ks, kTile), id, k > 0 || ks > 0);
                mma_commit(&bar_mma[st]);
                // the stage of head k - 1 takes head k - 1 + NST once MMA k - 1 has read it
                // (MMA k stays queued behind it meanwhile)
                if (k >= 1 && k - 1 + NST < nh) {
                    if (mbar_wait(&bar_mma[(k - 1) % NST], (uint32_t)(((k - 1) / NST) & 1))) {
                        issue(k - 1 + NST);
                        issued = k + NST;
                    } else {
                        okt = false;
                    }
                }
            }
        }
        if (ok && nh > 0) okt = mbar_wait(&bar_mma[(nh - 1) % NST], (uint32_t)(((nh - 1) / NST) & 1)) && okt;
        tc_fence_after();
        if (ok && nh > 0) {
            tmem_ld32(tmem_addr(tm, 32 * q4, colp(0)), acc);
            tmem_ld32(tmem_addr(tm, 32 * q4, colp(1)), acc + 32);
        }
    } else {
        if (nh > 0) {
            fetch(0);
            stash(0);
        }
        if (nh > 1) {
            fetch(1);
            stash(1);
        }
        if (nh > 2) fetch(2);
        if (nh > 3) fetch(3);
        __syncthreads();
        if (nh > 0) derive(0);
        // Wait for head k's tiles, zero x rows past valid_len, and (thread 0) issue
        // dW_k into TMEM buffer k & 1.  Returns a CTA-uniform status.
        auto land_and_mma = [&](int k, bool ok_in) -> bool {
            const int st = k % NST, tb2 = k & 1;  // TMA stage, TMEM buffer
            bool ok = ok_in && mbar_wait(&bar_tma[st], (uint32_t)((k / NST) & 1));
            if (tid == 0 && ok) landed = k + 1;
            if (ok && xrow < 128) {
                zero_rows_from(sm + st * STG + kTile, 128, xrow);
                fence_async_smem();
            }
            tc_fence_before();
            ok = __syncthreads_and(ok ? 1 : 0) != 0;
            tc_fence_after();
            if (tid == 0 && ok) {
                const uint32_t dys = smem_u32(sm + st * STG), xs = dys + kTile;
                const uint32_t id = idesc_bf16(128, 128, false, false);
#pragma unroll
                for (int ks = 0; ks < kP / 16; ++ks)
                    mma_bf16(tm + 128 * tb2, sdesc_kmajor(dys, ks, kTile), sdesc_kmajor(xs, ks, kTile), id, ks > 0);
                mma_commit(&bar_mma[tb2]);
            }
            return ok;
        };
        ok = nh > 0 ? land_and_mma(0, true) : true;
        const bool row_ok = t < vrows;
        const int tr = tl >> 6, u16 = (tl & 63) >> 4;  // 64-row block and 16-row sub-block (diagonal blocks)
        for (int k = 0; k < nh && ok; ++k) {
            const int st = k & 1;
            if (k + 1 < nh) {
                ok = land_and_mma(k + 1, okt);  // the epilogue of head k - 1 has left buffer (k + 1) & 1
            } else {
                ok = __syncthreads_and(okt ? 1 : 0) != 0;
            }
            if (k + 2 < nh) stash(k + 2);
            if (k + 4 < nh) fetch(k + 4);  // set k & 1, just staged
            if (k + 1 < nh) derive(k + 1);
            okt = ok && mbar_wait(&bar_mma[st], (uint32_t)((k >> 1) & 1));
            tc_fence_after();
            if (tid == 0 && okt && k + NST < nh) {
                issue(k + NST);  // the stage of head k is free: MMA k has read it
                issued = k + NST + 1;
            }
            const float *f = fbuf + (k % NSC) * FST;
            const float ct = f[t];
            // ---- epilogue of head k: acc += dt_s exp(cumA_t - cumA_s) dW[t, s]
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float dw[32];
                tmem_ld32(tmem_addr(tm, 32 * q4, 128 * st + colp(half)), dw);
                const int s0 = 128 * sk + colp(half);  // the piece's 64-column block is `half`
                float *a = acc + 32 * half;
                if (row_ok && (!diag || half < tr)) {
                    // one pivot for all 32 columns
                    const float e = __expf(ct - (diag ? f[4 * Q + (s0 >> 6)] : f[128 * sk + 127]));
                    const float4 *gv = reinterpret_cast<const float4 *>(f + 2 * Q + s0);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 gq = gv[i];
                        a[4 * i + 0] = fmaf(dw[4 * i + 0] * gq.x, e, a[4 * i + 0]);
                        a[4 * i + 1] = fmaf(dw[4 * i + 1] * gq.y, e, a[4 * i + 1]);
                        a[4 * i + 2] = fmaf(dw[4 * i + 2] * gq.z, e, a[4 * i + 2]);
                        a[4 * i + 3] = fmaf(dw[4 * i + 3] * gq.w, e, a[4 * i + 3]);
                    }
                } else if (row_ok && half == tr) {
#pragma unroll
                    for (int v2 = 0; v2 < 2; ++v2) {
                        const int sv = s0 + 16 * v2, v16 = 2 * hf + v2;
                        float *av = a + 16 * v2;
                        const float *dv = dw + 16 * v2;
                        if (v16 < u16) {
                            const float e = __expf(ct - f[4 * Q + Q / 64 + (sv >> 4)]);
                            const float4 *gv = reinterpret_cast<const float4 *>(f + 3 * Q + sv);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const float4 gq = gv[i];
                                av[4 * i + 0] = fmaf(dv[4 * i + 0] * gq.x, e, av[4 * i + 0]);
                                av[4 * i + 1] = fmaf(dv[4 * i + 1] * gq.y, e, av[4 * i + 1]);
                                av[4 * i + 2] = fmaf(dv[4 * i + 2] * gq.z, e, av[4 * i + 2]);
                                av[4 * i + 3] = fmaf(dv[4 * i + 3] * gq.w, e, av[4 * i + 3]);
                            }
                        } else if (v16 == u16) {
                            if (f[FLOFF + (t >> 4)] != 0.f) {
                                // span below e^64: factored through cumA[16 v] (row factor <= 1)
                                const float e = __expf(ct - f[sv]);
                                const float4 *gv = reinterpret_cast<const float4 *>(f + OWNOFF + sv);
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const float4 gq = gv[i];
                                    const float g4[4] = {gq.x, gq.y, gq.z, gq.w};
#pragma unroll
                                    for (int c4 = 0; c4 < 4; ++c4)
                                        if (sv + 4 * i + c4 <= t) av[4 * i + c4] = fmaf(dv[4 * i + c4] * g4[c4], e, av[4 * i + c4]);
                                }
                            } else {
#pragma unroll
                                for (int i = 0; i < 16; ++i) {
                                    const int s = sv + i;
                                    if (s <= t) av[i] = fmaf(dv[i] * f[Q + s], __expf(ct - f[s]), av[i]);
                                }
                            }
                        }
                    }
                }
            }
        }
    }
    tc_fence_before();
    ok = __syncthreads_and(ok && okt ? 1 : 0) != 0;
    tc_fence_after();
    if (!ok && tid == 0) flag_timeout(p);
    if (tid == 0)
        for (int k = landed; k < issued; ++k) mbar_wait(&bar_tma[k % NST], (uint32_t)((k / NST) & 1));
    tc_sync();
    if (warp == 0) tmem_dealloc(tm, 256);
    if (!ok) return;
    // ---- sum over head slices: every slice writes its fp32 partial; the last
    // to arrive adds them in slice order (the same sum whichever CTA is last)
    // and writes the block in bf16
    const int ns = p.nslice_cb;
    if (ns > 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            reinterpret_cast<float4 *>(p.d_cb + slice * pstride + rbase + colp(i >> 3))[i & 7] =
                make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
        __threadfence();
        __syncthreads();
        if (tid == 0) s_last = atomicAdd(p.cb_count + cbase * NBLK + blk, 1) == ns - 1;
        __syncthreads();
        if (!s_last) return;
        __threadfence();
        // in place, four columns at a time: acc <- sum over slices in slice order
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int sl = 0; sl < ns; ++sl) {
                const float4 u = sl == slice ? make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3])
                                             : __ldcg(reinterpret_cast<const float4 *>(p.d_cb + sl * pstride + rbase + colp(i >> 3)) + (i & 7));
                v.x += u.x;
                v.y += u.y;
                v.z += u.z;
                v.w += u.w;
            }
            acc[4 * i] = v.x;
            acc[4 * i + 1] = v.y;
            acc[4 * i + 2] = v.z;
            acc[4 * i + 3] = v.w;
        }
        write_bf16(acc);
        if (tid == 0) p.cb_count[cbase * NBLK + blk] = 0;  // ready for the next call
    } else {
        write_bf16(acc);
    }
}

// G2: CTA per (b, chunk, group, head slice): 8 consumer warps and one TMA
// producer warp.  TMEM: dC accumulators at [tb*128), dB accumulators at
// [NT*128 + mb*128).
//   slice 0 only:  dC += d_cb B        (A = d_cb K-major, B = B MN-major)
//                  dB += d_cb^T C      (A = d_cb MN-major view, B = C MN-major)
//   every slice:   dC += sum_h (dy_h exp(cumA_h)) s_in_h      (long-K over heads)
//                  dB += sum_h (x_h bbs_h) d_intra_h
// The producer refills a stage as soon as the MMAs of the head that used it
// complete; consumer thread t scales row t of the landed dy / x tiles (its
// scalars fetched into registers two heads ahead) and one thread issues the
// MMAs, so the loop runs at the rate the tiles arrive.  Writes the fp32
// partial sums of the slice.
template <int Q>
__global__ void __launch_bounds__(kThreadsWide + 32, 1) tc_bwd_dbc_kernel(const Params p, const __grid_constant__ TcMaps maps) {
    constexpr int NT = Q / 128;
    constexpr uint32_t XB = Q * 128, RB = Q * 128, SB = 64 * 128;
    constexpr uint32_t STG = 2 * XB + 4 * SB;  // dy, x, s_in (2 r-blocks), d_intra (2 r-blocks)
    constexpr uint32_t NCOL = NT == 2 ? 512 : 256;
    constexpr uint32_t DBCOL = NT * 128;
    constexpr int NCONS = kThreadsWide;         // consumer threads; the producer warp follows
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    __shared__ uint64_t bar_tma[2], bar_mma[2], bar_scaled[2], bar_a;
    __shared__ uint32_t s_tmem;
    __shared__ int s_issued, s_landed, s_perr;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, hf = (warp >> 2) & 1;
    int idx = blockIdx.x;
    const int slice = idx % p.nslice;
    idx /= p.nslice;
    const int g = idx % p.G, c = (idx / p.G) % p.n, bi = idx / (p.G * p.n);
    const int t0 = c * Q;
    const int vrows = min(Q, valid_len_of(p, bi) - t0);
    // slice j takes heads j, j + nslice, ... of the group: CTAs running side by
    // side read neighbouring heads, i.e. neighbouring 128-byte pieces of each token row
    const int h_begin = g * p.hpg + slice;
    auto head = [&](int k) { return h_begin + k * p.nslice; };
    const size_t pstride = (size_t)p.b * p.n * p.G * Q * kN;
    float *outC = p.dBC_part + ((size_t)slice * 2 + 0) * pstride + (((size_t)bi * p.n + c) * p.G + g) * (size_t)Q * kN;
    float *outB = p.dBC_part + ((size_t)slice * 2 + 1) * pstride + (((size_t)bi * p.n + c) * p.G + g) * (size_t)Q * kN;
    const bool do_k2 = slice == 0;
    const int nh = max(0, (p.hpg - slice + p.nslice - 1) / p.nslice);
    if (vrows <= 0 || (!do_k2 && nh == 0)) {
        for (int i = tid; i < Q * kN; i += blockDim.x) {
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
        mbar_init(&bar_scaled[0], NCONS / 32);
        mbar_init(&bar_scaled[1], NCONS / 32);
        mbar_init(&bar_a, 1);
        mbar_fence_init();
        s_issued = 0;
        s_landed = 0;
        s_perr = 0;
    }
    if (warp == 0) tmem_alloc(&s_tmem, NCOL);
    tc_sync();
    const uint32_t tm = s_tmem;
    bool ok = true;
    uint32_t pa = 0;  // bar_a phase
    bool have_acc = false;
    if (do_k2) {
        // d_cb (bf16 [t][s], 64-column blocks of Q rows; only blocks on or
        // below the diagonal are loaded or read) and B, then C, in one buffer
        uint8_t *dcb = sm, *BCs = sm + (uint32_t)Q * Q * 2;
        if (tid == 0) {
            mbar_arrive_expect_tx(&bar_a, NT * (NT + 1) * kTile + 2 * RB);
            const int row0 = ((bi * p.n + c) * p.G + g) * Q;
            for (int tb = 0; tb < NT; ++tb)
                for (int j = 0; j < 2 * (tb + 1); ++j)
                    tma_load_2d(dcb + j * RB + tb * kTile, &maps.dcb, &bar_a, 64 * j, row0 + 128 * tb);
            for (int rb = 0; rb < 2; ++rb)
                for (int j = 0; j < NT; ++j)
                    tma_load_4d(BCs + rb * RB + j * kTile, &maps.B, &bar_a, 64 * rb, g, t0 + 128 * j, bi);
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
        tc_sync();  // the stage area is free again
        have_acc = true;
    }
    if (warp == NCONS / 32) {
        // ---- producer: TMA for head k + 1 once head k - 1's MMAs are done (its
        // stage is free), and the MMAs of head k once the consumers have scaled it
        if (lane == 0 && ok) {
            auto issue = [&](int k) {
                const int h = head(k), st = k & 1;
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
                s_issued = k + 1;
            };
            if (nh > 0) issue(0);
            if (nh > 1) issue(1);
            for (int k = 0; k < nh; ++k) {
                const int st = k & 1;
                // stage (k + 1) & 1 held head k - 1: refill it as soon as that head's MMAs are
                // done (issued just before), while the consumers are still scaling head k
                if (k >= 1 && k + 1 < nh) {
                    if (!mbar_wait(&bar_mma[(k - 1) & 1], (uint32_t)(((k - 1) >> 1) & 1))) {
                        s_perr = 1;
                        break;
                    }
                    issue(k + 1);
                }
                if (!mbar_wait(&bar_scaled[st], (uint32_t)((k >> 1) & 1)) || s_perr) {
                    s_perr = 1;
                    break;
                }
                s_landed = k + 1;
                tc_fence_after();
                uint8_t *base = sm + st * STG;
                uint8_t *dys = base, *xs = base + XB, *sis = base + 2 * XB, *dis = sis + 2 * SB;
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
            }
        }
    } else if (ok) {
        // ---- consumers: thread t owns token row t of the chunk
        const int t = tid;
        const bool valid = t < vrows;
        float c_cur = 0.f, d_cur = 0.f, e_cur = 0.f, c_nx = 0.f, d_nx = 0.f, e_nx = 0.f;
        auto fetch = [&](int k, float &cc, float &dd, float &ce) {
            const size_t ck = ix_chunk(p, bi, head(k), c);
            ce = p.endA[ck];
            cc = t < Q ? p.cumA[ck * Q + t] : 0.f;
            dd = valid ? p.dt[ix_dt(p, bi, head(k), t0 + t)] : 0.f;
        };
        if (nh > 0) fetch(0, c_cur, d_cur, e_cur);
        if (nh > 1) fetch(1, c_nx, d_nx, e_nx);
        for (int k = 0; k < nh; ++k) {
            const int st = k & 1;
            uint8_t *base = sm + st * STG;
            uint8_t *dys = base, *xs = base + XB;
            const float e_row = __expf(c_cur);                // dy row factor exp(cumA_t)
            const float b_row = d_cur * __expf(e_cur - c_cur);  // x row factor bbs_t
            c_cur = c_nx;
            d_cur = d_nx;
            e_cur = e_nx;
            if (k + 2 < nh) fetch(k + 2, c_nx, d_nx, e_nx);
            const bool okk = mbar_wait(&bar_tma[st], (uint32_t)((k >> 1) & 1));
            if (okk && t < Q) {
                scale_row_bf16x2(dys, t, e_row, valid);
                scale_row_bf16x2(xs, t, b_row, valid);
            }
            if (!okk) s_perr = 1;
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_scaled[st]);  // the producer issues head k's MMAs
        }
        // the last head's MMAs complete after all earlier ones
        if (nh > 0) ok = mbar_wait(&bar_mma[(nh - 1) & 1], (uint32_t)(((nh - 1) >> 1) & 1)) && ok;
    }
    tc_fence_before();
    ok = __syncthreads_and(ok && s_perr == 0 ? 1 : 0) != 0;
    tc_fence_after();
    if (tid < NCONS) {
        if (ok) {
            // fp32 partials through the (now idle) stage area: 128-row x 32-column
            // boxes in the 128-byte swizzled layout of the store's tensor map (so
            // the row-per-thread shared stores do not collide on banks), written
            // out by TMA, dC first, then dB
            constexpr int NBOX = NT * 4;  // boxes per output
            const int row = 32 * q4 + lane;
            const long long rows_out = (long long)p.b * p.n * p.G * Q;
            const long long rbase = (((long long)bi * p.n + c) * p.G + g) * Q;
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                uint8_t *boxes = sm + (NT == 2 ? 0 : which * NBOX * kTile);
                if (which == 1 && NT == 2) {  // the dC boxes must have been read out first
                    if (tid == 0) bulk_wait_read_all();
                    bar_sync_n(1, NCONS);
                }
#pragma unroll 1
                for (int tb = 0; tb < NT; ++tb)
#pragma unroll 1
                    for (int r0 = 64 * hf; r0 < 64 * hf + 64; r0 += 32) {
                        float v[32];
                        tmem_ld32(tmem_addr(tm, 32 * q4, (which ? DBCOL : 0) + tb * 128 + r0), v);
                        const uint32_t bb = smem_u32(boxes + (tb * 4 + r0 / 32) * kTile) + (uint32_t)row * 128u;
#pragma unroll
                        for (int c4 = 0; c4 < 8; ++c4)
                            st_shared_v4(bb + (uint32_t)((c4 ^ (row & 7)) * 16), __float_as_uint(v[4 * c4]),
                                         __float_as_uint(v[4 * c4 + 1]), __float_as_uint(v[4 * c4 + 2]),
                                         __float_as_uint(v[4 * c4 + 3]));
                    }
                fence_async_smem();
                bar_sync_n(1, NCONS);
                if (tid == 0) {
                    const long long y0 = ((long long)slice * 2 + which) * rows_out + rbase;
                    for (int bx = 0; bx < NBOX; ++bx)
                        tma_store_2d(&maps.part, boxes + bx * kTile, 32 * (bx & 3), (int)(y0 + 128 * (bx >> 2)));
                    bulk_commit();
                }
            }
            if (tid == 0) bulk_wait_all();
        } else if (tid == 0) {
            flag_timeout(p);
        }
    }
    // loads issued for heads that were never consumed have to land before exit
    if (tid == 0)
        for (int k = s_landed; k < s_issued; ++k) mbar_wait(&bar_tma[k & 1], (uint32_t)((k >> 1) & 1));
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
        // up to 8 slices' loads in flight before they are summed (in slice order)
#pragma unroll 1
        for (int s0 = 0; s0 < p.nslice; s0 += 8) {
            float4 av[8], bv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (s0 + j < p.nslice) {
                    av[j] = __ldcs(reinterpret_cast<const float4 *>(p.dBC_part + ((s0 + j) * 2 + 0) * pstride + off));
                    bv[j] = __ldcs(reinterpret_cast<const float4 *>(p.dBC_part + ((s0 + j) * 2 + 1) * pstride + off));
                }
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (s0 + j < p.nslice) {
                    sc.x += av[j].x; sc.y += av[j].y; sc.z += av[j].z; sc.w += av[j].w;
                    sb.x += bv[j].x; sb.y += bv[j].y; sb.z += bv[j].z; sb.w += bv[j].w;
                }
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

// ====================================================================== state moments
// Raw moments of the per-token states (burn-mamba, "modules/state_moments.rs":
// m2 = sum_t S_t^T S_t over the valid tokens, pooling the P rows of each
// state, and m1 = sum_t sum_p S_t[p, :]) in closed form per 128-token chunk,
// so that no per-token state is formed.  CTA per (b, h, range of chunks), 256
// threads; the chunk-input states s come from the chunk-state scan run at
// chunk 128.  With c = cumA, S_t = exp(c_t) s + sum_{u <= t} w_tu x_u B_u^T,
// w_tu = exp(c_t - c_u) dt_u, the chunk's sum over its valid tokens t < vr is
//   c0 s^T s + U^T D B + B^T D U + B^T (K o G) B,
//   U = X s, D = diag(alpha), alpha_u = dt_u exp(c_u) sigma_u, c0 = sum_t exp(2 c_t),
//   G = X X^T, K[u, v] = sum_{t >= max(u, v)} w_tu w_tv
//                      = dt_u dt_v sigma_m exp(2 c_m - c_u - c_v), m = max(u, v),
//   sigma_m = sum_{t = m}^{vr - 1} exp(2 (c_t - c_m))  (every exponent <= 0).
// Three MMAs per chunk (bf16 operands, fp32 in TMEM):
//   MMA1  G = X X^T                                (TMEM columns 0..127)
//   MMA2  Y = F B + (2 alpha o X) s,  F = K o G    (columns 128..255)
//   MMA3  A += B^T Y + (sqrt(c0) s)^T (sqrt(c0) s) (columns 256..383, over all chunks)
// so that A + A^T = 2 (chunk sums): the range's partial A (stored transposed)
// and m1 go to the workspace and ssd_moments_reduce sums the ranges in order
// and symmetrises.  m1 += sum_u beta_u (sum_p x_u[p]) B_u + (sum_t exp(c_t)) sum_p s[p, :]
// with beta_u = dt_u tau_u, tau_u = sum_{t >= u} exp(c_t - c_u), rides along
// MMA3 as a 144th column (w1 = beta * row sums of x beside Y, and
// sum exp(c) / sqrt(c0) beside sqrt(c0) s).  sigma and tau are suffix sums of the recurrences
// sigma_t = 1 + exp(2 (c_{t+1} - c_t)) sigma_{t+1}, tau_t = 1 + exp(c_{t+1} - c_t) tau_{t+1}:
// one warp composes their affine maps (four tokens per lane, then a suffix scan
// across the lanes).
__device__ __forceinline__ void affine_compose(float &A1, float &B1, float A2, float B2) {
    // (x -> B1 + A1 x) after (x -> B2 + A2 x)
    B1 = fmaf(A1, B2, B1);
    A1 = A1 * A2;
}

constexpr int kMomMain = 512;     // 16 warps: 4 per TMEM lane quadrant
constexpr int kMomThreads = kMomMain + 128;  // + 4 scalar warps, a chunk ahead

__global__ void __launch_bounds__(kMomThreads, 1) tc_moments_kernel(const Params p, const __grid_constant__ TcMaps maps) {
    constexpr int Q = 128;
    constexpr uint32_t XT = 128 * 128;  // [128 tokens][64] bf16
    constexpr uint32_t BT = 2 * XT;     // B: two 64-column halves
    constexpr uint32_t ST = 64 * 128;   // one [64 p][64 r] half of s
    constexpr int ISSUER = 128;         // the thread that issues TMA and MMAs (warp 4: not a scan warp)
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    // X x 2 | B x 2 | s | sqrt(c0) s | F | Y | 2 alpha X.  MMA3 reads N = 144 columns:
    // Y's two blocks then the (dead by then) 2 alpha X tile holding the w1 column,
    // and sqrt(c0) s's two blocks then the (dead) first 8 KB of F holding the
    // sum_t exp(c_t) / sqrt(c0) column; column 128 of A accumulates m1.
    uint8_t *Xs = sm, *Bs = Xs + 2 * XT, *Ss = Bs + 2 * BT, *Ssc = Ss + 2 * ST, *Fs = Ssc + 2 * ST;
    uint8_t *Ys = Fs + 2 * XT, *XAs = Ys + 2 * XT;
    __shared__ uint64_t bar_xb[2], bar_s, bar_g, bar_y, bar_a, bar_tab[2], bar_tabfree[2];
    __shared__ uint32_t s_tmem;
    // per-chunk tables, double-buffered: written by the scalar warps a chunk ahead
    __shared__ float t_c[2][Q], t_dt[2][Q], t_ds[2][Q], t_al2[2][Q], t_w1[2][Q], t_rs[Q];
    __shared__ float s_c0[2], s_asum[2];
    __shared__ int s_abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, cq = warp >> 2;  // TMEM lane quadrant, 32-column quarter
    int idx = blockIdx.x;
    const int range = idx % p.mom_ranges;
    const int bh = idx / p.mom_ranges, h = bh % p.H, bi = bh / p.H, g = h / p.hpg;
    const int V = valid_len_of(p, bi);
    const int nv = (V + Q - 1) / Q;
    const int per = (p.n + p.mom_ranges - 1) / p.mom_ranges;
    const int c_begin = range * per, c_end = min(nv, c_begin + per);
    const int nk = max(0, c_end - c_begin);
    float *Apart = p.mom_A + ((size_t)range * p.b * p.H + bh) * (size_t)kN * kN;
    float *m1part = p.mom_m1 + ((size_t)range * p.b * p.H + bh) * kN;
    if (nk == 0) {
        for (int i = tid; i < kN * kN; i += blockDim.x) Apart[i] = 0.f;
        if (tid < kN) m1part[tid] = 0.f;
        return;
    }
    auto issue_xb = [&](int k) {
        const int c = c_begin + k, buf = k & 1;
        mbar_arrive_expect_tx(&bar_xb[buf], XT + BT);
        tma_load_4d(Xs + buf * XT, &maps.x, &bar_xb[buf], 0, h, Q * c, bi);
        for (int rb = 0; rb < 2; ++rb) tma_load_4d(Bs + buf * BT + rb * XT, &maps.B, &bar_xb[buf], 64 * rb, g, Q * c, bi);
    };
    auto issue_s = [&](int k) {
        const int sidx = (bi * p.n + c_begin + k) * p.H + h;
        mbar_arrive_expect_tx(&bar_s, 2 * ST);
        for (int rb = 0; rb < 2; ++rb) tma_load_3d(Ss + rb * ST, &maps.st, &bar_s, 64 * rb, 0, sidx);
    };
    if (tid == 0) {
        mbar_init(&bar_xb[0], 1);
        mbar_init(&bar_xb[1], 1);
        mbar_init(&bar_s, 1);
        mbar_init(&bar_g, 1);
        mbar_init(&bar_y, 1);
        mbar_init(&bar_a, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_tab[i], 1);
            mbar_init(&bar_tabfree[i], 1);
        }
        mbar_fence_init();
        s_abort = 0;
    }
    if (warp == 0) tmem_alloc(&s_tmem, 512);
    tc_sync();
    const uint32_t tm = s_tmem;
    if (tid == ISSUER) {
        issue_xb(0);
        issue_s(0);
    }
    bool ok = true;
    int xb_issued = 1, s_issued = 1, xb_landed = 0, s_landed = 0;
    // barriers of the main group (the scalar warps run their own loop)
    auto main_sync = [&]() {
        tc_fence_before();
        bar_sync_n(1, kMomMain);
        tc_fence_after();
    };
    auto main_wait = [&](uint64_t *bar, uint32_t parity, bool okv) {
        const bool r = okv ? mbar_wait(bar, parity) : false;
        return bar_and(1, kMomMain, r);
    };
    if (tid >= kMomMain) {
        // ---- scalar warps: the tables of chunk k into slot k & 1 (t = token)
        const int t = tid - kMomMain, sw = (tid - kMomMain) >> 5;
        float r_c = 0.f, r_dt = 0.f;
        auto fetch = [&](int k) {
            const int c = c_begin + k, vr = min(Q, V - Q * c);
            r_c = p.cumA[ix_chunk(p, bi, h, c) * Q + t];
            r_dt = t < vr ? p.dt[ix_dt(p, bi, h, Q * c + t)] : 0.f;
        };
        fetch(0);
        bool sok = true;
        for (int k = 0; k < nk; ++k) {
            const int c = c_begin + k, vr = min(Q, V - Q * c), sl = k & 1;
            const float cur_c = r_c, cur_dt = r_dt;
            if (k + 1 < nk) fetch(k + 1);
            // the main group has finished with the tables of chunk k - 2
            if (k >= 2) sok = sok && mbar_wait(&bar_tabfree[sl], (uint32_t)(((k - 2) >> 1) & 1));
            // X of chunk k (its rows past valid_len are not read)
            sok = sok && mbar_wait(&bar_xb[k & 1], (uint32_t)((k >> 1) & 1));
            sok = bar_and(2, 128, sok);
            if (!sok) break;
            t_c[sl][t] = cur_c;
            t_dt[sl][t] = cur_dt;
            float rs = 0.f;
            if (t < vr) {
                const uint32_t rowb = smem_u32(Xs + (k & 1) * XT) + (uint32_t)t * 128u;
                float r4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    const uint4 u = ld_shared_v4(rowb + (uint32_t)c8 * 16u);
                    r4[c8 & 3] += (bf_lo(u.x) + bf_hi(u.x)) + (bf_lo(u.y) + bf_hi(u.y)) + (bf_lo(u.z) + bf_hi(u.z)) +
                                  (bf_lo(u.w) + bf_hi(u.w));
                }
                rs = (r4[0] + r4[1]) + (r4[2] + r4[3]);
            }
            t_rs[t] = rs;
            bar_sync_n(2, 128);
            if (sw == 0) {
                const int lane_ = t;
                // suffix recurrences over the valid tokens; lane l owns tokens 4 l .. 4 l + 3
                float sA = 1.f, sB = 0.f, uA = 1.f, uB = 0.f;  // lane map (identity)
                float e2[4], e1[4];
#pragma unroll
                for (int i = 3; i >= 0; --i) {
                    const int t = 4 * lane_ + i;
                    float a2 = 0.f, a1 = 0.f, b = 0.f;  // token map x -> b + a x
                    if (t < vr - 1) {
                        const float d = t_c[sl][t + 1] - t_c[sl][t];
                        a2 = __expf(2.f * d);
                        a1 = __expf(d);
                        b = 1.f;
                    } else if (t == vr - 1) {
                        b = 1.f;
                    }
                    e2[i] = a2;
                    e1[i] = a1;
                    // lane map = token map after the maps of the lane's later tokens
                    float tA = a2, tB = b;
                    affine_compose(tA, tB, sA, sB);
                    sA = tA;
                    sB = tB;
                    float vA = a1, vB = b;
                    affine_compose(vA, vB, uA, uB);
                    uA = vA;
                    uB = vB;
                }
                // inclusive suffix scan of the lane maps: lane l gets map_l after ... after map_31
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float oA = __shfl_down_sync(0xffffffffu, sA, o), oB = __shfl_down_sync(0xffffffffu, sB, o);
                    const float pA = __shfl_down_sync(0xffffffffu, uA, o), pB = __shfl_down_sync(0xffffffffu, uB, o);
                    if (lane_ + o < 32) {
                        affine_compose(sA, sB, oA, oB);
                        affine_compose(uA, uB, pA, pB);
                    }
                }
                // value entering the lane's last token: the next lane's suffix applied to 0
                float sig = __shfl_down_sync(0xffffffffu, sB, 1), tau = __shfl_down_sync(0xffffffffu, uB, 1);
                if (lane_ == 31) sig = tau = 0.f;
                float c0 = 0.f, asum = 0.f;
#pragma unroll
                for (int i = 3; i >= 0; --i) {
                    const int t = 4 * lane_ + i;
                    const bool valid = t < vr;
                    sig = valid ? fmaf(e2[i], sig, 1.f) : 0.f;
                    tau = valid ? fmaf(e1[i], tau, 1.f) : 0.f;
                    const float ec = valid ? __expf(t_c[sl][t]) : 0.f, dt = t_dt[sl][t];
                    t_ds[sl][t] = dt * sig;
                    t_al2[sl][t] = 2.f * dt * ec * sig;
                    t_w1[sl][t] = dt * tau * t_rs[t];
                    c0 += ec * ec;
                    asum += ec;
                }
                c0 = warp_sum(c0);
                asum = warp_sum(asum);
                if (lane_ == 0) {
                    s_c0[sl] = c0;
                    s_asum[sl] = asum;
                }
            }
            bar_sync_n(2, 128);
            if (t == 0) mbar_arrive(&bar_tab[sl]);
        }
        if (!sok) s_abort = 1;
    } else {
    for (int k = 0; k < nk && ok; ++k) {
        const int c = c_begin + k, vr = min(Q, V - Q * c), buf = k & 1;
        uint8_t *Xb = Xs + buf * XT, *Bb = Bs + buf * BT;
        // MMA3 of chunk k - 1 done: Y, sqrt(c0) s, F, 2 alpha X and the X, B of buffer (k - 1) & 1 are free
        const int sl = k & 1;
        if (k > 0) ok = main_wait(&bar_a, (uint32_t)((k - 1) & 1), ok);
        tc_fence_after();
        if (tid == ISSUER && ok && k + 1 < nk) {
            issue_xb(k + 1);
            xb_issued = k + 2;
        }
        ok = main_wait(&bar_xb[buf], (uint32_t)((k >> 1) & 1), ok);
        if (ok) xb_landed = k + 1;
        ok = main_wait(&bar_s, (uint32_t)(k & 1), ok);
        if (ok) s_landed = k + 1;
        if (!ok) break;
        if (vr < Q) {  // rows past valid_len may hold anything: zero them (a select)
            zero_rows_from_n(Xb, Q, vr, kMomMain);
            zero_rows_from_n(Bb, Q, vr, kMomMain);
            zero_rows_from_n(Bb + XT, Q, vr, kMomMain);
        }
        fence_async_smem();
        main_sync();
        if (tid == ISSUER) {  // MMA1: G = X X^T (both operands the K-major X tile)
            const uint32_t id = idesc_bf16(128, 128, false, false);
            for (int ks = 0; ks < kP / 16; ++ks)
                mma_bf16(tm, sdesc_kmajor(smem_u32(Xb), ks, XT), sdesc_kmajor(smem_u32(Xb), ks, XT), id, ks > 0);
            mma_commit(&bar_g);
        }
        // ---- the chunk's tables (the scalar warps)
        ok = main_wait(&bar_tab[sl], (uint32_t)((k >> 1) & 1), ok);
        if (!ok) break;
        // ---- A operand (2 alpha o X) and sqrt(c0) s
        {
            const uint32_t xb = smem_u32(Xb), xa = smem_u32(XAs);
            for (int i = tid; i < Q * 8; i += kMomMain) {
                const int row = i >> 3;
                const uint32_t off = (uint32_t)i * 16u;
                if (row >= vr) {
                    st_shared_v4(xa + off, 0u, 0u, 0u, 0u);
                    continue;
                }
                const uint32_t f2 = pack_bf2(t_al2[sl][row], t_al2[sl][row]);
                const uint4 v = ld_shared_v4(xb + off);
                st_shared_v4(xa + off, bmul2(v.x, f2), bmul2(v.y, f2), bmul2(v.z, f2), bmul2(v.w, f2));
            }
            const float sq = sqrtf(s_c0[sl]);
            const uint32_t f2 = pack_bf2(sq, sq), ss = smem_u32(Ss), sc = smem_u32(Ssc);
            for (int i = tid; i < 2 * ST / 16; i += kMomMain) {
                const uint4 v = ld_shared_v4(ss + (uint32_t)i * 16u);
                st_shared_v4(sc + (uint32_t)i * 16u, bmul2(v.x, f2), bmul2(v.y, f2), bmul2(v.z, f2), bmul2(v.w, f2));
            }
        }
        // ---- F = K o G into the K-major A tile: row u, columns 32 cq .. 32 cq + 31
        ok = main_wait(&bar_g, (uint32_t)(k & 1), ok);
        tc_fence_after();
        if (ok) {
            const int u = 32 * q4 + lane;
            float gv[32];
            tmem_ld32(tmem_addr(tm, 32 * q4, 32 * cq), gv);
            const float cu = t_c[sl][u], dtu = t_dt[sl][u], dsu = t_ds[sl][u];
            const bool vu = u < vr;
            const uint32_t rowf = smem_u32(Fs) + (uint32_t)(cq >> 1) * XT + (uint32_t)u * 128u;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                float f[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int v = 32 * cq + 8 * c4 + j;
                    // exp(2 c_m - c_u - c_v) = exp(-|c_u - c_v|); the sigma_m dt factor sits on the later token
                    const float e = __expf(-fabsf(cu - t_c[sl][v]));
                    const float fac = v <= u ? dsu * t_dt[sl][v] : dtu * t_ds[sl][v];
                    f[j] = (vu && v < vr) ? gv[8 * c4 + j] * e * fac : 0.f;
                }
                const int c8 = 4 * (cq & 1) + c4;
                st_shared_v4(rowf + (uint32_t)(((c8 ^ (u & 7)) & 7) << 4), pack_bf2(f[0], f[1]), pack_bf2(f[2], f[3]),
                             pack_bf2(f[4], f[5]), pack_bf2(f[6], f[7]));
            }
        }
        fence_async_smem();
        tc_fence_before();
        ok = bar_and(1, kMomMain, ok);
        tc_fence_after();
        if (!ok) break;
        if (tid == ISSUER) {  // MMA2: Y = F B + (2 alpha o X) s
            const uint32_t id = idesc_bf16(128, 128, false, true);
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16(tm + 128, sdesc_kmajor(smem_u32(Fs), ks, XT), sdesc_mnmajor(smem_u32(Bb), ks, XT), id, ks > 0);
            for (int ks = 0; ks < kP / 16; ++ks)
                mma_bf16(tm + 128, sdesc_kmajor(smem_u32(XAs), ks, XT), sdesc_mnmajor(smem_u32(Ss), ks, ST), id, true);
            mma_commit(&bar_y);
        }
        // ---- Y into the MN-major B tile of MMA3 (row u, columns 32 cq ..), and the two
        // extra columns: w1 beside Y (in the 2 alpha X tile), sum exp(c) / sqrt(c0) beside sqrt(c0) s
        ok = main_wait(&bar_y, (uint32_t)(k & 1), ok);
        tc_fence_after();
        if (ok) {
            const int u = 32 * q4 + lane;
            float yv[32];
            tmem_ld32(tmem_addr(tm, 32 * q4, 128 + 32 * cq), yv);
            const uint32_t rowy = smem_u32(Ys) + (uint32_t)(cq >> 1) * XT + (uint32_t)u * 128u;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const int c8 = 4 * (cq & 1) + c4;
                st_shared_v4(rowy + (uint32_t)(((c8 ^ (u & 7)) & 7) << 4), pack_bf2(yv[8 * c4], yv[8 * c4 + 1]),
                             pack_bf2(yv[8 * c4 + 2], yv[8 * c4 + 3]), pack_bf2(yv[8 * c4 + 4], yv[8 * c4 + 5]),
                             pack_bf2(yv[8 * c4 + 6], yv[8 * c4 + 7]));
            }
            if (tid < Q) {  // row u of the third Y block: (w1[u], 0, ..., 0) over columns 0 .. 15
                const uint32_t row = smem_u32(XAs) + (uint32_t)tid * 128u;
                st_shared_v4(row + (uint32_t)(((0 ^ (tid & 7)) & 7) << 4), pack_bf2(t_w1[sl][tid], 0.f), 0u, 0u, 0u);
                st_shared_v4(row + (uint32_t)(((1 ^ (tid & 7)) & 7) << 4), 0u, 0u, 0u, 0u);
            } else if (tid < Q + kP) {  // row p of the third sqrt(c0) s block: sum exp(c) / sqrt(c0)
                const int pp = tid - Q;
                const uint32_t row = smem_u32(Fs) + (uint32_t)pp * 128u;
                st_shared_v4(row + (uint32_t)(((0 ^ (pp & 7)) & 7) << 4), pack_bf2(s_asum[sl] / sqrtf(s_c0[sl]), 0.f),
                             0u, 0u, 0u);
                st_shared_v4(row + (uint32_t)(((1 ^ (pp & 7)) & 7) << 4), 0u, 0u, 0u, 0u);
            }
        }
        fence_async_smem();
        tc_fence_before();
        ok = bar_and(1, kMomMain, ok);
        tc_fence_after();
        if (!ok) break;
        if (tid == 0) mbar_arrive(&bar_tabfree[sl]);  // the tables of chunk k are no longer read
        if (tid == ISSUER) {
            // s of the next chunk (MMA2 has read this one; sqrt(c0) s is a copy)
            if (k + 1 < nk) {
                issue_s(k + 1);
                s_issued = k + 2;
            }
            // MMA3: [A | m1] += B^T [Y | w1] + (sqrt(c0) s)^T [sqrt(c0) s | sum exp(c) / sqrt(c0)]
            const uint32_t id = idesc_bf16(128, 144, true, true);
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16(tm + 256, sdesc_mnmajor(smem_u32(Bb), ks, XT), sdesc_mnmajor(smem_u32(Ys), ks, XT), id,
                         k > 0 || ks > 0);
            for (int ks = 0; ks < kP / 16; ++ks)
                mma_bf16(tm + 256, sdesc_mnmajor(smem_u32(Ssc), ks, ST), sdesc_mnmajor(smem_u32(Ssc), ks, ST), id, true);
            mma_commit(&bar_a);
        }
    }
    if (ok) ok = main_wait(&bar_a, (uint32_t)((nk - 1) & 1), ok);
    tc_fence_after();
    if (ok && s_abort) ok = false;
    if (ok) {
        // the range's A, transposed (coalesced: lanes hold consecutive r), and m1 (column 128)
        const int r = 32 * q4 + lane;
        float av[32];
        tmem_ld32(tmem_addr(tm, 32 * q4, 256 + 32 * cq), av);
#pragma unroll
        for (int j = 0; j < 32; ++j) Apart[(size_t)(32 * cq + j) * kN + r] = av[j];
        if (cq == 0) {
            float mv[16];
            tmem_ld16(tmem_addr(tm, 32 * q4, 256 + 128), mv);
            m1part[r] = mv[0];
        }
    } else if (tid == 0) {
        flag_timeout(p);
    }
    }  // main group
    // loads issued for chunks that were never waited for have to land before exit
    if (tid == ISSUER) {
        if (xb_issued > xb_landed)
            for (int k = xb_landed; k < xb_issued; ++k) mbar_wait(&bar_xb[k & 1], (uint32_t)((k >> 1) & 1));
        if (s_issued > s_landed) mbar_wait(&bar_s, (uint32_t)((s_issued - 1) & 1));
    }
    tc_sync();
    if (warp == 0) tmem_dealloc(tm, 512);
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
                   const cuuint32_t *box, CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, dtype, (cuuint32_t)rank, const_cast<void *>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// [b, L, H or G, 64 or 128] bf16 activations: boxes of 64 columns x `tokens` tokens.
cudaError_t map_tokens(CUtensorMap *m, const void *base, int b, int L, int heads, int width, int tokens = 128) {
    cuuint64_t dims[4] = {(cuuint64_t)width, (cuuint64_t)heads, (cuuint64_t)L, (cuuint64_t)b};
    cuuint64_t strides[3] = {(cuuint64_t)width * 2, (cuuint64_t)heads * width * 2, (cuuint64_t)L * heads * width * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)tokens, 1};
    return encode(m, base, 4, dims, strides, box);
}

// [b*n*H, P, N] bf16 chunk states: boxes of 64 dstate columns x 64 headdim rows.
cudaError_t map_states(CUtensorMap *m, const void *base, long long count) {
    cuuint64_t dims[3] = {(cuuint64_t)kN, (cuuint64_t)kP, (cuuint64_t)count};
    cuuint64_t strides[2] = {(cuuint64_t)kN * 2, (cuuint64_t)kP * kN * 2};
    cuuint32_t box[3] = {64, 64, 1};
    return encode(m, base, 3, dims, strides, box);
}

// Heads per CTA of the chunk-state scan (one CTA per SM): one while the (b, head)
// chains fit the 152 SMs in one wave, else two (sharing B), which halves the waves.
int scan_heads_per_cta(const Params &p) { return (long long)p.b * p.H > 152 ? 2 : 1; }

cudaError_t make_maps(const Params &p, TcMaps *mp, bool backward) {
    memset(mp, 0, sizeof(*mp));
    cudaError_t e;
    if ((e = map_tokens(&mp->x, p.x, p.b, p.L, p.H, kP)) != cudaSuccess) return e;
    if ((e = map_tokens(&mp->B, p.B, p.b, p.L, p.G, kN)) != cudaSuccess) return e;
    if ((e = map_tokens(&mp->C, p.C, p.b, p.L, p.G, kN)) != cudaSuccess) return e;
    {  // x as [b][head][token][64] boxes of (1 or 2 heads) x 128 or 64 tokens: dims (p, token, head, b)
        const int hpc = scan_heads_per_cta(p);
        cuuint64_t dims[4] = {(cuuint64_t)kP, (cuuint64_t)p.L, (cuuint64_t)p.H, (cuuint64_t)p.b};
        cuuint64_t strides[3] = {(cuuint64_t)p.H * kP * 2, (cuuint64_t)kP * 2, (cuuint64_t)p.L * p.H * kP * 2};
        cuuint32_t box[4] = {64, (cuuint32_t)scan_tok(hpc), (cuuint32_t)hpc, 1};
        if ((e = encode(&mp->xs, p.x, 4, dims, strides, box)) != cudaSuccess) return e;
    }
    {  // B as [half][token][64] boxes of 2 halves x the scan's sub-stage: dims (column, token, half, group, b)
        cuuint64_t dims[5] = {64, (cuuint64_t)p.L, 2, (cuuint64_t)p.G, (cuuint64_t)p.b};
        cuuint64_t strides[4] = {(cuuint64_t)p.G * kN * 2, 128, (cuuint64_t)kN * 2, (cuuint64_t)p.L * p.G * kN * 2};
        cuuint32_t box[5] = {64, (cuuint32_t)scan_tok(scan_heads_per_cta(p)), 2, 1, 1};
        if ((e = encode(&mp->Bs, p.B, 5, dims, strides, box)) != cudaSuccess) return e;
    }
    if (p.states_bf && (e = map_states(&mp->st, p.states_bf, (long long)p.b * p.n * p.H)) != cudaSuccess) return e;
    if (!backward && p.y && (e = map_tokens(&mp->y, p.y, p.b, p.L, p.H, kP)) != cudaSuccess) return e;
    if (p.CBh) {  // CB and CB^T, bf16 [b*n*G*Q rows][Q]: boxes of 64 columns x 128 rows
        cuuint64_t dims[2] = {(cuuint64_t)p.Q, (cuuint64_t)p.b * p.n * p.G * p.Q};
        cuuint64_t strides[1] = {(cuuint64_t)p.Q * 2};
        cuuint32_t box[2] = {64, 128};
        if ((e = encode(&mp->cb, p.CBh, 2, dims, strides, box)) != cudaSuccess) return e;
        if ((e = encode(&mp->cbt, p.CBt, 2, dims, strides, box)) != cudaSuccess) return e;
        cuuint32_t box64[2] = {64, 64};  // the lower halves of the tiles whose upper halves are zero
        if ((e = encode(&mp->cb64, p.CBh, 2, dims, strides, box64)) != cudaSuccess) return e;
    }
    if (backward) {
        if (p.d_cb_bf) {  // summed d_cb, bf16 [b*n*G*Q rows][Q]: boxes of 64 columns x 128 rows
            cuuint64_t dims[2] = {(cuuint64_t)p.Q, (cuuint64_t)p.b * p.n * p.G * p.Q};
            cuuint64_t strides[1] = {(cuuint64_t)p.Q * 2};
            cuuint32_t box[2] = {64, 128};
            if ((e = encode(&mp->dcb, p.d_cb_bf, 2, dims, strides, box)) != cudaSuccess) return e;
        }
        if ((e = map_tokens(&mp->dy, p.dy, p.b, p.L, p.H, kP)) != cudaSuccess) return e;
        if (p.dx && (e = map_tokens(&mp->dx, p.dx, p.b, p.L, p.H, kP)) != cudaSuccess) return e;
        if (p.dBC_part) {  // G2 fp32 partials [nslice * 2 * b*n*G*Q rows][N]: boxes of 32 columns x 128 rows
            cuuint64_t dims[2] = {(cuuint64_t)kN, (cuuint64_t)p.nslice * 2 * p.b * p.n * p.G * p.Q};
            cuuint64_t strides[1] = {(cuuint64_t)kN * 4};
            cuuint32_t box[2] = {32, 128};
            if ((e = encode(&mp->part, p.dBC_part, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32)) !=
                cudaSuccess)
                return e;
        }
        if (p.dstates_bf && (e = map_states(&mp->dst, p.dstates_bf, (long long)p.b * p.n * p.H)) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

template <typename K>
cudaError_t launch(K kernel, unsigned grid, size_t smem, cudaStream_t s, const Params &p, const TcMaps &maps,
                   int threads = kThreads) {
    // every kernel here sizes its CTAs against the whole 228 KB: ask for that carveout
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    kernel<<<grid, threads, smem, s>>>(p, maps);
    return cudaGetLastError();
}

// Q = 128 holds 256 TMEM columns per CTA: padded so that at most two CTAs share an SM.
constexpr size_t smem_k2(int Q) { return Q == 128 ? 80 * 1024 : 1024 + 4 * (size_t)Q * 128; }
// B | x stages | two bf16 state tiles
constexpr size_t smem_k3(int Q) { return 1024 + 2 * (size_t)Q * 128 + 4 * (size_t)Q * 128 + 2 * (size_t)kP * kN * 2; }
// X x 2 | B x 2 | s | sqrt(c0) s | F | Y | 2 alpha X (one CTA per SM: 512 TMEM columns)
constexpr size_t smem_moments() { return 1024 + (size_t)(2 + 4 + 1 + 2 + 1 + 2) * 128 * 128 + 2 * 64 * 128; }
// C | CB tiles (full ones and lower halves) | x | s_in | y staging tile | scalar tables
constexpr size_t smem_k5(int Q) {
    return 1024 + 3 * (size_t)Q * 128 + 2 * 64 * 128 +
           (size_t)kTile * ((Q / 128) * (Q / 128 + 1) - Q / 128) + (size_t)(kTile / 2) * (Q / 128) + kTile +
           4 * 3 * (2 * Q + Q / 2 + (Q / 64) * 128 + 8 + Q / 2 + Q / 16);
}
constexpr size_t smem_blue(int Q) { return 1024 + 2 * (size_t)Q * 128 + 3 * ((size_t)Q * 128 + 2 * 64 * 128); }
constexpr size_t smem_k3bwd(int Q) {
    return 1024 + 2 * (size_t)Q * 128 + 2 * ((size_t)Q * 128 + 2 * 64 * 128) + (size_t)Q * 128 + 4 * (3 * 3 * Q + 2 * Q);
}
// Padded above half of the SM's shared memory: a CTA holding 512 TMEM columns
// must never share its SM with another CTA of the same kernel.
// W^T tiles | x half tiles (Q = 256: two lower, one upper; Q = 128: two) | dy x 2 | scalar tables
constexpr size_t smem_orange_raw(int Q) {
    return 1024 + (size_t)kTile * (Q == 256 ? 6 : 2) + (size_t)kTile * (Q == 256 ? 3 : 2) + 2 * (size_t)Q * 128 +
           4 * 3 * (2 * Q + 732 + Q / 2 + Q / 16);
}
constexpr size_t smem_orange(int Q) { return smem_orange_raw(Q) > 120 * 1024 ? smem_orange_raw(Q) : 120 * 1024; }
// Padded above a third of the SM's shared memory: two CTAs of 256 TMEM columns
// each may share an SM, a third must not.
constexpr size_t dcb_fst(int Q) { return (((4 * Q + Q / 64 + Q / 16 + 3) & ~3) + Q + Q / 16 + 3) & ~3; }
constexpr size_t smem_dcb(int Q) {
    return 1024 + 6 * (size_t)kTile + 4 * 3 * dcb_fst(Q) > 80 * 1024 ? 1024 + 6 * (size_t)kTile + 4 * 3 * dcb_fst(Q)
                                                                   : 80 * 1024;
}
constexpr size_t smem_dbc(int Q) {
    return 1024 + 2 * (2 * (size_t)Q * 128 + 4 * 64 * 128) + 4 * 4 * Q;
}
static_assert(smem_orange(256) <= 232448 && smem_orange(128) > 116 * 1024, "ORANGE backward: one CTA per SM");
static_assert(smem_k3bwd(256) <= 232448 && smem_k3bwd(256) > 116 * 1024, "K3 backward: one CTA per SM");
static_assert(smem_k2(256) > 116 * 1024, "K2 (512 TMEM columns): one CTA per SM");
static_assert(smem_k2(128) >= 1024 + 4 * 128 * 128 && 3 * (smem_k2(128) + 1024) > 233472,
              "K2 at Q = 128 (256 TMEM columns): at most two CTAs per SM");
static_assert(smem_k5(256) <= 232448 && smem_k5(256) > 116 * 1024, "K5: one CTA per SM");
static_assert(smem_moments() + 6 * 128 * 4 + 64 <= 232448 && smem_moments() > 116 * 1024, "moments: one CTA per SM");
static_assert(ScanGeom<2>::smem + 4 * (4 * 2 * 256 + 2 * 4) + 512 <= 232448 &&
                  ScanGeom<1>::smem + 4 * (4 * 1 * 256 + 4) + 512 <= 232448,
              "chunk-state scan shared memory");
static_assert(smem_k3(256) <= 232448 && smem_blue(256) <= 232448, "K3 / BLUE shared memory");
static_assert(smem_blue(128) > 116 * 1024, "BLUE (512 TMEM columns): one CTA per SM");
static_assert(smem_dbc(256) <= 232448, "group backward shared memory");
static_assert(3 * (smem_dcb(128) + 1024) > 233472 && 2 * (smem_dcb(256) + 1024) <= 233472,
              "G1: two CTAs per SM, never three");
static_assert(2 * (size_t)256 * 256 + 2 * 256 * 128 <= 2 * (2 * (size_t)256 * 128 + 4 * 64 * 128),
              "d_cb + B tile must fit the two long-K stages");


// The bounded wait of the kernels above, on a barrier that one arrival
// completes (arrive = 1) or that nothing completes (arrive = 0), with the
// caller's limit; a timeout is recorded in the status word as they record it.
// One thread, no copies or tensor-memory in flight: giving up is always safe.
__global__ void wait_selftest_kernel(Params p, uint64_t limit_ns, int arrive) {
    __shared__ __align__(8) uint64_t bar;
    mbar_init(&bar, 1);
    mbar_fence_init();
    if (arrive) mbar_arrive(&bar);
    if (!mbar_wait(&bar, 0, limit_ns)) flag_timeout(p);
}

}  // namespace

bool tc_supported(int64_t P, int64_t N, int64_t Q) { return P == kP && N == kN && (Q == 128 || Q == 256); }
int tc_dD_per(int64_t) { return kThreadsWide / 32; }  // one dD partial per ORANGE consumer warp
int tc_dcb_slices(const ssd_dims &d) {
    // CTAs: one per 128 x 128 block on or below the diagonal and head slice;
    // two fit an SM.  Head slices only when the blocks alone leave SMs idle
    // (each slice adds a partial d_cb to write and read back): then minimise
    // (waves x heads per CTA) over up to two waves, fewest slices on ties.
    const long long hpg = d.nheads / d.ngroups;
    const long long n = (d.seqlen + d.chunk_len - 1) / d.chunk_len;
    const long long nt = d.chunk_len / 128;
    const long long ctas = d.batch * n * d.ngroups * (nt * (nt + 1) / 2);
    const long long slots = 2 * 152;
    if (ctas >= slots) return 1;
    long long best = 1, best_cost = -1;
    for (long long s = 1; s <= hpg && ctas * s <= 2 * slots + ctas; ++s) {
        const long long cost = ((ctas * s + slots - 1) / slots) * ((hpg + s - 1) / s);
        if (best_cost < 0 || cost < best_cost) {
            best = s;
            best_cost = cost;
        }
    }
    return (int)best;
}
int tc_k5_slices(const ssd_dims &d) {
    // one CTA per SM: heads per CTA chosen to minimise waves x (heads per CTA + 1),
    // the +1 standing for the CTA's fixed cost (resident operands, TMEM, tables)
    const long long hpg = d.nheads / d.ngroups;
    const long long n = (d.seqlen + d.chunk_len - 1) / d.chunk_len;
    const long long groups = d.batch * n * d.ngroups;
    long long best = 1, best_cost = -1;
    for (long long per = hpg; per >= 1; --per) {
        const long long ns = (hpg + per - 1) / per;
        const long long cost = ((groups * ns + 151) / 152) * (per + 1);
        if (best_cost < 0 || cost < best_cost) {
            best = ns;
            best_cost = cost;
        }
    }
    return (int)best;
}
int tc_k3_slices(const ssd_dims &d) {
    // one CTA per SM: minimise waves x (heads per CTA + the resident operand's
    // load, about two heads' worth), fewest slices on ties
    const long long hpg = d.nheads / d.ngroups;
    const long long n = (d.seqlen + d.chunk_len - 1) / d.chunk_len;
    const long long groups = d.batch * n * d.ngroups;
    long long best = 1, best_cost = -1;
    for (long long s = 1; s <= hpg; ++s) {
        const long long cost = ((groups * s + 151) / 152) * ((hpg + s - 1) / s + 2);
        if (best_cost < 0 || cost < best_cost) {
            best = s;
            best_cost = cost;
        }
    }
    return (int)best;
}
int tc_group_slices(const ssd_dims &d) {
    // one CTA per SM; heads per CTA chosen to minimise waves x (heads per CTA + 1),
    // the +1 standing for the CTA's fixed cost (prologue, partial write-out)
    const long long hpg = d.nheads / d.ngroups;
    const long long n = (d.seqlen + d.chunk_len - 1) / d.chunk_len;
    const long long groups = d.batch * n * d.ngroups;
    long long best = 1, best_cost = -1;
    for (long long per = hpg; per >= 1; --per) {
        const long long ns = (hpg + per - 1) / per;
        const long long cost = ((groups * ns + 151) / 152) * (per + 1);
        if (best_cost < 0 || cost < best_cost) {
            best = ns;
            best_cost = cost;
        }
    }
    return (int)best;
}

#define SSD_TC_DISPATCH(Q_, call) ((Q_) == 256 ? call(256) : call(128))

cudaError_t launch_tc_k2(const Params &p, cudaStream_t s) {
    TcMaps m;
    cudaError_t e = make_maps(p, &m, false);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(p.b * p.n * p.G * (p.Q / 128));
#define CALL(Q) launch(tc_k2_kernel<Q>, grid, smem_k2(Q), s, p, m, kThreadsWide)
    return SSD_TC_DISPATCH(p.Q, CALL);
#undef CALL
}

cudaError_t launch_tc_k3(const Params &p, cudaStream_t s) {
    TcMaps m;
    cudaError_t e = make_maps(p, &m, false);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(p.b * p.n * p.G * p.nslice_k3);
#define CALL(Q) launch(tc_k3_kernel<Q>, grid, smem_k3(Q), s, p, m, kThreadsWide + 32)
    return SSD_TC_DISPATCH(p.Q, CALL);
#undef CALL
}


template <int Q, int HPC>
cudaError_t launch_scan(const Params &p, const TcMaps &m, bool write_final, cudaStream_t s) {
    auto kernel = tc_state_scan_kernel<Q, HPC>;
    const size_t smem = ScanGeom<HPC>::smem;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(p.b * p.G * ((p.hpg + HPC - 1) / HPC));
    kernel<<<grid, kScanConsumers + 32 * (2 + HPC), smem, s>>>(p, m, write_final ? 1 : 0);
    return cudaGetLastError();
}

long long tc_state_scan_ctas(const Params &p) {
    const int hpc = scan_heads_per_cta(p);
    return (long long)p.b * p.G * ((p.hpg + hpc - 1) / hpc);
}

cudaError_t launch_tc_state_scan(const Params &p, bool write_final, cudaStream_t s) {
    TcMaps m;
    cudaError_t e = make_maps(p, &m, false);
    if (e != cudaSuccess) return e;
    const int hpc = scan_heads_per_cta(p);
    if (p.Q == 256) return hpc == 2 ? launch_scan<256, 2>(p, m, write_final, s) : launch_scan<256, 1>(p, m, write_final, s);
    return hpc == 2 ? launch_scan<128, 2>(p, m, write_final, s) : launch_scan<128, 1>(p, m, write_final, s);
}

cudaError_t launch_tc_moments(const Params &p, cudaStream_t s) {
    TcMaps m;
    cudaError_t e = make_maps(p, &m, false);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(p.b * p.H * p.mom_ranges);
    return launch(tc_moments_kernel, grid, smem_moments(), s, p, m, kMomThreads);
}

cudaError_t launch_tc_k5(const Params &p, cudaStream_t s) {
    TcMaps m;
    cudaError_t e = make_maps(p, &m, false);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(p.b * p.n * p.G * p.nslice_k5);
#define CALL(Q) launch(tc_k5_kernel<Q>, grid, smem_k5(Q), s, p, m, kThreadsWide)
    return SSD_TC_DISPATCH(p.Q, CALL);
#undef CALL
}

cudaError_t launch_tc_bwd_blue(const Params &p, cudaStream_t s) {
    TcMaps m;
    cudaError_t e = make_maps(p, &m, true);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(p.b * p.n * p.G * p.nslice_k3);
#define CALL(Q) launch(tc_bwd_blue_kernel<Q>, grid, smem_blue(Q), s, p, m, kThreadsWide + 32)
    return SSD_TC_DISPATCH(p.Q, CALL);
#undef CALL
}

cudaError_t launch_tc_bwd_k3(const Params &p, cudaStream_t s) {
    TcMaps m;
    cudaError_t e = make_maps(p, &m, true);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(p.b * p.n * p.G * p.nslice_k5);
#define CALL(Q) launch(tc_bwd_k3_kernel<Q>, grid, smem_k3bwd(Q), s, p, m, kThreadsWide)
    return SSD_TC_DISPATCH(p.Q, CALL);
#undef CALL
}

cudaError_t launch_tc_bwd_orange(const Params &p, cudaStream_t s) {
    TcMaps m;
    cudaError_t e = make_maps(p, &m, true);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(p.b * p.n * p.G * p.nslice_k5);
#define CALL(Q) launch(tc_bwd_orange_kernel<Q>, grid, smem_orange(Q), s, p, m, kThreadsWide)
    return SSD_TC_DISPATCH(p.Q, CALL);
#undef CALL
}

cudaError_t launch_tc_bwd_dcb(const Params &p, cudaStream_t s) {
    TcMaps m;
    cudaError_t e = make_maps(p, &m, true);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(p.b * p.n * p.G * p.nslice_cb * (p.Q == 256 ? 3 : 1));
#define CALL(Q) launch(tc_bwd_dcb_kernel<Q>, grid, smem_dcb(Q), s, p, m, kThreadsWide)
    return SSD_TC_DISPATCH(p.Q, CALL);
#undef CALL
}

cudaError_t launch_tc_bwd_dbc(const Params &p, cudaStream_t s) {
    TcMaps m;
    cudaError_t e = make_maps(p, &m, true);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(p.b * p.n * p.G * p.nslice);
#define CALL(Q) launch(tc_bwd_dbc_kernel<Q>, grid, smem_dbc(Q), s, p, m, kThreadsWide + 32)
    return SSD_TC_DISPATCH(p.Q, CALL);
#undef CALL
}

cudaError_t launch_tc_bwd_dbc_reduce(const Params &p, cudaStream_t s) {
    const size_t nvec = (size_t)p.b * p.L * p.G * (kN / 4);
    const unsigned grid = (unsigned)((nvec + 255) / 256);
    if (p.Q == 256) tc_bwd_dbc_reduce<256><<<grid, 256, 0, s>>>(p);
    else tc_bwd_dbc_reduce<128><<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(int *status, uint64_t limit_ns, int arrive, cudaStream_t s) {
    Params p;
    memset(&p, 0, sizeof(p));
    p.status = status;
    wait_selftest_kernel<<<1, 1, 0, s>>>(p, limit_ns, arrive);
    return cudaGetLastError();
}

}  // namespace ssd
