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

// The 16 entries of vector index e of a state.  With IL (P * N a multiple of
// 2048) thread t of each 128-thread slice holds 16-byte pieces q at entries
// (q * 128 + t) * EP of the slice (EP = 8 bf16 or 4 fp32 entries a piece), so a
// warp's access to one piece is 512 contiguous bytes, whole sectors; without
// IL the 16 consecutive entries 16 e (two or four 16-byte pieces a thread, each
// warp access touching half of every sector).  fp32 arrays beside a state
// (initial / final state and their gradients) follow the state's mapping.
template <typename S, bool IL>
__device__ __forceinline__ size_t piece_off(size_t e, int q) {
    constexpr int PC = kVec * (int)sizeof(S) / 16, EP = kVec / PC;
    if (IL) return (e / kK4Threads) * (size_t)(kK4Threads * kVec) + (size_t)(q * kK4Threads + e % kK4Threads) * EP;
    return kVec * e + (size_t)q * EP;
}
template <typename S, bool IL>
__device__ __forceinline__ Packed<S> ld_packed(const S *base, size_t e) {
    constexpr int PC = kVec * (int)sizeof(S) / 16;
    Packed<S> x;
    uint4 *w = reinterpret_cast<uint4 *>(&x);
#pragma unroll
    for (int q = 0; q < PC; ++q) w[q] = *reinterpret_cast<const uint4 *>(base + piece_off<S, IL>(e, q));
    return x;
}
template <typename S, bool IL>
__device__ __forceinline__ void st_vals(S *base, size_t e, const float *v) {
    constexpr int PC = kVec * (int)sizeof(S) / 16, EP = kVec / PC;
#pragma unroll
    for (int q = 0; q < PC; ++q) {
        S *dst = base + piece_off<S, IL>(e, q);
        if constexpr (sizeof(S) == 4) {
            *reinterpret_cast<float4 *>(dst) = make_float4(v[q * EP], v[q * EP + 1], v[q * EP + 2], v[q * EP + 3]);
        } else {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                __nv_bfloat162 h2 = __floats2bfloat162_rn(v[q * EP + 2 * i], v[q * EP + 2 * i + 1]);
                w[i] = *reinterpret_cast<uint32_t *>(&h2);
            }
            *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}
template <typename S, bool IL>
__device__ __forceinline__ void ld_f32(const float *base, size_t e, float *v) {
    constexpr int PC = kVec * (int)sizeof(S) / 16, EP = kVec / PC;
#pragma unroll
    for (int q = 0; q < PC; ++q) {
        const float4 *src = reinterpret_cast<const float4 *>(base + piece_off<S, IL>(e, q));
#pragma unroll
        for (int k = 0; k < EP / 4; ++k) {
            const float4 x = src[k];
            v[q * EP + 4 * k] = x.x; v[q * EP + 4 * k + 1] = x.y; v[q * EP + 4 * k + 2] = x.z; v[q * EP + 4 * k + 3] = x.w;
        }
    }
}
template <typename S, bool IL>
__device__ __forceinline__ void st_f32(float *base, size_t e, const float *v) {
    constexpr int PC = kVec * (int)sizeof(S) / 16, EP = kVec / PC;
#pragma unroll
    for (int q = 0; q < PC; ++q) {
        float4 *dst = reinterpret_cast<float4 *>(base + piece_off<S, IL>(e, q));
#pragma unroll
        for (int k = 0; k < EP / 4; ++k)
            dst[k] = make_float4(v[q * EP + 4 * k], v[q * EP + 4 * k + 1], v[q * EP + 4 * k + 2], v[q * EP + 4 * k + 3]);
    }
}

// Chunks read ahead (U): bounded by registers, since the grid must stay one
// wave.  A grid of at most one block per SM (few (b, h) chains: the 131k-token
// workload has 32, 128 blocks) takes a deep read-ahead and the registers it
// needs; larger grids keep five blocks per SM and a short one.  MB: the blocks
// per SM the launch bounds promise.
constexpr int k4_min_blocks(int U, int bytes) { return U * bytes >= 32 ? 1 : (U * bytes >= 16 ? 2 : 5); }

template <typename S, int U, bool IL>
__global__ void __launch_bounds__(kK4Threads, k4_min_blocks(U, sizeof(S)))
    k4_state_passing(Params p, S *st, int write_final) {
    const size_t PN = (size_t)p.P * p.N, nvec = PN / kVec;
    const size_t gid = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    if (gid >= (size_t)p.b * p.H * nvec) return;
    const size_t e = gid % nvec, bh = gid / nvec;
    const int h = (int)(bh % p.H), bi = (int)(bh / p.H);
    float s[kVec];
    if (p.init) ld_f32<S, IL>(p.init + bh * PN, e, s);
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
            in[u] = ld_packed<S, IL>(st + ix_state(p, bi, u, h), e);
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
                    in[u] = ld_packed<S, IL>(st + ix_state(p, bi, c + U, h), e);
                    ea[u] = endA[c + U];
                }
                st_vals<S, IL>(st + ix_state(p, bi, c, h), e, s);
                float v[kVec];
                unpack16(cur, v);
#pragma unroll
                for (int i = 0; i < kVec; ++i) s[i] = fmaf(a, s[i], v[i]);
            }
        }
    }
    if (write_final && p.final_state) st_f32<S, IL>(p.final_state + bh * PN, e, s);
}

// ------------------------------------------------------- K4, time-segmented
// For few, long chains (the 131k-token sequence: 32 chains of 512 chunks).
// The recurrence is linear in the state, so a run of chunks acts on its
// input state as s -> D s + V, with D the product of the chunks' exp(endA)
// and V the state the run ends in from a zero start.  The chunks of a chain
// are cut into K segments of T; a ticket (pair, r) is segment r of one
// 2048-entry slice of one (b, h) state:
//   1. its T chunks are reduced from zero to (D_r, V_r), which are
//      published (ready flag);
//   2. its carry-in is rebuilt from the published values of earlier
//      segments, always in one order: from the carry of the first segment of
//      its group of kK4SegGroup (or, for a group's first segment, of the
//      previous group's first), folding V_j, D_j of the segments in between,
//      so the result does not depend on timing; a group's first segment
//      publishes its carry;
//   3. its chunks are rescanned from the carry, writing every chunk-input
//      state.
// Tickets are drawn from a counter in segment order, so a ticket waits only
// on smaller ones.  Waits are bounded (2 s); on expiry the call's status
// records SSD_ERR_TIMEOUT and the block goes on with what it has.
// Measured on the 131k-token sequence (GB300): 137 us against 389 us for the
// chunk-serial kernel.  The backward keeps its chunk-serial kernel, which ran
// faster there than this scheme in reverse chunk order (207 against 271 us).
//
// Entries map to threads as in the chunk-serial kernels with whole slices
// (piece_off above): a warp's access to one 16-byte piece is 512 contiguous
// bytes.  With a thread's 32 contiguous bytes copied as two pieces, half of
// every sector went to a second request and the copies landed at about a
// third of the rate.  The segmented path takes states whose P * N is a
// multiple of the 2048-entry slice.
constexpr uint64_t kSegWaitNs = 2000000000ull;
constexpr int kSegSlice = kK4Threads * kVec;  // entries of one slice

__device__ __forceinline__ int ld_acquire(const int *f) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(int *f, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}
__device__ __forceinline__ uint64_t seg_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
// Spins until *f != 0; false after kSegWaitNs.
__device__ bool seg_wait(const int *f) {
    if (ld_acquire(f)) return true;
    const uint64_t t0 = seg_timer_ns();
    for (uint32_t it = 0;; ++it) {
        __nanosleep(64);
        if (ld_acquire(f)) return true;
        if ((it & 63u) == 63u && seg_timer_ns() - t0 > kSegWaitNs) return false;
    }
}

struct SegDev {
    int K, KG, slices;
    long long pairs;
    int *ticket, *aggflag, *carryflag;  // aggflag [pairs, K], carryflag [pairs, KG]
};

// Draws the block's next ticket (segment-major: t = r * pairs + pair) into
// shared slot `sh`; the slots alternate so that a slot is rewritten only after
// a later block barrier.
__device__ __forceinline__ long long seg_draw(const SegDev &g, int *sh) {
    if (threadIdx.x == 0) *sh = atomicAdd(g.ticket, 1);
    __syncthreads();
    return *sh;
}

// ---- this thread's 16 entries of a slice, 16-byte pieces (see above): the
// chunk-serial kernels' helpers with e = threadIdx.x address them from the
// slice's first entry
template <typename S>
__host__ __device__ constexpr int seg_pieces() { return kVec * (int)sizeof(S) / 16; }
// The published 16 fp32 values of a ticket: 2048 floats as [4][128 threads] float4.
__device__ __forceinline__ void seg_st_pub(float *blk, const float *v) {
    float4 *d = reinterpret_cast<float4 *>(blk);
#pragma unroll
    for (int k = 0; k < 4; ++k) d[k * kK4Threads + threadIdx.x] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
}

// Publishes this thread's 16 values at blk (every thread), then the flag (the
// barrier orders every thread's stores before the release store, which warp 1
// issues so that warp 0, which waits on flags next, does not stall on it).
__device__ __forceinline__ void seg_publish(float *blk, const float *v, int *flag) {
    seg_st_pub(blk, v);
    __syncthreads();
    if (threadIdx.x == 32) st_release(flag, 1);
}

// Step 2: the carry into segment r of `pair` (16 entries of this thread), from
// `base` (the chain's initial value at this slice, nullptr for zero) when the
// fold starts at segment 0.  Publishes the carry when r starts a group.
template <typename S>
__device__ void seg_carry(const Params &p, const SegDev &g, long long pair, int r, const float *base, float *c) {
    const int G = kK4SegGroup;
    const int start = (r % G == 0) ? (r >= G ? r - G : 0) : (r / G) * G;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        bool ok = true;
        if (lane < r - start) ok = seg_wait(g.aggflag + pair * g.K + start + lane);
        if (lane == 31 && start > 0) ok = seg_wait(g.carryflag + pair * g.KG + start / G) && ok;
        if (!ok) atomicExch(p.status + kStatusCode, (int)SSD_ERR_TIMEOUT);
    }
    __syncthreads();
    if (start > 0) {
        const float4 *q = reinterpret_cast<const float4 *>(p.k4s_carry + ((size_t)pair * g.KG + start / G) * kSegSlice);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 t = __ldcg(q + k * kK4Threads + threadIdx.x);
            c[4 * k] = t.x; c[4 * k + 1] = t.y; c[4 * k + 2] = t.z; c[4 * k + 3] = t.w;
        }
    } else if (base) {
        ld_f32<S, true>(base, threadIdx.x, c);
    } else {
#pragma unroll
        for (int i = 0; i < kVec; ++i) c[i] = 0.f;
    }
    // the fold's loads are issued together (at most kK4SegGroup segments), half
    // of the 16 entries at a time, then applied in segment order
    const int m = r - start;
    float dd[kK4SegGroup];
#pragma unroll
    for (int jj = 0; jj < kK4SegGroup; ++jj) dd[jj] = jj < m ? __ldcg(p.k4s_dec + (size_t)pair * g.K + start + jj) : 0.f;
    const float4 *q0 = reinterpret_cast<const float4 *>(p.k4s_agg + ((size_t)pair * g.K + start) * kSegSlice);
#pragma unroll
    for (int k2 = 0; k2 < 4; k2 += 2) {
        float4 t[2][kK4SegGroup];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int jj = 0; jj < kK4SegGroup; ++jj)
                if (jj < m) t[h][jj] = __ldcg(q0 + (size_t)jj * (kSegSlice / 4) + (k2 + h) * kK4Threads + threadIdx.x);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int k = k2 + h;
#pragma unroll
            for (int jj = 0; jj < kK4SegGroup; ++jj)
                if (jj < m) {
                    c[4 * k] = fmaf(dd[jj], c[4 * k], t[h][jj].x);
                    c[4 * k + 1] = fmaf(dd[jj], c[4 * k + 1], t[h][jj].y);
                    c[4 * k + 2] = fmaf(dd[jj], c[4 * k + 2], t[h][jj].z);
                    c[4 * k + 3] = fmaf(dd[jj], c[4 * k + 3], t[h][jj].w);
                }
        }
    }
    if (r > 0 && r % G == 0 && r < g.K - 1)
        seg_publish(p.k4s_carry + ((size_t)pair * g.KG + r / G) * kSegSlice, c, g.carryflag + pair * g.KG + r / G);
}

// Step 1's loads go to shared memory by per-thread asynchronous 16-byte copies
// (each thread reads back only what it copied, so no block barrier is needed).
// Layout: [slot][piece][thread], conflict-free.
constexpr int kSegSmem = 64 * 1024;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
                 "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
// Copies this thread's pieces of one chunk's slice into slot `slot`.
template <typename S>
__device__ __forceinline__ void seg_stage(uint4 *sm, int slot, const S *slice) {
    constexpr int PC = seg_pieces<S>();
#pragma unroll
    for (int q = 0; q < PC; ++q)
        cp_async16(sm + ((size_t)slot * PC + q) * kK4Threads + threadIdx.x, slice + piece_off<S, true>(threadIdx.x, q));
}
template <typename S>
__device__ __forceinline__ void seg_unpack(const uint4 *sm, int slot, float *v) {
    constexpr int PC = seg_pieces<S>();
    Packed<S> x;
    uint4 *w = reinterpret_cast<uint4 *>(&x);
#pragma unroll
    for (int q = 0; q < PC; ++q) w[q] = sm[((size_t)slot * PC + q) * kK4Threads + threadIdx.x];
    unpack16(x, v);  // pieces in order: entries q * EP .. q * EP + EP - 1
}

// Where ticket t lies: segment r of state slice `slice` of chain (bi, h).
struct SegPos {
    int r, slice, h, bi;
    long long bh;
};
__device__ __forceinline__ SegPos seg_pos(const Params &p, const SegDev &g, long long t) {
    SegPos q;
    q.r = (int)(t / g.pairs);
    const long long pair = t % g.pairs;
    q.slice = (int)(pair % g.slices);
    q.bh = pair / g.slices;
    q.h = (int)(q.bh % p.H);
    q.bi = (int)(q.bh / p.H);
    return q;
}

// Persistent blocks, two segment buffers each: a block draws its next ticket
// and issues that segment's copies as soon as the current segment's reduction
// is published, so the copies run under the current segment's wait, fold and
// rescan.  A block finishes its tickets in the order it drew them, and a
// ticket waits only on smaller ones, so the smallest unfinished ticket can
// always finish.
template <typename S, int T>
__global__ void __launch_bounds__(kK4Threads, 3) k4_state_passing_seg(Params p, S *st, SegDev g, int write_final) {
    extern __shared__ uint4 seg_sm[];
    __shared__ int tk[2];
    const long long total = g.pairs * g.K;
    const size_t PN = (size_t)p.P * p.N;
    auto issue = [&](long long t, int buf) {
        const SegPos q = seg_pos(p, g, t);
        for (int u = 0; u < T; ++u) {
            const int c = q.r * T + u;
            if (c < p.n) seg_stage<S>(seg_sm, buf * T + u, st + ix_state(p, q.bi, c, q.h) + (size_t)q.slice * kSegSlice);
        }
    };
    int slot = 0, buf = 0;
    long long t = seg_draw(g, &tk[slot]);
    if (t < total) issue(t, buf);
    while (t < total) {
        // the next ticket's atomic goes out first; its value is needed only
        // after the reduction (so its round trip overlaps the copy wait)
        int nxt = 0;
        if (threadIdx.x == 0) nxt = atomicAdd(g.ticket, 1);
        const SegPos q = seg_pos(p, g, t);
        const long long pair = t % g.pairs;
        const int c0 = q.r * T;
        const size_t soff = (size_t)q.slice * kSegSlice;
        const float *endA = p.endA + ix_chunk(p, q.bi, q.h, 0);
        float a[T];
#pragma unroll
        for (int u = 0; u < T; ++u) a[u] = c0 + u < p.n ? __expf(endA[c0 + u]) : 1.f;
        cp_async_wait_all();
        // 1. the segment's reduction from a zero state
        float acc[kVec], dec = 1.f;
#pragma unroll
        for (int i = 0; i < kVec; ++i) acc[i] = 0.f;
#pragma unroll
        for (int u = 0; u < T; ++u) {
            if (c0 + u < p.n) {
                dec *= a[u];
                float x[kVec];
                seg_unpack<S>(seg_sm, buf * T + u, x);
#pragma unroll
                for (int i = 0; i < kVec; ++i) acc[i] = fmaf(a[u], acc[i], x[i]);
            }
        }
        // (the slot was last read before the previous iteration's barriers)
        slot ^= 1;
        if (threadIdx.x == 0) tk[slot] = nxt;
        if (q.r < g.K - 1) {
            if (threadIdx.x == 0) p.k4s_dec[(size_t)pair * g.K + q.r] = dec;
            seg_publish(p.k4s_agg + ((size_t)pair * g.K + q.r) * kSegSlice, acc, g.aggflag + pair * g.K + q.r);
        } else {
            __syncthreads();
        }
        // the next segment's copies go out now
        const long long t2 = tk[slot];
        if (t2 < total) issue(t2, buf ^ 1);
        // 2. the carry in
        float sv[kVec];
        seg_carry<S>(p, g, pair, q.r, p.init ? p.init + q.bh * PN + soff : nullptr, sv);
        // 3. the chunk-input states
#pragma unroll
        for (int u = 0; u < T; ++u) {
            const int c = c0 + u;
            if (c < p.n) {
                st_vals<S, true>(st + ix_state(p, q.bi, c, q.h) + soff, threadIdx.x, sv);
                float x[kVec];
                seg_unpack<S>(seg_sm, buf * T + u, x);
#pragma unroll
                for (int i = 0; i < kVec; ++i) sv[i] = fmaf(a[u], sv[i], x[i]);
            }
        }
        if (q.r == g.K - 1 && write_final && p.final_state) st_f32<S, true>(p.final_state + q.bh * PN + soff, threadIdx.x, sv);
        t = t2;
        buf ^= 1;
    }
}

// Shared memory (64 KB: three blocks per SM) and grid of a segmented kernel:
// the blocks that fit on the device at once, at most one per ticket.
template <typename K>
static cudaError_t seg_prepare(K kernel, const K4SegGeom &sg, unsigned *blocks) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSegSmem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kK4Threads, kSegSmem)) != cudaSuccess)
        return e;
    const long long total = sg.pairs * sg.K, fit = (long long)sms * (per_sm > 0 ? per_sm : 1);
    *blocks = (unsigned)(total < fit ? total : fit);
    return cudaSuccess;
}

// chunks per segment: 64 KB of shared memory holds two buffers of T chunks of
// 16 entries a thread
K4SegGeom k4_seg_geom(long long b, long long H, long long P, long long N, long long n, bool fp32_states) {
    K4SegGeom g;
    g.slices = (int)((P * N / kVec + kK4Threads - 1) / kK4Threads);
    g.pairs = b * H * g.slices;
    g.T = fp32_states ? 4 : 8;
    g.K = (int)((n + g.T - 1) / g.T);
    g.KG = (g.K + kK4SegGroup - 1) / kK4SegGroup;
    // (the 32-bit ticket counter ends at the tickets plus one per block)
    g.on = (P * N) % (kK4Threads * kVec) == 0 && g.pairs <= kK4SegMaxBlocks && g.K >= 2 &&
           g.pairs * (long long)g.K <= (1LL << 30);
    return g;
}

size_t k4_seg_sync_ints(long long b, long long H, long long P, long long N, long long n, bool fp32_states) {
    const K4SegGeom f = k4_seg_geom(b, H, P, N, n, fp32_states);
    return f.on ? kK4SegSyncHead + (size_t)f.pairs * (f.K + f.KG) : 0;
}

// Device view of the geometry: ticket counter, then the ready flags.
static SegDev seg_dev(const Params &p, const K4SegGeom &g) {
    SegDev d;
    d.K = g.K;
    d.KG = g.KG;
    d.slices = g.slices;
    d.pairs = g.pairs;
    d.ticket = p.k4s_sync;
    d.aggflag = p.k4s_sync + kK4SegSyncHead;
    d.carryflag = d.aggflag + (size_t)g.pairs * g.K;
    return d;
}

// blocks per SM of a K4 grid on this device (1: at most one block on every SM)
static int k4_per_sm(long long blocks) {
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return (int)((blocks + sms - 1) / sms);
}

// The same recurrence for grids of at most two blocks per SM (few chains): two
// register batches of U chunks, the next batch's loads issued before the
// current one is processed, so every wait is on loads issued a batch earlier.
template <typename S, int U, int MB, bool IL>
__global__ void __launch_bounds__(kK4Threads, MB) k4_state_passing_batched(Params p, S *st, int write_final) {
    const size_t PN = (size_t)p.P * p.N, nvec = PN / kVec;
    const size_t gid = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    if (gid >= (size_t)p.b * p.H * nvec) return;
    const size_t e = gid % nvec, bh = gid / nvec;
    const int h = (int)(bh % p.H), bi = (int)(bh / p.H);
    float s[kVec];
    if (p.init) ld_f32<S, IL>(p.init + bh * PN, e, s);
    else {
#pragma unroll
        for (int i = 0; i < kVec; ++i) s[i] = 0.f;
    }
    const float *endA = p.endA + ix_chunk(p, bi, h, 0);
    Packed<S> ba[U], bb[U];
    float ea[U], eb[U];
    auto issue = [&](Packed<S>(&buf)[U], float(&eav)[U], int c0) {
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (c0 + u < p.n) {
                buf[u] = ld_packed<S, IL>(st + ix_state(p, bi, c0 + u, h), e);
                eav[u] = endA[c0 + u];
            }
    };
    auto step = [&](Packed<S>(&buf)[U], float(&eav)[U], int c0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + u;
            if (c < p.n) {
                st_vals<S, IL>(st + ix_state(p, bi, c, h), e, s);
                const float a = __expf(eav[u]);
                float v[kVec];
                unpack16(buf[u], v);
#pragma unroll
                for (int i = 0; i < kVec; ++i) s[i] = fmaf(a, s[i], v[i]);
            }
        }
    };
    issue(ba, ea, 0);
    for (int c0 = 0; c0 < p.n; c0 += 2 * U) {
        issue(bb, eb, c0 + U);
        step(ba, ea, c0);
        issue(ba, ea, c0 + 2 * U);
        step(bb, eb, c0 + U);
    }
    if (write_final && p.final_state) st_f32<S, IL>(p.final_state + bh * PN, e, s);
}

template <bool IL>
static cudaError_t launch_k4_plain(const Params &p, bool write_final, cudaStream_t s) {
    const long long nthr = (long long)p.b * p.H * ((long long)p.P * p.N / kVec);
    const long long blocks = (nthr + kK4Threads - 1) / kK4Threads;
    const int per_sm = k4_per_sm(blocks), wf = write_final ? 1 : 0;
    const unsigned g = (unsigned)blocks;
    if (p.states) {  // fp32 states: 16 registers per chunk in a batch
        if (per_sm <= 1) k4_state_passing_batched<float, 4, 1, IL><<<g, kK4Threads, 0, s>>>(p, p.states, wf);
        else if (per_sm <= 2) k4_state_passing_batched<float, 2, 2, IL><<<g, kK4Threads, 0, s>>>(p, p.states, wf);
        else k4_state_passing<float, 2, IL><<<g, kK4Threads, 0, s>>>(p, p.states, wf);
    } else {         // bf16 states: 8 registers per chunk
        if (per_sm <= 1) k4_state_passing_batched<bf16, 8, 1, IL><<<g, kK4Threads, 0, s>>>(p, p.states_bf, wf);
        else if (per_sm <= 2) k4_state_passing_batched<bf16, 4, 2, IL><<<g, kK4Threads, 0, s>>>(p, p.states_bf, wf);
        else k4_state_passing<bf16, 4, IL><<<g, kK4Threads, 0, s>>>(p, p.states_bf, wf);
    }
    return cudaGetLastError();
}

cudaError_t launch_k4_state_passing(const Params &p, bool write_final, cudaStream_t s) {
    const K4SegGeom sg = k4_seg_geom(p.b, p.H, p.P, p.N, p.n, p.states != nullptr);
    if (sg.on) {
        const SegDev g = seg_dev(p, sg);
        const int wf = write_final ? 1 : 0;
        if (p.states) {
            auto k = k4_state_passing_seg<float, 4>;
            unsigned blocks = 0;
            cudaError_t e = seg_prepare(k, sg, &blocks);
            if (e != cudaSuccess) return e;
            k<<<blocks, kK4Threads, kSegSmem, s>>>(p, p.states, g, wf);
        } else {
            auto k = k4_state_passing_seg<bf16, 8>;
            unsigned blocks = 0;
            cudaError_t e = seg_prepare(k, sg, &blocks);
            if (e != cudaSuccess) return e;
            k<<<blocks, kK4Threads, kSegSmem, s>>>(p, p.states_bf, g, wf);
        }
        return cudaGetLastError();
    }
    const bool il = ((long long)p.P * p.N) % (kK4Threads * kVec) == 0;
    return il ? launch_k4_plain<true>(p, write_final, s) : launch_k4_plain<false>(p, write_final, s);
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
template <typename S, int U, int MB, bool IL>
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
    if (active && p.d_final) ld_f32<S, IL>(p.d_final + (size_t)bh * PN, e, d);
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
                const size_t off = ix_state(p, bi, c, h);
                dsin[u] = ld_packed<S, IL>(dst + off, e);
                sin_[u] = ld_packed<S, IL>(st + off, e);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 - u;
            if (c < 0) break;
            const float a = __expf(endA[c]);
            float part = 0.f;
            if (active) {
                st_vals<S, IL>(dst + ix_state(p, bi, c, h), e, d);
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
    if (active && p.d_init) st_f32<S, IL>(p.d_init + (size_t)bh * PN, e, d);
}

template <bool IL>
static cudaError_t launch_bwd_k4_plain(const Params &p, cudaStream_t s) {
    const long long nvec = (long long)p.P * p.N / kVec;
    const long long blocks = (long long)p.b * p.H * ((nvec + kK4Threads - 1) / kK4Threads);
    const int per_sm = k4_per_sm(blocks);
    const unsigned g = (unsigned)blocks;
    // two chunks (d_s_in and s_in) per step read ahead in batches of U; one block per
    // SM: deep, else five per SM.  (Measured on the 131k-token sequence: a time-
    // segmented backward and two register batches of half the depth were both slower.)
    if (p.dstates) {
        if (per_sm <= 1) bwd_k4_state_passing<float, 4, 1, IL><<<g, kK4Threads, 0, s>>>(p, p.dstates, p.states);
        else bwd_k4_state_passing<float, 2, 5, IL><<<g, kK4Threads, 0, s>>>(p, p.dstates, p.states);
    } else {
        if (per_sm <= 1) bwd_k4_state_passing<bf16, 8, 1, IL><<<g, kK4Threads, 0, s>>>(p, p.dstates_bf, p.states_bf);
        else bwd_k4_state_passing<bf16, 4, 5, IL><<<g, kK4Threads, 0, s>>>(p, p.dstates_bf, p.states_bf);
    }
    return cudaGetLastError();
}

cudaError_t launch_bwd_k4(const Params &p, cudaStream_t s) {
    const bool il = ((long long)p.P * p.N) % (kK4Threads * kVec) == 0;
    return il ? launch_bwd_k4_plain<true>(p, s) : launch_bwd_k4_plain<false>(p, s);
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
