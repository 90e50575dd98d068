// ssd_simt.cu -- CUDA-core (FFMA) kernels for the contractions of the SSD scan.
//
// This is the fp32 product path (tensor cores cannot hold the fp32 path's
// accuracy) and the general-shape path of bf16.  Every kernel stages its
// operands through shared memory in small token tiles and accumulates in fp32
// registers; all reductions run in a fixed order, so results are
// deterministic.  The formulas are those of burn-mamba's "combined_backward.rs"
// page: K2 (CB = C B^T per chunk), K3 extended (intra-chunk state with the
// scale dt * exp(cumA_last - cumA)), the BLUE / ORANGE / skip terms of the
// chunk scan, and their backward (BLUE, ORANGE, K3 and K2 backward blocks).
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr int kThreads = 256;
constexpr int kTok = 32;     // token tile of the staged operands
constexpr int kOutPer = 8;   // outputs per thread in the P x N / rows x P kernels

template <typename T>
__device__ __forceinline__ float ld_tok(const Params &p, const T *a, size_t i, int t, int V) {
    return t < V ? ldf(a, i) : 0.f;
}

// Floats of the "other rows" buffer of the main backward kernel: 32 rows of P
// (+1 pad), reused as a [P][33] state tile.
__host__ __device__ __forceinline__ int main_other_floats(int P) {
    return 32 * (P + 1) > 33 * P ? 32 * (P + 1) : 33 * P;
}

// exp(cumA_t - cumA_s) for s <= t, 0 otherwise (the causal decay of ORANGE).
__device__ __forceinline__ float causal_decay(const float *cum, int t, int s) {
    return s <= t ? __expf(cum[t] - cum[s]) : 0.f;
}

}  // namespace

// ================================================================== K2: CB = C B^T
// Block = one 16 x 16 (t, s) tile of one (b, chunk, group); tiles strictly above
// the diagonal are never read and are skipped.
template <typename T>
__global__ void simt_k2(Params p) {
    __shared__ float Cs[16][17], Bs[16][17];
    const int nt = p.Q / 16;
    const int ts = blockIdx.x % (nt * nt), bng = blockIdx.x / (nt * nt);
    const int tt = ts / nt, st = ts % nt;
    if (st > tt) return;
    const int g = bng % p.G, c = (bng / p.G) % p.n, bi = bng / (p.G * p.n);
    const int V = valid_len_of(p, bi);
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    const T *Bp = (const T *)p.B, *Cp = (const T *)p.C;
    float acc = 0.f;
    for (int r0 = 0; r0 < p.N; r0 += 16) {
        const int tC = c * p.Q + tt * 16 + ty, tB = c * p.Q + st * 16 + ty, r = r0 + tx;
        Cs[ty][tx] = (r < p.N) ? ld_tok(p, Cp, ix_bc(p, bi, tC, g, r), tC, V) : 0.f;
        Bs[ty][tx] = (r < p.N) ? ld_tok(p, Bp, ix_bc(p, bi, tB, g, r), tB, V) : 0.f;
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 16; ++k) acc += Cs[ty][k] * Bs[tx][k];
        __syncthreads();
    }
    p.CB[ix_cb(p, bi, c, g) + (size_t)(tt * 16 + ty) * p.Q + st * 16 + tx] = acc;
}

template <typename T>
cudaError_t launch_simt_k2(const Params &p, cudaStream_t s) {
    const int nt = p.Q / 16;
    simt_k2<T><<<(unsigned)((long long)nt * nt * p.b * p.n * p.G), 256, 0, s>>>(p);
    return cudaGetLastError();
}

// ================================================================== "outer" contraction
// out[p, r] = sum_l U[l, p] * V[l, r] over the chunk's Q tokens, one block per
// (b, chunk, head) and output slice of kThreads * kOutPer entries.  Used by K3
// (U = x, V = B * dt * exp(cumA_last - cumA)) and by the BLUE backward
// (U = dy * exp(cumA), V = C).
template <typename T, bool kBlue>
__global__ void simt_outer(Params p, float *out) {
    extern __shared__ float sm[];
    float *Us = sm;                  // [kTok][P]
    float *Vs = sm + kTok * p.P;     // [kTok][N]
    const int PN = p.P * p.N;
    const int nslice = (PN + kThreads * kOutPer - 1) / (kThreads * kOutPer);
    const int slice = blockIdx.x % nslice, bnh = blockIdx.x / nslice;
    const int h = bnh % p.H, c = (bnh / p.H) % p.n, bi = bnh / (p.H * p.n);
    const int g = h / p.hpg;
    const int V = valid_len_of(p, bi);
    const float *cum = p.cumA + ix_chunk(p, bi, h, c) * p.Q;
    const float cend = p.endA[ix_chunk(p, bi, h, c)];
    const T *Up = kBlue ? (const T *)p.dy : (const T *)p.x;
    const T *Vp = kBlue ? (const T *)p.C : (const T *)p.B;
    float acc[kOutPer];
#pragma unroll
    for (int j = 0; j < kOutPer; ++j) acc[j] = 0.f;
    for (int l0 = 0; l0 < p.Q; l0 += kTok) {
        for (int i = threadIdx.x; i < kTok * p.P; i += kThreads) {
            const int l = i / p.P, pp = i % p.P, t = c * p.Q + l0 + l;
            float v = 0.f;
            if (l0 + l < p.Q && t < V) {
                v = ldf(Up, ix_x(p, bi, t, h, pp));
                if (kBlue) v *= __expf(cum[l0 + l]);
            }
            Us[i] = v;
        }
        for (int i = threadIdx.x; i < kTok * p.N; i += kThreads) {
            const int l = i / p.N, r = i % p.N, t = c * p.Q + l0 + l;
            float v = 0.f;
            if (l0 + l < p.Q && t < V) {
                v = ldf(Vp, ix_bc(p, bi, t, g, r));
                if (!kBlue) v *= p.dt[ix_dt(p, bi, h, t)] * __expf(cend - cum[l0 + l]);
            }
            Vs[i] = v;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kOutPer; ++j) {
            const int o = (slice * kOutPer + j) * kThreads + threadIdx.x;
            if (o < PN) {
                const int pp = o / p.N, r = o % p.N;
                float a = acc[j];
                for (int l = 0; l < kTok; ++l) a += Us[l * p.P + pp] * Vs[l * p.N + r];
                acc[j] = a;
            }
        }
        __syncthreads();
    }
    float *dst = out + ix_state(p, bi, c, h);
#pragma unroll
    for (int j = 0; j < kOutPer; ++j) {
        const int o = (slice * kOutPer + j) * kThreads + threadIdx.x;
        if (o < PN) dst[o] = acc[j];
    }
}

template <typename T>
cudaError_t launch_simt_k3(const Params &p, cudaStream_t s) {
    const int PN = p.P * p.N;
    const int nslice = (PN + kThreads * kOutPer - 1) / (kThreads * kOutPer);
    const size_t smem = sizeof(float) * kTok * (p.P + p.N);
    simt_outer<T, false><<<(unsigned)((long long)p.b * p.n * p.H * nslice), kThreads, smem, s>>>(
        p, p.states);
    return cudaGetLastError();
}

// ================================================================== row-block contraction
// For rows t of one (b, chunk, head) row tile:
//   blue[t, p] = exp(cumA_t) * sum_r C[t, r] * s_in[p, r]
// computed into acc[] (thread owns rows x P outputs o = tid + kThreads * j).
template <typename T>
__device__ void blue_rows(const Params &p, int bi, int c, int h, int t0, int rows, int V,
                          float *Cs, float *Ss, float *acc) {
    const int g = h / p.hpg;
    const float *cum = p.cumA + ix_chunk(p, bi, h, c) * p.Q;
    const float *sin_ = p.states + ix_state(p, bi, c, h);
    const T *Cp = (const T *)p.C;
    for (int r0 = 0; r0 < p.N; r0 += 32) {
        for (int i = threadIdx.x; i < rows * 32; i += kThreads) {
            const int tl = i / 32, r = r0 + i % 32, q = t0 + tl, t = c * p.Q + q;
            float v = 0.f;
            if (r < p.N && q < p.Q && t < V) v = ldf(Cp, ix_bc(p, bi, t, g, r)) * __expf(cum[q]);
            Cs[i] = v;
        }
        for (int i = threadIdx.x; i < p.P * 32; i += kThreads) {
            const int pp = i / 32, r = r0 + i % 32;
            Ss[pp * 33 + i % 32] = r < p.N ? sin_[(size_t)pp * p.N + r] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kOutPer; ++j) {
            const int o = j * kThreads + threadIdx.x;
            if (o < rows * p.P) {
                const int tl = o / p.P, pp = o % p.P;
                float a = acc[j];
#pragma unroll 8
                for (int k = 0; k < 32; ++k) a += Cs[tl * 32 + k] * Ss[pp * 33 + k];
                acc[j] = a;
            }
        }
        __syncthreads();
    }
}

// ================================================================== K5: chunk scan
// Block = (b, chunk, head, tile of kRows5 target rows t).  y = BLUE + ORANGE + D x,
// ORANGE[t, p] = sum_{s <= t} CB[t, s] exp(cumA_t - cumA_s) dt_s x[s, p].
constexpr int kRows5 = 16;

template <typename T>
__global__ void simt_k5(Params p) {
    extern __shared__ float sm[];
    float *Cs = sm;                        // [kRows5][32]
    float *Ss = Cs + kRows5 * 32;          // [P][33]
    float *Ws = Ss + p.P * 33;             // [kRows5][32]
    float *Xs = Ws + kRows5 * 32;          // [32][P]
    const int ntile = p.Q / kRows5;
    const int tile = blockIdx.x % ntile, bnh = blockIdx.x / ntile;
    const int h = bnh % p.H, c = (bnh / p.H) % p.n, bi = bnh / (p.H * p.n);
    const int g = h / p.hpg;
    const int V = valid_len_of(p, bi);
    const int t0 = tile * kRows5;
    const float *cum = p.cumA + ix_chunk(p, bi, h, c) * p.Q;
    const float *cb = p.CB + ix_cb(p, bi, c, g);
    const T *Xp = (const T *)p.x;
    float acc[kOutPer];
#pragma unroll
    for (int j = 0; j < kOutPer; ++j) acc[j] = 0.f;
    blue_rows<T>(p, bi, c, h, t0, kRows5, V, Cs, Ss, acc);
    // ORANGE over source tiles that intersect s <= t
    for (int s0 = 0; s0 < t0 + kRows5; s0 += 32) {
        for (int i = threadIdx.x; i < kRows5 * 32; i += kThreads) {
            const int tl = i / 32, sl = i % 32, q = t0 + tl, sq = s0 + sl;
            const int ts = c * p.Q + sq;
            float w = 0.f;
            if (sq < p.Q && sq <= q && ts < V)
                w = cb[(size_t)q * p.Q + sq] * causal_decay(cum, q, sq) * p.dt[ix_dt(p, bi, h, ts)];
            Ws[i] = w;
        }
        for (int i = threadIdx.x; i < 32 * p.P; i += kThreads) {
            const int sl = i / p.P, pp = i % p.P, sq = s0 + sl, ts = c * p.Q + sq;
            Xs[i] = (sq < p.Q && ts < V) ? ldf(Xp, ix_x(p, bi, ts, h, pp)) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kOutPer; ++j) {
            const int o = j * kThreads + threadIdx.x;
            if (o < kRows5 * p.P) {
                const int tl = o / p.P, pp = o % p.P;
                float a = acc[j];
#pragma unroll 8
                for (int k = 0; k < 32; ++k) a += Ws[tl * 32 + k] * Xs[k * p.P + pp];
                acc[j] = a;
            }
        }
        __syncthreads();
    }
    T *Yp = (T *)p.y;
    const float Dh = p.D[h];
#pragma unroll
    for (int j = 0; j < kOutPer; ++j) {
        const int o = j * kThreads + threadIdx.x;
        if (o < kRows5 * p.P) {
            const int tl = o / p.P, pp = o % p.P, t = c * p.Q + t0 + tl;
            if (t < p.L) {
                const size_t xi = ix_x(p, bi, t, h, pp);
                stf(Yp, xi, t < V ? acc[j] + Dh * ldf(Xp, xi) : 0.f);
            }
        }
    }
}

template <typename T>
cudaError_t launch_simt_k5(const Params &p, cudaStream_t s) {
    const size_t smem = sizeof(float) * (kRows5 * 32 * 2 + p.P * 33 + 32 * p.P);
    simt_k5<T><<<(unsigned)((long long)p.b * p.n * p.H * (p.Q / kRows5)), kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

// ================================================================== BLUE backward
// d_s_in[p, r] = sum_l dy[l, p] exp(cumA_l) C[l, r]          (into dstates)
// d_cumA_blue[l] = sum_p dy[l, p] * blue[l, p]                (BLUE row dot)
template <typename T>
__global__ void simt_bwd_blue_da(Params p) {
    extern __shared__ float sm[];
    __shared__ float red[32];
    float *Cs = sm;                  // [kRows5][32]
    float *Ss = Cs + kRows5 * 32;    // [P][33]
    float *rowv = Ss + p.P * 33;     // [kRows5]
    const int ntile = p.Q / kRows5;
    const int tile = blockIdx.x % ntile, bnh = blockIdx.x / ntile;
    const int h = bnh % p.H, c = (bnh / p.H) % p.n, bi = bnh / (p.H * p.n);
    const int V = valid_len_of(p, bi);
    const int t0 = tile * kRows5;
    float acc[kOutPer];
#pragma unroll
    for (int j = 0; j < kOutPer; ++j) acc[j] = 0.f;
    blue_rows<T>(p, bi, c, h, t0, kRows5, V, Cs, Ss, acc);
    const T *DYp = (const T *)p.dy;
    for (int i = threadIdx.x; i < kRows5; i += kThreads) rowv[i] = 0.f;
    __syncthreads();
    // row dots in a fixed order: per row, sum over p of dy * blue
    for (int tl = 0; tl < kRows5; ++tl) {
        float v = 0.f;
#pragma unroll
        for (int j = 0; j < kOutPer; ++j) {
            const int o = j * kThreads + threadIdx.x;
            if (o < kRows5 * p.P && o / p.P == tl) {
                const int t = c * p.Q + t0 + tl;
                if (t < V) v += acc[j] * ldf(DYp, ix_x(p, bi, t, h, o % p.P));
            }
        }
        v = block_sum(v, red);
        if (threadIdx.x == 0) rowv[tl] = v;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kRows5; i += kThreads)
        p.dcum_blue[ix_chunk(p, bi, h, c) * p.Q + t0 + i] = rowv[i];
}

template <typename T>
cudaError_t launch_simt_bwd_blue(const Params &p, cudaStream_t s) {
    const int PN = p.P * p.N;
    const int nslice = (PN + kThreads * kOutPer - 1) / (kThreads * kOutPer);
    const size_t smem_o = sizeof(float) * kTok * (p.P + p.N);
    simt_outer<T, true><<<(unsigned)((long long)p.b * p.n * p.H * nslice), kThreads, smem_o, s>>>(
        p, p.dstates);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem_d = sizeof(float) * (kRows5 * 32 + p.P * 33 + kRows5);
    simt_bwd_blue_da<T><<<(unsigned)((long long)p.b * p.n * p.H * (p.Q / kRows5)), kThreads,
                          smem_d, s>>>(p);
    return cudaGetLastError();
}

// ================================================================== main backward
// Block = (b, chunk, head, tile of kMainRows rows k).  For the tile's rows, as
// SOURCE positions s:
//   dx[s, p]        = D dy[s, p] + sum_{t >= s} W[t, s] dy[t, p] + bbs[s] U[s, p]
//   ddt_orange[s]   = sum_{t >= s} dW[t, s] CB[t, s] decay[t, s]
//   src[s]          = sum_{t >= s} dW[t, s] W[t, s]
// as TARGET positions t:
//   tgt[t]          = sum_{s <= t} dW[t, s] W[t, s]
// with dW = dy x^T, W = CB * decay * dt_s (causal), U = B d_intra^T, and the
// K3 terms d_bbs[s] = sum_p x[s, p] U[s, p], ddt_k3 = d_bbs decay_end,
// d_delta = d_bbs dt decay_end.  Writes dx, ddt_main = ddt_orange + ddt_k3,
// dcum_main = tgt - src - d_delta, d_delta, and the tile's dD partial.
template <typename T>
__global__ void simt_bwd_main(Params p) {
    extern __shared__ float sm[];
    __shared__ float red[32];
    constexpr int R = kMainRows;
    const int ot_sz = main_other_floats(p.P);
    float *DYk = sm;                  // [R][P]   dy of the tile rows
    float *Xk = DYk + R * p.P;        // [R][P]   x of the tile rows
    float *Ot = Xk + R * p.P;         // [32][P+1] other-side rows (dy or x); later d_intra [P][33]
    float *Wt = Ot + ot_sz;           // [32][R]  W (as [t][s]) for the current other tile
    float *Gt = Wt + 32 * R;          // [32][R]  dW * CB * decay
    float *Bk = Gt + 32 * R;          // [R][32]  B tile for U
    float *acc_s = Bk + R * 32;       // [R] ddt_orange, [R] src, [R] tgt, [R] d_bbs
    const int ntile = p.Q / R;
    const int tile = blockIdx.x % ntile, bnh = blockIdx.x / ntile;
    const int h = bnh % p.H, c = (bnh / p.H) % p.n, bi = bnh / (p.H * p.n);
    const int g = h / p.hpg;
    const int V = valid_len_of(p, bi);
    const int k0 = tile * R;
    const float *cum = p.cumA + ix_chunk(p, bi, h, c) * p.Q;
    const float cend = p.endA[ix_chunk(p, bi, h, c)];
    const float *cb = p.CB + ix_cb(p, bi, c, g);
    const T *Xp = (const T *)p.x, *DYp = (const T *)p.dy, *Bp = (const T *)p.B;
    auto dt_of = [&](int q) -> float {
        const int t = c * p.Q + q;
        return (q < p.Q && t < V) ? p.dt[ix_dt(p, bi, h, t)] : 0.f;
    };

    for (int i = threadIdx.x; i < R * p.P; i += kThreads) {
        const int kl = i / p.P, pp = i % p.P, t = c * p.Q + k0 + kl;
        const bool ok = k0 + kl < p.Q && t < V;
        DYk[i] = ok ? ldf(DYp, ix_x(p, bi, t, h, pp)) : 0.f;
        Xk[i] = ok ? ldf(Xp, ix_x(p, bi, t, h, pp)) : 0.f;
    }
    for (int i = threadIdx.x; i < 4 * R; i += kThreads) acc_s[i] = 0.f;
    float dxa[kOutPer];
#pragma unroll
    for (int j = 0; j < kOutPer; ++j) dxa[j] = 0.f;
    __syncthreads();

    // ---- (1) tile rows as sources s: loop over target tiles t >= k0
    for (int t0 = (k0 / 32) * 32; t0 < p.Q; t0 += 32) {
        for (int i = threadIdx.x; i < 32 * p.P; i += kThreads) {
            const int tl = i / p.P, pp = i % p.P, q = t0 + tl, t = c * p.Q + q;
            Ot[tl * (p.P + 1) + pp] = (q < p.Q && t < V) ? ldf(DYp, ix_x(p, bi, t, h, pp)) : 0.f;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < 32 * R; i += kThreads) {
            const int tl = i / R, sl = i % R, q = t0 + tl, sq = k0 + sl;
            float w = 0.f, gv = 0.f;
            if (q < p.Q && sq <= q) {
                float dw = 0.f;
                for (int pp = 0; pp < p.P; ++pp) dw += Ot[tl * (p.P + 1) + pp] * Xk[sl * p.P + pp];
                const float cbd = cb[(size_t)q * p.Q + sq] * causal_decay(cum, q, sq);
                w = cbd * dt_of(sq);
                gv = dw * cbd;
            }
            Wt[i] = w;
            Gt[i] = gv;
        }
        __syncthreads();
        // per-source sums (fixed order over t)
        for (int sl = threadIdx.x; sl < R; sl += kThreads) {
            float a = 0.f, b = 0.f;
            for (int tl = 0; tl < 32; ++tl) {
                a += Gt[tl * R + sl];
                b += Gt[tl * R + sl] * dt_of(k0 + sl);
            }
            acc_s[sl] += a;          // ddt_orange
            acc_s[R + sl] += b;      // src = sum dW * W
        }
#pragma unroll
        for (int j = 0; j < kOutPer; ++j) {
            const int o = j * kThreads + threadIdx.x;
            if (o < R * p.P) {
                const int sl = o / p.P, pp = o % p.P;
                float a = dxa[j];
                for (int tl = 0; tl < 32; ++tl) a += Wt[tl * R + sl] * Ot[tl * (p.P + 1) + pp];
                dxa[j] = a;
            }
        }
        __syncthreads();
    }

    // ---- (2) tile rows as targets t: loop over source tiles s <= k0 + R - 1
    for (int s0 = 0; s0 < k0 + R; s0 += 32) {
        for (int i = threadIdx.x; i < 32 * p.P; i += kThreads) {
            const int sl = i / p.P, pp = i % p.P, q = s0 + sl, t = c * p.Q + q;
            Ot[sl * (p.P + 1) + pp] = (q < p.Q && t < V) ? ldf(Xp, ix_x(p, bi, t, h, pp)) : 0.f;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < 32 * R; i += kThreads) {
            const int sl = i / R, kl = i % R, sq = s0 + sl, q = k0 + kl;
            float v = 0.f;
            if (sq < p.Q && sq <= q) {
                float dw = 0.f;
                for (int pp = 0; pp < p.P; ++pp) dw += DYk[kl * p.P + pp] * Ot[sl * (p.P + 1) + pp];
                v = dw * cb[(size_t)q * p.Q + sq] * causal_decay(cum, q, sq) * dt_of(sq);
            }
            Gt[i] = v;
        }
        __syncthreads();
        for (int kl = threadIdx.x; kl < R; kl += kThreads) {
            float a = 0.f;
            for (int sl = 0; sl < 32; ++sl) a += Gt[sl * R + kl];
            acc_s[2 * R + kl] += a;  // tgt
        }
        __syncthreads();
    }

    // ---- (3) K3 backward: U[s, p] = sum_r B[s, r] d_intra[p, r]
    const float *dint = p.dstates + ix_state(p, bi, c, h);
    float ua[kOutPer];
#pragma unroll
    for (int j = 0; j < kOutPer; ++j) ua[j] = 0.f;
    for (int r0 = 0; r0 < p.N; r0 += 32) {
        for (int i = threadIdx.x; i < R * 32; i += kThreads) {
            const int kl = i / 32, r = r0 + i % 32, q = k0 + kl, t = c * p.Q + q;
            Bk[i] = (r < p.N && q < p.Q && t < V) ? ldf(Bp, ix_bc(p, bi, t, g, r)) : 0.f;
        }
        for (int i = threadIdx.x; i < p.P * 32; i += kThreads) {
            const int pp = i / 32, r = r0 + i % 32;
            Ot[pp * 33 + i % 32] = r < p.N ? dint[(size_t)pp * p.N + r] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kOutPer; ++j) {
            const int o = j * kThreads + threadIdx.x;
            if (o < R * p.P) {
                const int kl = o / p.P, pp = o % p.P;
                float a = ua[j];
                for (int k = 0; k < 32; ++k) a += Bk[kl * 32 + k] * Ot[pp * 33 + k];
                ua[j] = a;
            }
        }
        __syncthreads();
    }
    // d_bbs[s] = sum_p x[s, p] U[s, p]  and the dD partial, fixed order
    float *dbbs = acc_s + 3 * R;
    for (int kl = 0; kl < R; ++kl) {
        float v = 0.f;
#pragma unroll
        for (int j = 0; j < kOutPer; ++j) {
            const int o = j * kThreads + threadIdx.x;
            if (o < R * p.P && o / p.P == kl) v += ua[j] * Xk[o];
        }
        v = block_sum(v, red);
        if (threadIdx.x == 0) dbbs[kl] = v;
    }
    float dd = 0.f;
    for (int i = threadIdx.x; i < R * p.P; i += kThreads) dd += DYk[i] * Xk[i];
    dd = block_sum(dd, red);
    __syncthreads();

    const size_t cbase = ix_chunk(p, bi, h, c) * p.Q;
    if (threadIdx.x == 0) p.dD_part[(((size_t)bi * p.n + c) * p.H + h) * p.dD_per + tile] = dd;
    for (int kl = threadIdx.x; kl < R; kl += kThreads) {
        const int q = k0 + kl;
        const float dec_end = __expf(cend - cum[q]);
        const float dbb = dbbs[kl];
        const float dtq = dt_of(q);
        const float ddelta = dbb * dtq * dec_end;
        p.ddt_main[cbase + q] = acc_s[kl] + dbb * dec_end;
        p.d_delta[cbase + q] = ddelta;
        p.dcum_main[cbase + q] = acc_s[2 * R + kl] - acc_s[R + kl] - ddelta;
    }
    T *DXp = (T *)p.dx;
    const float Dh = p.D[h];
#pragma unroll
    for (int j = 0; j < kOutPer; ++j) {
        const int o = j * kThreads + threadIdx.x;
        if (o < R * p.P) {
            const int kl = o / p.P, pp = o % p.P, q = k0 + kl, t = c * p.Q + q;
            if (q < p.Q && t < p.L) {
                const float bbs = dt_of(q) * __expf(cend - cum[q]);
                const float v = Dh * DYk[o] + dxa[j] + bbs * ua[j];
                stf(DXp, ix_x(p, bi, t, h, pp), t < V ? v : 0.f);
            }
        }
    }
}

template <typename T>
cudaError_t launch_simt_bwd_main(const Params &p, cudaStream_t s) {
    constexpr int R = kMainRows;
    const size_t smem = sizeof(float) * (2 * R * p.P + main_other_floats(p.P) + 3 * 32 * R + 4 * R);
    simt_bwd_main<T><<<(unsigned)((long long)p.b * p.n * p.H * (p.Q / R)), kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

// ================================================================== group backward
// (a) d_cb[t, s] = sum_{h in g} dt_h[s] decay_h[t, s] sum_p dy_h[t, p] x_h[s, p]   (s <= t)
template <typename T>
__global__ void simt_bwd_dcb(Params p) {
    extern __shared__ float sm[];
    float *DYs = sm;              // [16][P+1]
    float *Xs = DYs + 16 * (p.P + 1);
    const int nt = p.Q / 16;
    const int ts = blockIdx.x % (nt * nt), bng = blockIdx.x / (nt * nt);
    const int tt = ts / nt, st = ts % nt;
    if (st > tt) return;
    const int g = bng % p.G, c = (bng / p.G) % p.n, bi = bng / (p.G * p.n);
    const int V = valid_len_of(p, bi);
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    const int q = tt * 16 + ty, sq = st * 16 + tx;
    const T *Xp = (const T *)p.x, *DYp = (const T *)p.dy;
    float acc = 0.f;
    for (int hh = 0; hh < p.hpg; ++hh) {
        const int h = g * p.hpg + hh;
        for (int i = threadIdx.x; i < 16 * p.P; i += 256) {
            const int rl = i / p.P, pp = i % p.P;
            const int tq = c * p.Q + tt * 16 + rl, sqq = c * p.Q + st * 16 + rl;
            DYs[rl * (p.P + 1) + pp] = tq < V ? ldf(DYp, ix_x(p, bi, tq, h, pp)) : 0.f;
            Xs[rl * (p.P + 1) + pp] = sqq < V ? ldf(Xp, ix_x(p, bi, sqq, h, pp)) : 0.f;
        }
        __syncthreads();
        if (sq <= q) {
            float dw = 0.f;
            for (int pp = 0; pp < p.P; ++pp) dw += DYs[ty * (p.P + 1) + pp] * Xs[tx * (p.P + 1) + pp];
            const float *cum = p.cumA + ix_chunk(p, bi, h, c) * p.Q;
            const int ts_ = c * p.Q + sq;
            const float dts = ts_ < V ? p.dt[ix_dt(p, bi, h, ts_)] : 0.f;
            acc += dw * dts * causal_decay(cum, q, sq);
        }
        __syncthreads();
    }
    p.d_cb[ix_cb(p, bi, c, g) + (size_t)q * p.Q + sq] = sq <= q ? acc : 0.f;
}

// (b) per (b, chunk, group, tile of 16 rows l):
//   dC[l, r] = sum_{s <= l} d_cb[l, s] B[s, r] + sum_h sum_p dy_h[l, p] exp(cumA_h[l]) s_in_h[p, r]
//   dB[l, r] = sum_{t >= l} d_cb[t, l] C[t, r] + sum_h bbs_h[l] sum_p x_h[l, p] d_intra_h[p, r]
template <typename T>
__global__ void simt_bwd_dbc(Params p) {
    extern __shared__ float sm[];
    float *Ls = sm;                 // [16][32]   d_cb rows (l, s) or (t, l) transposed, or u rows
    float *Ms = Ls + 16 * 32;       // [32][N]    B / C rows, or state rows
    const int ntile = p.Q / 16;
    const int tile = blockIdx.x % ntile, bng = blockIdx.x / ntile;
    const int g = bng % p.G, c = (bng / p.G) % p.n, bi = bng / (p.G * p.n);
    const int V = valid_len_of(p, bi);
    const int l0 = tile * 16;
    const float *dcb = p.d_cb + ix_cb(p, bi, c, g);
    const T *Bp = (const T *)p.B, *Cp = (const T *)p.C, *Xp = (const T *)p.x, *DYp = (const T *)p.dy;
    constexpr int J = 16;  // 16 rows x N (<= 256) outputs / 256 threads
    float dC[J], dB[J];
#pragma unroll
    for (int j = 0; j < J; ++j) dC[j] = dB[j] = 0.f;
    const int nout = 16 * p.N;
    // K2 backward terms, over 32-row tiles of the other index
    for (int m0 = 0; m0 < p.Q; m0 += 32) {
        for (int pass = 0; pass < 2; ++pass) {
            // pass 0: dC += d_cb[l, m] B[m, :]  (m <= l);  pass 1: dB += d_cb[m, l] C[m, :]  (m >= l)
            if (pass == 0 && m0 > l0 + 15) continue;
            if (pass == 1 && m0 + 31 < l0) continue;
            for (int i = threadIdx.x; i < 16 * 32; i += 256) {
                const int ll = i / 32, ml = i % 32, lq = l0 + ll, mq = m0 + ml;
                float v = 0.f;
                if (mq < p.Q) v = pass == 0 ? (mq <= lq ? dcb[(size_t)lq * p.Q + mq] : 0.f)
                                            : (mq >= lq ? dcb[(size_t)mq * p.Q + lq] : 0.f);
                Ls[i] = v;
            }
            for (int i = threadIdx.x; i < 32 * p.N; i += 256) {
                const int ml = i / p.N, r = i % p.N, mq = m0 + ml, t = c * p.Q + mq;
                Ms[i] = (mq < p.Q && t < V) ? ldf(pass == 0 ? Bp : Cp, ix_bc(p, bi, t, g, r)) : 0.f;
            }
            __syncthreads();
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int o = j * 256 + threadIdx.x;
                if (o < nout) {
                    const int ll = o / p.N, r = o % p.N;
                    float a = 0.f;
                    for (int ml = 0; ml < 32; ++ml) a += Ls[ll * 32 + ml] * Ms[ml * p.N + r];
                    if (pass == 0) dC[j] += a; else dB[j] += a;
                }
            }
            __syncthreads();
        }
    }
    // BLUE dC and K3 dB terms, summed over the group's heads in order
    for (int hh = 0; hh < p.hpg; ++hh) {
        const int h = g * p.hpg + hh;
        const float *cum = p.cumA + ix_chunk(p, bi, h, c) * p.Q;
        const float cend = p.endA[ix_chunk(p, bi, h, c)];
        for (int pass = 0; pass < 2; ++pass) {
            const float *st = (pass == 0 ? p.states : p.dstates) + ix_state(p, bi, c, h);
            for (int p0 = 0; p0 < p.P; p0 += 32) {
                for (int i = threadIdx.x; i < 16 * 32; i += 256) {
                    const int ll = i / 32, pp = p0 + i % 32, q = l0 + ll, t = c * p.Q + q;
                    float v = 0.f;
                    if (pp < p.P && t < V) {
                        if (pass == 0) v = ldf(DYp, ix_x(p, bi, t, h, pp)) * __expf(cum[q]);
                        else v = ldf(Xp, ix_x(p, bi, t, h, pp)) * p.dt[ix_dt(p, bi, h, t)] *
                                 __expf(cend - cum[q]);
                    }
                    Ls[i] = v;
                }
                for (int i = threadIdx.x; i < 32 * p.N; i += 256) {
                    const int pl = i / p.N, r = i % p.N, pp = p0 + pl;
                    Ms[i] = pp < p.P ? st[(size_t)pp * p.N + r] : 0.f;
                }
                __syncthreads();
#pragma unroll
                for (int j = 0; j < J; ++j) {
                    const int o = j * 256 + threadIdx.x;
                    if (o < nout) {
                        const int ll = o / p.N, r = o % p.N;
                        float a = 0.f;
                        for (int pl = 0; pl < 32; ++pl) a += Ls[ll * 32 + pl] * Ms[pl * p.N + r];
                        if (pass == 0) dC[j] += a; else dB[j] += a;
                    }
                }
                __syncthreads();
            }
        }
    }
    T *dBp = (T *)p.dB, *dCp = (T *)p.dC;
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int o = j * 256 + threadIdx.x;
        if (o < nout) {
            const int ll = o / p.N, r = o % p.N, t = c * p.Q + l0 + ll;
            if (t < p.L) {
                const size_t i = ix_bc(p, bi, t, g, r);
                stf(dCp, i, t < V ? dC[j] : 0.f);
                stf(dBp, i, t < V ? dB[j] : 0.f);
            }
        }
    }
}

template <typename T>
cudaError_t launch_simt_bwd_group(const Params &p, cudaStream_t s) {
    const int nt = p.Q / 16;
    const size_t smem_a = sizeof(float) * 2 * 16 * (p.P + 1);
    simt_bwd_dcb<T><<<(unsigned)((long long)nt * nt * p.b * p.n * p.G), 256, smem_a, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem_b = sizeof(float) * (16 * 32 + 32 * p.N);
    simt_bwd_dbc<T><<<(unsigned)((long long)nt * p.b * p.n * p.G), 256, smem_b, s>>>(p);
    return cudaGetLastError();
}

#define SSD_INSTANTIATE(T)                                                        \
    template cudaError_t launch_simt_k2<T>(const Params &, cudaStream_t);         \
    template cudaError_t launch_simt_k3<T>(const Params &, cudaStream_t);         \
    template cudaError_t launch_simt_k5<T>(const Params &, cudaStream_t);         \
    template cudaError_t launch_simt_bwd_blue<T>(const Params &, cudaStream_t);   \
    template cudaError_t launch_simt_bwd_main<T>(const Params &, cudaStream_t);   \
    template cudaError_t launch_simt_bwd_group<T>(const Params &, cudaStream_t);
SSD_INSTANTIATE(float)
SSD_INSTANTIATE(bf16)
#undef SSD_INSTANTIATE

}  // namespace ssd
