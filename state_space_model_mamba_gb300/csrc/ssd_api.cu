// ssd_api.cu -- the C ABI declared in include/ssd.h: argument validation,
// workspace carving and the launch sequence of the forward and of the
// recompute backward (burn-mamba, "combined_backward.rs": recompute K1-K4
// from the leaves, BLUE backward, K4 backward, ORANGE + K3 backward, K2
// backward, K1 backward and the dA / dD reductions).
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <map>
#include <memory>
#include <mutex>
#include <utility>

#include "ssd.h"
#include "ssd_check.cuh"
#include "ssd_internal.cuh"
#include "ssd_tc.cuh"

namespace ssd {
namespace {

thread_local char g_last_error[512] = "";

ssd_status fail(ssd_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
ssd_status fail(ssd_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

// Diagnostics: kernels enqueued by the current call, and optional CUDA-event
// pairs recorded around every launch (ssd_profile_begin / ssd_profile_end).
thread_local int g_launches = 0;
struct Recorder {
    cudaEvent_t *ev = nullptr;  // 2 events per kernel: start, end
    int cap = 0;                // capacity in events
    int n = 0;                  // events recorded
    const char *names[4096];
};
thread_local Recorder g_rec;
thread_local char g_rec_only[64] = "";  // record only this kernel ("" = all)

cudaError_t mark_start(const char *name, cudaStream_t s) {
    ++g_launches;
    if (!g_rec.ev || g_rec.n + 2 > g_rec.cap) return cudaSuccess;
    if (g_rec_only[0] && strcmp(name, g_rec_only) != 0) return cudaSuccess;
    g_rec.names[(g_rec.n / 2) % 4096] = name;
    return cudaEventRecord(g_rec.ev[g_rec.n++], s);
}

cudaError_t mark_end(cudaStream_t s) {
    if (!g_rec.ev || (g_rec.n & 1) == 0) return cudaSuccess;
    return cudaEventRecord(g_rec.ev[g_rec.n++], s);
}

// A second stream per (device, caller stream), so that the backward's K2 (CB
// and CB^T, which only the ORANGE backward reads) and group kernels run on the
// SMs that the caller's chain leaves idle instead of between its kernels.  The
// caller's stream forks to it and joins back through events (aux marks the end
// of the group chain).  Each caller stream has its own side stream and lock, so
// callers on different streams neither serialise their enqueue nor queue their
// side kernels behind one another; the lock (held from the fork to the last
// join) only orders calls that share a caller stream.  Side streams and their
// events live until the process exits, one set per caller stream seen.
struct SideStream {
    cudaStream_t st = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr, aux = nullptr;
    std::mutex mu;
};
// The stream for the side chain's launches: the caller's own while every launch is
// being timed (ssd_profile_begin without a ssd_profile_only filter), so that each
// event pair brackets one kernel running alone; the side stream otherwise.
cudaStream_t side_stream_for(const SideStream *sd, cudaStream_t s) {
    return (g_rec.ev && !g_rec_only[0]) ? s : sd->st;
}
std::mutex g_side_mu;  // guards the table below (lookup and insertion only)
std::map<std::pair<int, cudaStream_t>, std::unique_ptr<SideStream>> g_side;

cudaError_t side_stream(cudaStream_t caller, SideStream **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_side_mu);
    std::unique_ptr<SideStream> &slot = g_side[std::make_pair(dev, caller)];
    if (!slot) {
        std::unique_ptr<SideStream> sd(new SideStream);
        if ((e = cudaStreamCreateWithFlags(&sd->st, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&sd->fork, cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&sd->join, cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&sd->aux, cudaEventDisableTiming)) != cudaSuccess) return e;
        slot = std::move(sd);
    }
    *out = slot.get();
    return cudaSuccess;
}

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct Layout {
    size_t status, cumA, endA, CB, states, states_bf, dstates, dstates_bf;
    size_t dcum_blue, dcum_main, d_delta, ddt_main, d_endA_part, dD_part, dA_part, d_cb, dBC_part;
    size_t d_cb_bf, cb_count, fin_count;
    size_t k4s_sync, k4s_agg, k4s_carry, k4s_dec;
    size_t clear;  // bytes from the workspace's start that every call zeroes (status words, K4 sync)
    int n_count;
    size_t total;
    int k4_nblk, dD_per, nslice, nslice_cb, nslice_k5, nslice_k3;
};

bool use_tensor_cores(const ssd_dims &d, ssd_dtype dt) {
    return dt == SSD_BF16 && !(d.flags & SSD_FLAG_SIMT) && tc_supported(d.headdim, d.dstate, d.chunk_len);
}

// The fused chunk-state scan (K1 + K3 + K4, one CTA per (b, head pair) walking
// the chunks in order) needs enough (b, h) chains to fill the GPU; with few,
// long chains the chunk-parallel K3 and the separate K4 pass are faster.
constexpr long long kMinScanChains = 64;
bool use_fused_scan(const Params &p, const ssd_dims &d) {
    return !(d.flags & SSD_FLAG_SPLIT_SCAN) && (long long)p.b * p.H >= kMinScanChains;
}

// In the backward the scan's chains may leave SMs idle (the 2.7B layer: 80 CTAs
// on 152 SMs); then K2 and the d_cb kernel, which read cumA but no chunk state,
// run beside it on the side stream.  Measured on GB300: 80 CTAs gain 2.7% of the
// step; 96 CTAs of the 130M layer (a 0.24 ms step) lose 3% to the extra launch
// on the critical path; 256 CTAs fill the GPU and lose 3%.  Hence at most 60%.
bool overlap_scan(const Params &p) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    return 5 * tc_state_scan_ctas(p) <= 3LL * sms;
}

Layout make_layout(const ssd_dims &d, ssd_dtype dt, bool backward) {
    Layout lo;
    memset(&lo, 0, sizeof(lo));
    const size_t b = d.batch, H = d.nheads, P = d.headdim, N = d.dstate, G = d.ngroups,
                 Q = d.chunk_len;
    const size_t n = (d.seqlen + d.chunk_len - 1) / d.chunk_len;
    const bool tc = use_tensor_cores(d, dt);
    const size_t tok = b * H * n * Q, nst = b * n * H * P * N;
    // one d_endA partial per warp of the K4 backward
    lo.k4_nblk = (int)((P * N / kK4Vec + kK4Threads - 1) / kK4Threads) * (kK4Threads / 32);
    lo.dD_per = tc ? tc_dD_per(d.chunk_len) : (int)(Q / kMainRows);
    lo.nslice = tc ? tc_group_slices(d) : 1;
    lo.nslice_cb = tc ? tc_dcb_slices(d) : 1;
    lo.nslice_k5 = tc ? tc_k5_slices(d) : 1;
    lo.nslice_k3 = tc ? tc_k3_slices(d) : 1;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off += align_up(bytes); return o; };
    lo.status = take(sizeof(int) * kStatusWords);
    // the segmented state passing's ticket counter and flags follow the status
    // words, so that one memset clears both
    const size_t sync_ints = k4_seg_sync_ints(b, H, P, N, n, !tc);
    lo.k4s_sync = sync_ints ? take(sizeof(int) * sync_ints) : 0;
    lo.clear = off;
    if (sync_ints) {
        const K4SegGeom g = k4_seg_geom(b, H, P, N, n, !tc);
        const size_t ent = (size_t)kK4Threads * kK4Vec;
        lo.k4s_agg = take(4 * (size_t)g.pairs * g.K * ent);
        lo.k4s_carry = take(4 * (size_t)g.pairs * g.KG * ent);
        lo.k4s_dec = take(4 * (size_t)g.pairs * g.K);
    }
    lo.cumA = take(4 * tok);
    lo.endA = take(4 * b * H * n);
    // CB: fp32 on the CUDA-core path; bf16 CB and CB^T on the tensor-core path, where
    // only the backward stores them (the forward's K5 computes CB itself)
    lo.CB = (tc && !backward) ? 0 : take(4 * b * n * G * Q * Q);
    // chunk states: fp32 on the CUDA-core path, bf16 only on the tensor-core path
    lo.states = tc ? 0 : take(4 * nst);
    lo.states_bf = tc ? take(2 * nst) : 0;
    if (backward) {
        lo.dstates = tc ? 0 : take(4 * nst);
        lo.dstates_bf = tc ? take(2 * nst) : 0;
        lo.dcum_blue = take(4 * tok);
        lo.dcum_main = take(4 * tok);
        lo.d_delta = take(4 * tok);
        lo.ddt_main = take(4 * tok);
        lo.d_endA_part = take(4 * b * H * n * lo.k4_nblk);
        lo.dD_part = take(4 * b * n * H * lo.dD_per);
        lo.dA_part = take(4 * b * H * n);
        lo.d_cb = take(4 * (size_t)lo.nslice_cb * b * n * G * Q * Q);
        lo.dBC_part = tc ? take(4 * (size_t)lo.nslice * 2 * b * n * G * Q * N) : 0;
        // summed d_cb in bf16 and one arrival counter per 128 x 128 block on or below the diagonal
        lo.d_cb_bf = tc ? take(2 * b * n * G * Q * Q) : 0;
        lo.n_count = tc ? (int)(b * n * G * ((Q / 128) * (Q / 128 + 1) / 2)) : 0;
        lo.cb_count = tc ? take(4 * (size_t)lo.n_count) : 0;
        lo.fin_count = take(4 * H);
    }
    lo.total = off;
    return lo;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

ssd_status validate_dims(const ssd_dims *d, ssd_dtype dt) {
    if (!d) return fail(SSD_ERR_INVALID_ARG, "dims is NULL");
    if (dt != SSD_F32 && dt != SSD_BF16) return fail(SSD_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
    if (d->reserved != 0) return fail(SSD_ERR_INVALID_ARG, "dims.reserved must be 0");
    if (d->flags & ~(uint32_t)(SSD_FLAG_SIMT | SSD_FLAG_CHECK_FINITE | SSD_FLAG_SPLIT_SCAN))
        return fail(SSD_ERR_INVALID_ARG, "unknown flags 0x%x", d->flags);
    if (d->batch < 1 || d->seqlen < 1 || d->nheads < 1 || d->headdim < 1 || d->dstate < 1 ||
        d->ngroups < 1 || d->chunk_len < 1)
        return fail(SSD_ERR_INVALID_ARG, "every dimension must be >= 1");
    if (d->nheads % d->ngroups != 0)
        return fail(SSD_ERR_INVALID_ARG, "nheads (%lld) must be a multiple of ngroups (%lld)",
                    (long long)d->nheads, (long long)d->ngroups);
    const int64_t q = d->chunk_len;
    if (!(q == 16 || q == 32 || q == 64 || q == 128 || q == 256))
        return fail(SSD_ERR_UNSUPPORTED, "chunk_len %lld not in {16,32,64,128,256}", (long long)q);
    if (d->headdim > 128 || d->headdim % 4 != 0)
        return fail(SSD_ERR_UNSUPPORTED, "headdim %lld: need a multiple of 4 <= 128", (long long)d->headdim);
    if (d->dstate > 256 || d->dstate % 4 != 0)
        return fail(SSD_ERR_UNSUPPORTED, "dstate %lld: need a multiple of 4 <= 256", (long long)d->dstate);
    // index and grid limits
    const int64_t n = (d->seqlen + q - 1) / q;
    const double tok = (double)d->batch * (double)(n * q) * (double)d->nheads;
    if (tok * (double)d->headdim > 4.0e15 || (double)d->batch * n * d->nheads > 2.0e9 ||
        d->seqlen > (1LL << 30) || d->nheads > (1LL << 20))
        return fail(SSD_ERR_UNSUPPORTED, "problem too large");
    return SSD_OK;
}

Params base_params(const ssd_dims &d, const Layout &lo, void *ws) {
    Params p;
    memset(&p, 0, sizeof(p));
    p.b = (int)d.batch;
    p.L = (int)d.seqlen;
    p.H = (int)d.nheads;
    p.P = (int)d.headdim;
    p.N = (int)d.dstate;
    p.G = (int)d.ngroups;
    p.Q = (int)d.chunk_len;
    p.n = (int)((d.seqlen + d.chunk_len - 1) / d.chunk_len);
    p.hpg = p.H / p.G;
    char *w = (char *)ws;
    auto f = [&](size_t off) { return (float *)(w + off); };
    p.status = (int *)(w + lo.status);
    p.cumA = f(lo.cumA);
    p.endA = f(lo.endA);
    if (lo.CB) {
        p.CB = f(lo.CB);
        p.CBh = (bf16 *)(w + lo.CB);
        p.CBt = p.CBh + (size_t)p.b * p.n * p.G * p.Q * p.Q;
    }
    p.k4s_sync = lo.k4s_sync ? (int *)(w + lo.k4s_sync) : nullptr;
    p.k4s_agg = lo.k4s_agg ? f(lo.k4s_agg) : nullptr;
    p.k4s_carry = lo.k4s_carry ? f(lo.k4s_carry) : nullptr;
    p.k4s_dec = lo.k4s_dec ? f(lo.k4s_dec) : nullptr;
    p.states = lo.states ? f(lo.states) : nullptr;
    p.states_bf = lo.states_bf ? (bf16 *)(w + lo.states_bf) : nullptr;
    if (lo.dcum_blue) {  // backward layout
        p.dstates = lo.dstates ? f(lo.dstates) : nullptr;
        p.dstates_bf = lo.dstates_bf ? (bf16 *)(w + lo.dstates_bf) : nullptr;
        p.dcum_blue = f(lo.dcum_blue);
        p.dcum_main = f(lo.dcum_main);
        p.d_delta = f(lo.d_delta);
        p.ddt_main = f(lo.ddt_main);
        p.d_endA_part = f(lo.d_endA_part);
        p.dD_part = f(lo.dD_part);
        p.dA_part = f(lo.dA_part);
        p.d_cb = f(lo.d_cb);
        p.dBC_part = lo.dBC_part ? f(lo.dBC_part) : nullptr;
        p.d_cb_bf = lo.d_cb_bf ? (bf16 *)(w + lo.d_cb_bf) : nullptr;
        p.cb_count = lo.cb_count ? (int *)(w + lo.cb_count) : nullptr;
        p.fin_count = lo.fin_count ? (int *)(w + lo.fin_count) : nullptr;
        p.n_count = lo.n_count;
    }
    p.k4_nblk = lo.k4_nblk;
    p.dD_per = lo.dD_per;
    p.nslice = lo.nslice;
    p.nslice_cb = lo.nslice_cb;
    p.nslice_k5 = lo.nslice_k5;
    p.nslice_k3 = lo.nslice_k3;
    return p;
}

#define SSD_TRY(expr)                                                                     \
    do {                                                                                  \
        cudaError_t e_ = (expr);                                                          \
        if (e_ != cudaSuccess)                                                            \
            return fail(SSD_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_));          \
    } while (0)

#define SSD_LAUNCH(name, expr, nk)                                                        \
    do {                                                                                  \
        SSD_TRY(mark_start(name, s));                                                     \
        g_launches += (nk) - 1;                                                           \
        SSD_TRY(expr);                                                                    \
        SSD_TRY(mark_end(s));                                                             \
    } while (0)

template <typename T>
ssd_status run_forward_chain(const Params &p, const ssd_dims &d, bool tc, bool write_final, cudaStream_t s,
                             SideStream *sd) {
    if (tc) {
        if (use_fused_scan(p, d) && sd && overlap_scan(p)) {
            // backward with a small scan grid: K1 first, so that the side chain (K2, then
            // the caller's G1, which reads cumA but no chunk state) runs on the SMs the
            // scan leaves idle; the scan then reads cumA instead of computing it
            SSD_LAUNCH("k1_chunk_cumsum", launch_k1_cumsum(p, s), 1);
            SSD_TRY(cudaEventRecord(sd->fork, s));
            SSD_TRY(cudaStreamWaitEvent(sd->st, sd->fork, 0));
            const cudaStream_t side = side_stream_for(sd, s);
            {
                cudaStream_t s = side;
                SSD_LAUNCH("k2_cb_tc", launch_tc_k2(p, s), 1);
            }
            SSD_TRY(cudaEventRecord(sd->join, sd->st));
            Params q = p;
            q.cumA_given = 1;
            SSD_LAUNCH("state_scan_tc", launch_tc_state_scan(q, write_final, s), 1);
            return SSD_OK;
        }
        if (use_fused_scan(p, d)) {
            // K1, K3 and K4 in one pass per (b, h) chain: the intra-chunk states stay on chip
            SSD_LAUNCH("state_scan_tc", launch_tc_state_scan(p, write_final, s), 1);
        } else {
            SSD_LAUNCH("k1_chunk_cumsum", launch_k1_cumsum(p, s), 1);
            SSD_LAUNCH("k3_state_tc", launch_tc_k3(p, s), 1);
        }
        if (sd) {
            // K2 (CB and CB^T for the ORANGE backward) on the side stream, forked once
            // the chunk states are enqueued; the caller joins before the first reader
            SSD_TRY(cudaEventRecord(sd->fork, s));
            SSD_TRY(cudaStreamWaitEvent(sd->st, sd->fork, 0));
            const cudaStream_t side = side_stream_for(sd, s);
            {
                cudaStream_t s = side;
                SSD_LAUNCH("k2_cb_tc", launch_tc_k2(p, s), 1);
            }
            SSD_TRY(cudaEventRecord(sd->join, sd->st));
        }
        if (!use_fused_scan(p, d)) SSD_LAUNCH("k4_state_passing", launch_k4_state_passing(p, write_final, s), 1);
        return SSD_OK;
    }
    SSD_LAUNCH("k1_chunk_cumsum", launch_k1_cumsum(p, s), 1);
    SSD_LAUNCH("k2_cb_simt", launch_simt_k2<T>(p, s), 1);
    SSD_LAUNCH("k3_state_simt", launch_simt_k3<T>(p, s), 1);
    SSD_LAUNCH("k4_state_passing", launch_k4_state_passing(p, write_final, s), 1);
    return SSD_OK;
}

// Chunk ranges per (b, h) of the state-moment kernel (one CTA per SM): the
// count that minimises waves x (chunks per range + the CTA's fixed cost, about
// two chunks), fewest ranges on ties.
int moment_ranges(const ssd_dims &d) {
    const long long bh = d.batch * d.nheads, n = (d.seqlen + 127) / 128;
    long long best = 1, best_cost = -1;
    for (long long r = 1; r <= n; ++r) {
        const long long cost = ((bh * r + 151) / 152) * ((n + r - 1) / r + 2);
        if (best_cost < 0 || cost < best_cost) {
            best = r;
            best_cost = cost;
        }
    }
    return (int)best;
}

struct MomentLayout {
    ssd_dims d;  // the caller's dims at chunk 128
    Layout lo;   // the forward's workspace at chunk 128
    size_t A, m1, total;
    int ranges;
};

MomentLayout moment_layout(const ssd_dims &dims, ssd_dtype dt) {
    MomentLayout m;
    m.d = dims;
    m.d.chunk_len = 128;
    m.lo = make_layout(m.d, dt, false);
    m.ranges = moment_ranges(m.d);
    const size_t bhn = (size_t)dims.batch * dims.nheads * dims.dstate;
    m.A = m.lo.total;
    m.m1 = m.A + align_up(4 * (size_t)m.ranges * bhn * dims.dstate);
    m.total = m.m1 + align_up(4 * (size_t)m.ranges * bhn);
    return m;
}

ssd_status moments_supported(const ssd_dims *d, ssd_dtype dt) {
    ssd_status st = validate_dims(d, dt);
    if (st != SSD_OK) return st;
    if (dt != SSD_BF16 || (d->flags & SSD_FLAG_SIMT) || !tc_supported(d->headdim, d->dstate, 128))
        return fail(SSD_ERR_UNSUPPORTED, "state moments run on the tensor-core path: SSD_BF16, headdim 64, dstate 128");
    return SSD_OK;
}

// The SSD_FLAG_CHECK_FINITE regions shared by both calls: cumA, endA and the
// chunk states (every element written by K1 / K3 / K4 on both paths).
void add_intermediates(CheckList &l, const Params &p) {
    const size_t nst = (size_t)p.b * p.n * p.H * p.P * p.N;
    l.r[l.n++] = {p.cumA, (size_t)p.b * p.H * p.n * p.Q, 0};
    l.r[l.n++] = {p.endA, (size_t)p.b * p.H * p.n, 0};
    if (p.states) l.r[l.n++] = {p.states, nst, 0};
    if (p.states_bf) l.r[l.n++] = {p.states_bf, nst, 1};
}

}  // namespace

void record_error(const char *msg) { snprintf(g_last_error, sizeof(g_last_error), "%s", msg); }

ssd_status read_status_words(const void *words, cudaStream_t s) {
    int v[kStatusWords] = {0, 0, 0, 0};
    SSD_TRY(cudaMemcpyAsync(v, words, sizeof(v), cudaMemcpyDeviceToHost, s));
    SSD_TRY(cudaStreamSynchronize(s));
    if (v[kStatusCode] == SSD_ERR_TIMEOUT) return fail(SSD_ERR_TIMEOUT, "a device-side wait gave up");
    if (v[kStatusCode] != SSD_OK) return fail(SSD_ERR_CUDA, "unexpected device status %d", v[kStatusCode]);
    if (v[kStatusNonFinite] > 0)
        return fail(SSD_ERR_NONFINITE, "%d non-finite values in the call's outputs or intermediates",
                    v[kStatusNonFinite]);
    if (v[kStatusValidLen] > 0)
        return fail(SSD_ERR_INVALID_ARG, "%d valid_len entries outside [0, seqlen] were clamped",
                    v[kStatusValidLen]);
    return SSD_OK;
}

}  // namespace ssd

using namespace ssd;

extern "C" {

int ssd_version(void) { return 10000; }

const char *ssd_last_error(void) { return g_last_error; }

const char *ssd_status_str(ssd_status st) {
    switch (st) {
        case SSD_OK: return "ok";
        case SSD_ERR_INVALID_ARG: return "invalid argument";
        case SSD_ERR_UNSUPPORTED: return "unsupported shape";
        case SSD_ERR_WORKSPACE: return "workspace too small";
        case SSD_ERR_CUDA: return "CUDA error";
        case SSD_ERR_TIMEOUT: return "device-side wait timed out";
        case SSD_ERR_NONFINITE: return "non-finite values found";
    }
    return "unknown status";
}

ssd_status ssd_supported(const ssd_dims *dims, ssd_dtype dtype) {
    g_last_error[0] = 0;
    return validate_dims(dims, dtype);
}

size_t ssd_workspace_bytes(const ssd_dims *dims, ssd_dtype dtype, int backward) {
    if (validate_dims(dims, dtype) != SSD_OK) return 0;
    return make_layout(*dims, dtype, backward != 0).total;
}

ssd_status ssd_forward(const ssd_dims *dims, ssd_dtype dtype, const void *x, const float *dt,
                       const float *A, const void *B, const void *C, const float *D,
                       const float *init_state, const int32_t *valid_len, void *y,
                       float *final_state, void *workspace, size_t workspace_bytes, void *stream) {
    g_last_error[0] = 0;
    ssd_status st = validate_dims(dims, dtype);
    if (st != SSD_OK) return st;
    const void *req[] = {x, dt, A, B, C, D, y, workspace};
    const char *names[] = {"x", "dt", "A", "B", "C", "D", "y", "workspace"};
    for (int i = 0; i < 8; ++i) {
        if (!req[i]) return fail(SSD_ERR_INVALID_ARG, "%s is NULL", names[i]);
        if (!aligned16(req[i])) return fail(SSD_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    }
    if ((init_state && !aligned16(init_state)) || (final_state && !aligned16(final_state)))
        return fail(SSD_ERR_INVALID_ARG, "state pointers must be 16-byte aligned");
    const Layout lo = make_layout(*dims, dtype, false);
    if (workspace_bytes < lo.total)
        return fail(SSD_ERR_WORKSPACE, "workspace %zu < required %zu", workspace_bytes, lo.total);
    const bool tc = use_tensor_cores(*dims, dtype);
    Params p = base_params(*dims, lo, workspace);
    p.x = x; p.dt = dt; p.A = A; p.B = B; p.C = C; p.D = D; p.init = init_state;
    p.valid_len = valid_len; p.y = y; p.final_state = final_state;
    cudaStream_t s = (cudaStream_t)stream;
    g_launches = 0;
    SSD_TRY(cudaMemsetAsync(workspace, 0, lo.clear, s));  // status words and K4 sync
    if (dtype == SSD_F32) {
        st = run_forward_chain<float>(p, *dims, false, true, s, nullptr);
        if (st != SSD_OK) return st;
        SSD_LAUNCH("k5_scan_simt", launch_simt_k5<float>(p, s), 1);
    } else if (tc) {
        // on the caller's stream: the chunk states (one fused scan per (b, h) chain,
        // or K1, K3, K4), then K5 with K2 computed inside it
        st = run_forward_chain<bf16>(p, *dims, true, true, s, nullptr);
        if (st != SSD_OK) return st;
        SSD_LAUNCH("k5_scan_tc", launch_tc_k5(p, s), 1);
    } else {
        st = run_forward_chain<bf16>(p, *dims, false, true, s, nullptr);
        if (st != SSD_OK) return st;
        SSD_LAUNCH("k5_scan_simt", launch_simt_k5<bf16>(p, s), 1);
    }
    if (dims->flags & SSD_FLAG_CHECK_FINITE) {
        const size_t tokens = (size_t)p.b * p.L, xe = tokens * p.H * p.P;
        const int bf = dtype == SSD_BF16;
        CheckList l;
        l.n = 0;
        l.r[l.n++] = {y, xe, bf};
        if (final_state) l.r[l.n++] = {final_state, (size_t)p.b * p.H * p.P * p.N, 0};
        add_intermediates(l, p);
        SSD_LAUNCH("check_finite", launch_check_finite(l, p.status + kStatusNonFinite, s), 1);
    }
    return SSD_OK;
}

ssd_status ssd_backward(const ssd_dims *dims, ssd_dtype dtype, const void *x, const float *dt,
                        const float *A, const void *B, const void *C, const float *D,
                        const float *init_state, const int32_t *valid_len, const void *dy,
                        const float *d_final_state, void *dx, float *ddt, float *dA, void *dB,
                        void *dC, float *dD, float *d_init_state, void *workspace,
                        size_t workspace_bytes, void *stream) {
    g_last_error[0] = 0;
    ssd_status st = validate_dims(dims, dtype);
    if (st != SSD_OK) return st;
    const void *req[] = {x, dt, A, B, C, D, dy, dx, ddt, dA, dB, dC, dD, workspace};
    const char *names[] = {"x", "dt", "A", "B", "C", "D", "dy", "dx", "ddt", "dA", "dB", "dC",
                           "dD", "workspace"};
    for (int i = 0; i < 14; ++i) {
        if (!req[i]) return fail(SSD_ERR_INVALID_ARG, "%s is NULL", names[i]);
        if (!aligned16(req[i])) return fail(SSD_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    }
    if ((init_state && !aligned16(init_state)) || (d_final_state && !aligned16(d_final_state)) ||
        (d_init_state && !aligned16(d_init_state)))
        return fail(SSD_ERR_INVALID_ARG, "state pointers must be 16-byte aligned");
    const Layout lo = make_layout(*dims, dtype, true);
    if (workspace_bytes < lo.total)
        return fail(SSD_ERR_WORKSPACE, "workspace %zu < required %zu", workspace_bytes, lo.total);
    const bool tc = use_tensor_cores(*dims, dtype);
    Params p = base_params(*dims, lo, workspace);
    p.x = x; p.dt = dt; p.A = A; p.B = B; p.C = C; p.D = D; p.init = init_state;
    p.valid_len = valid_len; p.dy = dy; p.d_final = d_final_state; p.dx = dx; p.ddt = ddt;
    p.dA = dA; p.dB = dB; p.dC = dC; p.dD = dD; p.d_init = d_init_state;
    cudaStream_t s = (cudaStream_t)stream;
    g_launches = 0;
    SSD_TRY(cudaMemsetAsync(workspace, 0, lo.clear, s));  // status words and K4 sync
    if (dtype == SSD_F32) {
        st = run_forward_chain<float>(p, *dims, false, false, s, nullptr);
        if (st != SSD_OK) return st;
        SSD_LAUNCH("bwd_blue_simt", launch_simt_bwd_blue<float>(p, s), 2);
        SSD_LAUNCH("bwd_k4_state_passing", launch_bwd_k4(p, s), 1);
        SSD_LAUNCH("bwd_main_simt", launch_simt_bwd_main<float>(p, s), 1);
        SSD_LAUNCH("bwd_group_simt", launch_simt_bwd_group<float>(p, s), 2);
        SSD_LAUNCH("bwd_k1_chunk_cumsum", launch_bwd_k1(p, s), 1);
    } else {
        SideStream *sd = nullptr;
        std::unique_lock<std::mutex> lock;
        if (tc) {
            SSD_TRY(side_stream(s, &sd));
            lock = std::unique_lock<std::mutex>(sd->mu);  // orders calls sharing this caller stream
        }
        st = run_forward_chain<bf16>(p, *dims, tc, false, s, sd);
        if (st != SSD_OK) return st;
        if (tc) {
            // Two chains from here on.  The group kernels (G1: d_cb; G2: dB, dC partials;
            // G3: their sum) read only the leaves, cumA, the chunk states and d_intra, and
            // nothing else reads what they write: they run on the side stream (G1 right
            // after K2 -- with a small fused-scan grid both follow K1 and run beside the scan, since
            // G1 reads cumA but no chunk state -- G2 once the K4 backward has written
            // d_intra) and fill the SMs that the per-head chain on the caller's stream
            // (scan, BLUE, K4 backward, ORANGE, K3 backward, K1 backward) leaves idle.
            // The caller's stream joins at the end.
            const cudaStream_t side = side_stream_for(sd, s);
            {
                cudaStream_t s = side;
                SSD_LAUNCH("bwd_dcb_tc", launch_tc_bwd_dcb(p, s), 1);
            }
            SSD_LAUNCH("bwd_blue_tc", launch_tc_bwd_blue(p, s), 1);
            SSD_LAUNCH("bwd_k4_state_passing", launch_bwd_k4(p, s), 1);
            SSD_TRY(cudaEventRecord(sd->fork, s));  // d_intra
            SSD_TRY(cudaStreamWaitEvent(sd->st, sd->fork, 0));
            {
                cudaStream_t s = side;
                SSD_LAUNCH("bwd_dbc_tc", launch_tc_bwd_dbc(p, s), 1);
                SSD_LAUNCH("bwd_dbc_reduce_tc", launch_tc_bwd_dbc_reduce(p, s), 1);
            }
            SSD_TRY(cudaEventRecord(sd->aux, sd->st));
            SSD_TRY(cudaStreamWaitEvent(s, sd->join, 0));  // CB^T
            SSD_LAUNCH("bwd_orange_tc", launch_tc_bwd_orange(p, s), 1);
            SSD_LAUNCH("bwd_k3_tc", launch_tc_bwd_k3(p, s), 1);
            SSD_LAUNCH("bwd_k1_chunk_cumsum", launch_bwd_k1(p, s), 1);
            SSD_TRY(cudaStreamWaitEvent(s, sd->aux, 0));  // dB, dC
        } else {
            SSD_LAUNCH("bwd_blue_simt", launch_simt_bwd_blue<bf16>(p, s), 2);
            SSD_LAUNCH("bwd_k4_state_passing", launch_bwd_k4(p, s), 1);
            SSD_LAUNCH("bwd_main_simt", launch_simt_bwd_main<bf16>(p, s), 1);
            SSD_LAUNCH("bwd_group_simt", launch_simt_bwd_group<bf16>(p, s), 2);
            SSD_LAUNCH("bwd_k1_chunk_cumsum", launch_bwd_k1(p, s), 1);
        }
    }
    if (dims->flags & SSD_FLAG_CHECK_FINITE) {
        const size_t tokens = (size_t)p.b * p.L, xe = tokens * p.H * p.P, bce = tokens * p.G * p.N;
        const size_t nst = (size_t)p.b * p.n * p.H * p.P * p.N;
        const int bf = dtype == SSD_BF16;
        CheckList l;
        l.n = 0;
        l.r[l.n++] = {dx, xe, bf};
        l.r[l.n++] = {ddt, (size_t)p.b * p.H * p.L, 0};
        l.r[l.n++] = {dA, (size_t)p.H, 0};
        l.r[l.n++] = {dB, bce, bf};
        l.r[l.n++] = {dC, bce, bf};
        l.r[l.n++] = {dD, (size_t)p.H, 0};
        if (d_init_state) l.r[l.n++] = {d_init_state, (size_t)p.b * p.H * p.P * p.N, 0};
        add_intermediates(l, p);
        if (p.dstates) l.r[l.n++] = {p.dstates, nst, 0};
        if (p.dstates_bf) l.r[l.n++] = {p.dstates_bf, nst, 1};
        SSD_LAUNCH("check_finite", launch_check_finite(l, p.status + kStatusNonFinite, s), 1);
    }
    return SSD_OK;
}

size_t ssd_moments_workspace_bytes(const ssd_dims *dims, ssd_dtype dtype) {
    if (moments_supported(dims, dtype) != SSD_OK) return 0;
    return moment_layout(*dims, dtype).total;
}

ssd_status ssd_state_moments(const ssd_dims *dims, ssd_dtype dtype, const void *x, const float *dt,
                             const float *A, const void *B, const float *init_state,
                             const int32_t *valid_len, float *m2, float *m1, int64_t *count,
                             void *workspace, size_t workspace_bytes, void *stream) {
    g_last_error[0] = 0;
    ssd_status st = moments_supported(dims, dtype);
    if (st != SSD_OK) return st;
    const void *req[] = {x, dt, A, B, m2, m1, workspace};
    const char *names[] = {"x", "dt", "A", "B", "m2", "m1", "workspace"};
    for (int i = 0; i < 7; ++i) {
        if (!req[i]) return fail(SSD_ERR_INVALID_ARG, "%s is NULL", names[i]);
        if (!aligned16(req[i])) return fail(SSD_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    }
    if ((init_state && !aligned16(init_state)) || (count && ((uintptr_t)count & 7u)))
        return fail(SSD_ERR_INVALID_ARG, "init_state must be 16-byte and count 8-byte aligned");
    const MomentLayout ml = moment_layout(*dims, dtype);
    if (workspace_bytes < ml.total)
        return fail(SSD_ERR_WORKSPACE, "workspace %zu < required %zu", workspace_bytes, ml.total);
    Params p = base_params(ml.d, ml.lo, workspace);
    p.x = x; p.dt = dt; p.A = A; p.B = B; p.init = init_state; p.valid_len = valid_len;
    p.mom_A = (float *)((char *)workspace + ml.A);
    p.mom_m1 = (float *)((char *)workspace + ml.m1);
    p.mom_ranges = ml.ranges;
    cudaStream_t s = (cudaStream_t)stream;
    g_launches = 0;
    SSD_TRY(cudaMemsetAsync(workspace, 0, ml.lo.clear, s));  // status words and K4 sync
    // the chunk-input states at chunk 128 (fused scan or K1 + K3 + K4), then the moments
    st = run_forward_chain<bf16>(p, ml.d, true, false, s, nullptr);
    if (st != SSD_OK) return st;
    SSD_LAUNCH("moments_tc", launch_tc_moments(p, s), 1);
    SSD_LAUNCH("moments_reduce", launch_moments_reduce(p, m2, m1, count, s), 1);
    if (dims->flags & SSD_FLAG_CHECK_FINITE) {
        CheckList l;
        l.n = 0;
        l.r[l.n++] = {m2, (size_t)p.b * p.H * p.N * p.N, 0};
        l.r[l.n++] = {m1, (size_t)p.b * p.H * p.N, 0};
        add_intermediates(l, p);
        SSD_LAUNCH("check_finite", launch_check_finite(l, p.status + kStatusNonFinite, s), 1);
    }
    return SSD_OK;
}

ssd_status ssd_state_pr(const float *m2, const float *m1, const int64_t *count, int64_t batch,
                        int64_t nheads, int64_t dstate, int center, int pairing, int64_t num,
                        int pool_batch, float *pr, float *trace, void *stream) {
    g_last_error[0] = 0;
    if (!m2 || !m1 || !count || !pr) return fail(SSD_ERR_INVALID_ARG, "m2, m1, count and pr are required");
    if (batch < 1 || nheads < 1 || dstate < 1) return fail(SSD_ERR_INVALID_ARG, "every dimension must be >= 1");
    if (dstate > 224) return fail(SSD_ERR_UNSUPPORTED, "dstate %lld above 224", (long long)dstate);
    if (batch * nheads > (1LL << 30)) return fail(SSD_ERR_UNSUPPORTED, "problem too large");
    const int64_t N = dstate;
    switch (pairing) {
        case SSD_PAIR_REAL: num = 0; break;
        case SSD_PAIR_COMPLEX_INTERLEAVED:
            if (num < 1 || 2 * num > N) return fail(SSD_ERR_INVALID_ARG, "interleaved pairing exceeds dstate");
            break;
        case SSD_PAIR_COMPLEX_HALF_HALF:
            if (num < 1 || num > N / 2) return fail(SSD_ERR_INVALID_ARG, "half-and-half pairing exceeds dstate / 2");
            break;
        case SSD_PAIR_QUATERNION:
            if (num < 1 || 4 * num > N) return fail(SSD_ERR_INVALID_ARG, "quaternion pairing exceeds dstate");
            break;
        default: return fail(SSD_ERR_INVALID_ARG, "unknown pairing %d", pairing);
    }
    cudaStream_t s = (cudaStream_t)stream;
    SSD_TRY(launch_state_pr(m2, m1, count, (int)batch, (int)nheads, (int)N, center ? 1 : 0, pairing, (int)num,
                            pool_batch ? 1 : 0, pr, trace, s));
    return SSD_OK;
}

ssd_status ssd_wait_selftest(void *workspace, size_t workspace_bytes, uint32_t limit_us, int arrive,
                             void *stream) {
    g_last_error[0] = 0;
    if (!workspace || workspace_bytes < sizeof(int) * kStatusWords) return fail(SSD_ERR_INVALID_ARG, "bad workspace");
    if (limit_us < 1 || limit_us > 2000000) return fail(SSD_ERR_INVALID_ARG, "limit_us must be in [1, 2000000]");
    if (arrive != 0 && arrive != 1) return fail(SSD_ERR_INVALID_ARG, "arrive must be 0 or 1");
    cudaStream_t s = (cudaStream_t)stream;
    SSD_TRY(cudaMemsetAsync(workspace, 0, sizeof(int) * kStatusWords, s));
    SSD_TRY(launch_wait_selftest((int *)workspace, 1000ull * limit_us, arrive, s));
    g_launches = 1;
    return SSD_OK;
}

int ssd_last_launch_count(void) { return g_launches; }

ssd_status ssd_profile_begin(void **events, int capacity) {
    g_last_error[0] = 0;
    if (!events || capacity < 2) return fail(SSD_ERR_INVALID_ARG, "need an array of >= 2 events");
    g_rec.ev = (cudaEvent_t *)events;
    g_rec.cap = capacity;
    g_rec.n = 0;
    return SSD_OK;
}

int ssd_profile_end(void) {
    const int n = g_rec.n;
    g_rec.ev = nullptr;
    g_rec.cap = 0;
    return n;
}

void ssd_profile_only(const char *name) {
    snprintf(g_rec_only, sizeof(g_rec_only), "%s", name ? name : "");
}

const char *ssd_profile_name(int i) {
    if (i < 0 || i >= 4096) return "";
    return g_rec.names[i];
}

ssd_status ssd_workspace_status(const void *workspace, size_t workspace_bytes, void *stream) {
    g_last_error[0] = 0;
    if (!workspace || workspace_bytes < sizeof(int) * kStatusWords)
        return fail(SSD_ERR_INVALID_ARG, "bad workspace");
    return read_status_words(workspace, (cudaStream_t)stream);
}

}  // extern "C"
