"""NumPy fp64 restatement of the pages' chunked SSD -- TEST INFRASTRUCTURE ONLY.

This is the *second* CPU implementation.  It follows the chunk-level structure
that burn-mamba's page "combined_backward.rs"
(``burn_mamba/mamba2/ssd/serial_recalculated/``) describes -- K1 chunk cumsum,
K2 C.B^T, K3 extended chunk state, K4 state passing, the BLUE and ORANGE
terms of the chunk scan, the skip term, and the recompute backward -- written
from the formulas in its comments, not from its code.  The serial C oracle is
the definition; this module exists to show that the pages' chunked formulas
reach the same numbers (chunked == serial) and to test the page's identities:

* reverse-cumsum form of the K1 backward ("SUM GRADIENT CONTRIBUTIONS + K1
  BACKWARD": suffix sum = total - shifted prefix sum),
* the ``out_x . dout - ddt . dt`` identity for the same-chunk d(cumA)
  (the ``d_da_local`` / ``d_dt_orange`` test-only fields of ``CombinedGrads``),
* ``d_da_blue[l] = sum_r dC_blue[l, r] C[l, r]`` (algebra of the BLUE block).

Readings where the page is silent (the forward of K1/K2/K4/K5 is not printed,
only recomputed): cumsum is inclusive; the causal mask keeps s <= t; A is used
as given (negative) with dA = dt*A; groups map head h to group h // (H/G);
tokens t >= valid_len are removed by zeroing dt, x, B, C, dy there and zeroing
every output and gradient there afterwards.
"""
from __future__ import annotations

import numpy as np


def _pad_and_mask(x, dt, B, C, dy, valid_len, Q):
    nb, L, H, P = x.shape
    n = -(-L // Q)
    Lp = n * Q
    V = np.full(nb, L, np.int64) if valid_len is None else np.clip(np.asarray(valid_len), 0, L)
    tmask = (np.arange(Lp)[None, :] < V[:, None])  # [b, Lp]

    def pad_t(a, axis):
        w = [(0, 0)] * a.ndim
        w[axis] = (0, Lp - L)
        return np.pad(a, w)

    xm = pad_t(x, 1) * tmask[:, :, None, None]
    dtm = pad_t(dt, 2) * tmask[:, None, :]
    Bm = pad_t(B, 1) * tmask[:, :, None, None]
    Cm = pad_t(C, 1) * tmask[:, :, None, None]
    dym = None if dy is None else pad_t(dy, 1) * tmask[:, :, None, None]
    return xm, dtm, Bm, Cm, dym, tmask, n, Lp


def _heads(Bg, H):
    """[b, L, G, N] -> per-head [b, L, H, N] (head h reads group h // (H/G))."""
    G = Bg.shape[2]
    return np.repeat(Bg, H // G, axis=2)


def forward_chunked(x, dt, A, B, C, D, init=None, valid_len=None, Q=16, return_parts=False):
    """Chunked five-kernel forward.  Returns (y, final[, parts])."""
    x, dt, A, B, C, D = (np.asarray(a, np.float64) for a in (x, dt, A, B, C, D))
    nb, L, H, P = x.shape
    N = B.shape[-1]
    xm, dtm, Bm, Cm, _, tmask, n, Lp = _pad_and_mask(x, dt, B, C, None, valid_len, Q)
    Bh, Ch = _heads(Bm, H), _heads(Cm, H)
    s0 = np.zeros((nb, H, P, N)) if init is None else np.asarray(init, np.float64)

    # chunked views: x [b,n,Q,H,P]; dt [b,H,n,Q]; B/C [b,n,Q,H,N]
    xc = xm.reshape(nb, n, Q, H, P)
    dtc = dtm.reshape(nb, H, n, Q)
    Bc = Bh.reshape(nb, n, Q, H, N)
    Cc = Ch.reshape(nb, n, Q, H, N)

    # K1: inclusive cumsum of dt*A within each chunk
    cumA = np.cumsum(dtc * A[None, :, None, None], axis=3)
    endA = cumA[..., -1]
    # K2: CB[b,n,h,t,s] = sum_r C[t,r] B[s,r]
    CB = np.einsum("bnthr,bnshr->bnhts", Cc, Bc)
    # K3 (extended): decay to chunk end, scale, zero-initial-state chunk-end state
    decay_end = np.exp(endA[..., None] - cumA)            # [b,H,n,Q]
    bbs = decay_end * dtc                                 # [b,H,n,Q]
    b_scaled = Bc * bbs.transpose(0, 2, 3, 1)[..., None]  # [b,n,Q,H,N]
    intra = np.einsum("bnlhp,bnlhr->bnhpr", xc, b_scaled)
    # K4: s_{i+1} = exp(endA_i) s_i + intra_i
    s_in = np.empty((nb, n, H, P, N))
    s = s0.copy()
    for i in range(n):
        s_in[:, i] = s
        s = np.exp(endA[:, :, i])[..., None, None] * s + intra[:, i]
    final = s
    # K5: BLUE + ORANGE + skip
    ecum = np.exp(cumA)                                    # [b,H,n,Q]
    blue = np.einsum("bnlhr,bnhpr->bnlhp", Cc, s_in) * ecum.transpose(0, 2, 3, 1)[..., None]
    diff = cumA[..., :, None] - cumA[..., None, :]        # [b,H,n,t,s]
    causal = np.tril(np.ones((Q, Q), bool))
    decay = np.where(causal, np.exp(np.where(causal, diff, 0.0)), 0.0)
    W = CB * decay.transpose(0, 2, 1, 3, 4) * dtc.transpose(0, 2, 1, 3)[:, :, :, None, :]
    orange = np.einsum("bnhts,bnshp->bnthp", W, xc)
    y = blue + orange + D[None, None, None, :, None] * xc
    y = y.reshape(nb, Lp, H, P)[:, :L] * tmask[:, :L, None, None]
    if not return_parts:
        return y, final
    parts = dict(cumA=cumA, endA=endA, CB=CB, intra=intra, s_in=s_in, decay_end=decay_end,
                 bbs=bbs, blue=blue.reshape(nb, Lp, H, P)[:, :L],
                 orange=orange.reshape(nb, Lp, H, P)[:, :L])
    return y, final, parts


def backward_chunked(x, dt, A, B, C, D, init, valid_len, dy, d_final=None, Q=16):
    """Recompute backward in the page's order.  Returns a dict of gradients plus
    the page's test-only fields and a few intermediates used by the identity
    tests (``d_da_local``, ``d_dt_orange``, ``d_da_blue``, ``dC_blue_h``,
    ``d_da_cumsum``, ``d_da``, ``d_da_suffix``)."""
    x, dt, A, B, C, D, dy = (np.asarray(a, np.float64) for a in (x, dt, A, B, C, D, dy))
    nb, L, H, P = x.shape
    N, G = B.shape[-1], B.shape[2]
    xm, dtm, Bm, Cm, dym, tmask, n, Lp = _pad_and_mask(x, dt, B, C, dy, valid_len, Q)
    Bh, Ch = _heads(Bm, H), _heads(Cm, H)
    s0 = np.zeros((nb, H, P, N)) if init is None else np.asarray(init, np.float64)
    dfin = np.zeros((nb, H, P, N)) if d_final is None else np.asarray(d_final, np.float64)

    xc = xm.reshape(nb, n, Q, H, P)
    dyc = dym.reshape(nb, n, Q, H, P)
    dtc = dtm.reshape(nb, H, n, Q)
    Bc = Bh.reshape(nb, n, Q, H, N)
    Cc = Ch.reshape(nb, n, Q, H, N)

    # ---- recompute K1..K4 from the leaves ----
    cumA = np.cumsum(dtc * A[None, :, None, None], axis=3)
    endA = cumA[..., -1]
    CB = np.einsum("bnthr,bnshr->bnhts", Cc, Bc)
    decay_end = np.exp(endA[..., None] - cumA)
    bbs = decay_end * dtc
    b_scaled = Bc * bbs.transpose(0, 2, 3, 1)[..., None]
    intra = np.einsum("bnlhp,bnlhr->bnhpr", xc, b_scaled)
    s_in = np.empty((nb, n, H, P, N))
    s = s0.copy()
    for i in range(n):
        s_in[:, i] = s
        s = np.exp(endA[:, :, i])[..., None, None] * s + intra[:, i]

    # ---- skip term ----
    dD = np.einsum("bnlhp,bnlhp->h", dyc, xc)
    dx_skip = dyc * D[None, None, None, :, None]

    # ---- reverse chunk loop: BLUE + ORANGE + K4 step ----
    causal = np.tril(np.ones((Q, Q), bool))
    dx_orange = np.zeros_like(xc)
    ddt_orange = np.zeros((nb, H, n, Q))
    dda_orange = np.zeros((nb, H, n, Q))
    dda_blue = np.zeros((nb, H, n, Q))
    dC_blue = np.zeros((nb, n, Q, H, N))
    d_cb = np.zeros((nb, n, H, Q, Q))
    d_intra = np.zeros((nb, n, H, P, N))
    d_endA = np.zeros((nb, H, n))
    d_run = dfin.copy()
    for i in reversed(range(n)):
        ca = cumA[:, :, i]                     # [b,H,Q]
        dti = dtc[:, :, i]                     # [b,H,Q]
        xi = xc[:, i].transpose(0, 2, 1, 3)    # [b,H,Q,P]
        dyi = dyc[:, i].transpose(0, 2, 1, 3)  # [b,H,Q,P]
        ci = Cc[:, i].transpose(0, 2, 1, 3)    # [b,H,Q,N]
        si = s_in[:, i]                        # [b,H,P,N]
        cbi = CB[:, i]                         # [b,H,Q,Q]
        # BLUE: blue[l,p] = exp(cumA[l]) sum_r C[l,r] s[p,r]
        d_ch = dyi * np.exp(ca)[..., None]
        d_sin = np.einsum("bhlr,bhlp->bhpr", ci, d_ch)
        dC_blue[:, i] = np.einsum("bhlp,bhpr->blhr", d_ch, si)
        ch = np.einsum("bhlr,bhpr->bhlp", ci, si)
        dda_blue[:, :, i] = np.sum(dyi * ch * np.exp(ca)[..., None], axis=3)
        # ORANGE: w[t,s] = CB[t,s] exp(cumA[t]-cumA[s]) dt[s] (s <= t)
        diff = ca[..., :, None] - ca[..., None, :]
        decay = np.where(causal, np.exp(np.where(causal, diff, 0.0)), 0.0)
        cb_decay = cbi * decay
        w = cb_decay * dti[..., None, :]
        dw = np.einsum("bhtp,bhsp->bhts", dyi, xi)
        dx_orange[:, i] = np.einsum("bhts,bhtp->bshp", w, dyi)
        dwm = np.where(causal, dw, 0.0)
        d_cb_decay = dwm * dti[..., None, :]
        ddt_orange[:, :, i] = np.sum(dwm * cb_decay, axis=2)
        d_cb[:, i] = d_cb_decay * decay
        d_diff = d_cb_decay * cbi * decay
        dda_orange[:, :, i] = np.sum(d_diff, axis=3) - np.sum(d_diff, axis=2)
        # K4 step: s_{i+1} = exp(endA_i) s_i + intra_i
        d_intra[:, i] = d_run
        dec = np.exp(endA[:, :, i])
        d_endA[:, :, i] = np.sum(d_run * si, axis=(2, 3)) * dec
        d_run = dec[..., None, None] * d_run + d_sin
    d_init = d_run

    # ---- K3 backward ----
    dx_k3 = np.einsum("bnhpr,bnlhr->bnlhp", d_intra, b_scaled)
    d_bs = np.einsum("bnlhp,bnhpr->bnlhr", xc, d_intra)
    dB_k3 = d_bs * bbs.transpose(0, 2, 3, 1)[..., None]
    d_bbs = np.sum(d_bs * Bc, axis=4).transpose(0, 3, 1, 2)   # [b,H,n,Q]
    d_fdecay = d_bbs * dtc
    ddt_k3 = d_bbs * decay_end
    d_delta = d_fdecay * decay_end
    dda_k3 = -d_delta
    dda_k3[..., -1] += np.sum(d_delta, axis=3)

    # ---- K2 backward ----
    dC_k2 = np.einsum("bnhts,bnshr->bnthr", d_cb, Bc)
    dB_k2 = np.einsum("bnhts,bnthr->bnshr", d_cb, Cc)

    # ---- sum + K1 backward ----
    dda_k4 = np.zeros((nb, H, n, Q))
    dda_k4[..., -1] = d_endA
    d_da_cumsum = dda_blue + dda_orange + dda_k3 + dda_k4
    total = np.sum(d_da_cumsum, axis=3, keepdims=True)
    prefix = np.cumsum(d_da_cumsum, axis=3)
    shifted = np.concatenate([np.zeros((nb, H, n, 1)), prefix[..., :-1]], axis=3)
    d_da = total - shifted
    d_da_suffix = np.flip(np.cumsum(np.flip(d_da_cumsum, 3), axis=3), 3)
    ddt_k1 = d_da * A[None, :, None, None]
    dA = np.sum(d_da * dtc, axis=(0, 2, 3))
    ddt = ddt_orange + ddt_k3 + ddt_k1
    dx = dx_skip + dx_k3 + dx_orange
    dBh = dB_k2 + dB_k3
    dCh = dC_k2 + dC_blue

    def to_tokens(a, last):  # [b,n,Q,H,last] -> [b,L,H,last] masked
        return a.reshape(nb, Lp, H, last)[:, :L] * tmask[:, :L, None, None]

    def to_groups(a):  # per-head [b,L,H,N] -> [b,L,G,N]
        return a.reshape(nb, L, G, H // G, N).sum(axis=3)

    tm3 = tmask[:, None, :L]
    return dict(
        dx=to_tokens(dx, P),
        ddt=ddt.reshape(nb, H, Lp)[:, :, :L] * tm3,
        dA=dA, dD=dD,
        dB=to_groups(to_tokens(dBh, N)),
        dC=to_groups(to_tokens(dCh, N)),
        d_init=d_init,
        # test-only fields named after the page's CombinedGrads
        d_da_local=(dda_blue + dda_orange).reshape(nb, H, Lp)[:, :, :L],
        d_dt_orange=ddt_orange.reshape(nb, H, Lp)[:, :, :L],
        d_da_blue=dda_blue, dC_blue_h=dC_blue,
        d_da_cumsum=d_da_cumsum, d_da=d_da, d_da_suffix=d_da_suffix,
    )
