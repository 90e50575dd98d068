"""CPU oracle for the two Mamba-3 pieces on the pages -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The CUDA library never imports, links
or calls it, and it imports nothing from the CUDA package.  Everything is
NumPy in fp64, vectorised over the independent chains / tokens and looping
over the sequence where the method is a recurrence.

* Quaternion cumulative product (burn-mamba, ``mamba3/quat_scan/backward.rs``,
  module doc "Gradient math"): ``cum[t] = q_t (x) cum[t-1]`` with
  ``cum[-1] = init`` and (x) the Hamilton product, components ordered
  (w, x, y, z) as on the ``modules/state_moments.rs`` page (QuaternionBlocks).
  :func:`quat_cumprod_vjp` is the reverse-mode derivative of that recurrence,
  written from its definition (valid for every quaternion);
  :func:`quat_cumprod_backward_closed` restates the page's closed form
  (prefix product, reverse cumsum, two products), which the page states is
  exact for unit quaternions only.
* Same-step gamma correction (burn-mamba,
  ``mamba3/single_ssd/ssd/serial_recalculated/diag.rs``): per token t and head
  h, ``qk = C B^T`` over the state axis and ``y_diag = gamma * qk V`` over the
  MIMO axis; :func:`y_diag_vjp` is its chain rule.  Tokens are flattened: the
  page's [b, n, l] axes become one axis T.
"""
from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------- quaternions
def qmul(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Hamilton product of quaternion arrays [..., 4] (w, x, y, z)."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    aw, ax, ay, az = a[..., 0], a[..., 1], a[..., 2], a[..., 3]
    bw, bx, by, bz = b[..., 0], b[..., 1], b[..., 2], b[..., 3]
    return np.stack([
        aw * bw - ax * bx - ay * by - az * bz,
        aw * bx + ax * bw + ay * bz - az * by,
        aw * by - ax * bz + ay * bw + az * bx,
        aw * bz + ax * by - ay * bx + az * bw,
    ], axis=-1)


def qconj(a: np.ndarray) -> np.ndarray:
    """Conjugate: (w, -x, -y, -z)."""
    a = np.asarray(a, np.float64)
    return a * np.array([1.0, -1.0, -1.0, -1.0])


def quat_cumprod(q: np.ndarray, init: np.ndarray) -> np.ndarray:
    """cum[:, t] = q[:, t] (x) cum[:, t-1], cum[:, -1] = init.

    q [b, L, H, J, 4], init [b, H, J, 4] -> cum [b, L, H, J, 4] (fp64)."""
    q = np.asarray(q, np.float64)
    cur = np.asarray(init, np.float64).copy()
    out = np.empty_like(q)
    for t in range(q.shape[1]):
        cur = qmul(q[:, t], cur)
        out[:, t] = cur
    return out


def quat_cumprod_vjp(q: np.ndarray, init: np.ndarray, d_cum: np.ndarray):
    """Reverse mode of :func:`quat_cumprod` from its definition.

    For o = a (x) b and a cotangent g of o (real inner product of the four
    components), d a = g (x) conj(b) and d b = conj(a) (x) g (the product is
    bilinear).  Walking the recurrence backwards, the cotangent reaching
    cum[t] is G[t] = d_cum[t] + conj(q[t+1]) (x) G[t+1]; then
    d q[t] = G[t] (x) conj(cum[t-1]) and d init = conj(q[0]) (x) G[0].
    Returns (d_q [b, L, H, J, 4], d_init [b, H, J, 4])."""
    q = np.asarray(q, np.float64)
    init = np.asarray(init, np.float64)
    d_cum = np.asarray(d_cum, np.float64)
    cum = quat_cumprod(q, init)
    L = q.shape[1]
    d_q = np.empty_like(q)
    G = np.zeros_like(init)
    for t in range(L - 1, -1, -1):
        G = d_cum[:, t] + (qmul(qconj(q[:, t + 1]), G) if t + 1 < L else 0.0)
        prev = cum[:, t - 1] if t > 0 else init
        d_q[:, t] = qmul(G, qconj(prev))
    d_init = qmul(qconj(q[:, 0]), G) if L > 0 else np.zeros_like(init)
    return d_q, d_init


def quat_cumprod_backward_closed(q: np.ndarray, init: np.ndarray, d_cum: np.ndarray):
    """The page's closed-form backward, its steps in the page's order:
    P[t] = q[t] (x) ... (x) q[0] (prefix product without the carry);
    cum[t] = P[t] (x) init; S[t] = sum_{s >= t} conj(P[s]) (x) d_cum[s];
    G[t] = P[t] (x) S[t]; d_q[t] = G[t] (x) conj(cum[t-1]) (cum[-1] = init);
    d_init = S[0].  Equal to :func:`quat_cumprod_vjp` when every q[t] has unit
    norm."""
    q = np.asarray(q, np.float64)
    init = np.asarray(init, np.float64)
    d_cum = np.asarray(d_cum, np.float64)
    one = np.zeros_like(init)
    one[..., 0] = 1.0
    P = quat_cumprod(q, one)
    cum = qmul(P, init[:, None])
    terms = qmul(qconj(P), d_cum)
    S = np.flip(np.cumsum(np.flip(terms, axis=1), axis=1), axis=1)
    G = qmul(P, S)
    prev = np.concatenate([init[:, None], cum[:, :-1]], axis=1)
    d_q = qmul(G, qconj(prev))
    return d_q, S[:, 0]


# ---------------------------------------------------------------- gamma correction
def y_diag(V: np.ndarray, B: np.ndarray, C: np.ndarray, gamma: np.ndarray) -> np.ndarray:
    """y[t, o, h, p] = gamma[t, h] * sum_i qk[t, h, o, i] V[t, i, h, p],
    qk[t, h, o, i] = sum_r C[t, o, h, r] B[t, i, h, r].

    V [T, m, H, P], B and C [T, m, H, N], gamma [T, H] -> y [T, m, H, P]."""
    V, B, C, gamma = (np.asarray(a, np.float64) for a in (V, B, C, gamma))
    qk = np.einsum("tohr,tihr->thoi", C, B)
    return gamma[:, None, :, None] * np.einsum("thoi,tihp->tohp", qk, V)


def y_diag_siso(V, B, C, gamma):
    """The mimo_rank = 1 special case the page takes as its fast path: one
    scalar qk = C . B per (t, h), then y = gamma qk V."""
    V, B, C, gamma = (np.asarray(a, np.float64) for a in (V, B, C, gamma))
    qk = np.sum(C * B, axis=-1)  # [T, 1, H]
    return V * (qk * gamma[:, None, :])[..., None]


def y_diag_vjp(dY, V, B, C, gamma):
    """Chain rule of :func:`y_diag` for a cotangent dY [T, m, H, P]:
    d gamma = sum_{o, p} dY (qk V); with e = gamma dY:
    d V = qk^T e, d qk = e V^T, d C = d qk B, d B = d qk^T C.
    Returns (dV, dB, dC, d_gamma)."""
    dY, V, B, C, gamma = (np.asarray(a, np.float64) for a in (dY, V, B, C, gamma))
    qk = np.einsum("tohr,tihr->thoi", C, B)
    unweighted = np.einsum("thoi,tihp->tohp", qk, V)
    d_gamma = np.einsum("tohp,tohp->th", dY, unweighted)
    e = gamma[:, None, :, None] * dY
    dV = np.einsum("thoi,tohp->tihp", qk, e)
    dqk = np.einsum("tohp,tihp->thoi", e, V)
    dC = np.einsum("thoi,tihr->tohr", dqk, B)
    dB = np.einsum("thoi,tohr->tihr", dqk, C)
    return dV, dB, dC, d_gamma
