"""Participation ratio of pooled state moments -- TEST INFRASTRUCTURE ONLY
(oracle package: only tests/, the package smoke check and the benchmark's CPU
baseline use it).

NumPy fp64 restatement of burn-mamba's ``modules/state_moments.rs``
(StateMoments::pr, ::pr_complex, ::trace), the steps in the page's order:
the covariance is the raw second moment over the sample count, optionally
centred by the sample mean; it is normalised by its trace (floored at the
smallest positive normal of fp32, the precision the page computes in) and the
ratio of the squared trace to the sum of squares (floored at 1e-12, the
denominator clamp the page names beside ``trace``) is returned.  The complex
and quaternionic forms treat the state axis as realified coordinates in the
page's layouts (interleaved pairs, half-and-half pairs, blocks of four w, x,
y, z) and take the sum of squares of the Hermitian moment.
"""
from __future__ import annotations

import numpy as np

MIN_POSITIVE_F32 = float(np.finfo(np.float32).tiny)
DIV_EPS = 1e-12

REAL, COMPLEX_INTERLEAVED, COMPLEX_HALF_HALF, QUATERNION_BLOCKS = 0, 1, 2, 3


def covariance(m2, m1, count, center):
    """Sigma per (batch, head): m2 / n, minus mu mu^T when centred (mu = m1 / n).
    count: per batch element (array [b]) or a scalar."""
    m2 = np.asarray(m2, np.float64)
    n = np.asarray(count, np.float64).reshape(-1, *([1] * (m2.ndim - 1)))
    sigma = m2 / n
    if center:
        mu = np.asarray(m1, np.float64) / n[..., 0]
        sigma = sigma - mu[..., :, None] * mu[..., None, :]
    return sigma


def _normalised(sigma):
    tr = np.trace(sigma, axis1=-2, axis2=-1)
    scale = np.maximum(tr, MIN_POSITIVE_F32)
    return sigma / scale[..., None, None]


def pr(m2, m1, count, center=False):
    """(tr S)^2 / tr(S^2) of the (centred) covariance S, per (batch, head)."""
    hat = _normalised(covariance(m2, m1, count, center))
    tr1 = np.trace(hat, axis1=-2, axis2=-1)
    tr2 = np.maximum(np.sum(hat * hat, axis=(-2, -1)), DIV_EPS)
    return tr1 * tr1 / tr2


def trace(m2, count):
    """tr(m2) / n: the mean squared state magnitude."""
    n = np.asarray(count, np.float64).reshape(-1, *([1] * (np.asarray(m2).ndim - 3)))
    return np.trace(np.asarray(m2, np.float64), axis1=-2, axis2=-1) / n


def pr_complex(m2, m1, count, pairing, num, center=False):
    """PR of the Hermitian moment for the pairing (REAL, COMPLEX_INTERLEAVED,
    COMPLEX_HALF_HALF with `num` pairs, QUATERNION_BLOCKS with `num` blocks)."""
    sigma = covariance(m2, m1, count, center)
    R = sigma.shape[-1]
    if pairing == REAL:
        return pr(m2, m1, count, center)
    if pairing == COMPLEX_INTERLEAVED:
        assert 0 < num and 2 * num <= R
        idx = [2 * a for a in range(num)] + [2 * a + 1 for a in range(num)] + list(range(2 * num, R))
        rotated = 2 * num
    elif pairing == COMPLEX_HALF_HALF:
        half = R // 2
        assert 0 < num <= half
        idx = list(range(num)) + [half + a for a in range(num)] + list(range(num, half)) + \
            list(range(half + num, R))
        rotated = 2 * num
    elif pairing == QUATERNION_BLOCKS:
        assert 0 < num and 4 * num <= R
        idx = list(range(R))
        rotated = 4 * num
    else:
        raise ValueError(pairing)
    idx = np.asarray(idx)
    sigma = sigma[..., idx, :][..., :, idx]
    hat = _normalised(sigma)
    tr1 = np.trace(hat, axis1=-2, axis2=-1)
    fro2 = lambda t: np.sum(t * t, axis=(-2, -1))
    if pairing == QUATERNION_BLOCKS:
        j = num
        q = hat[..., :4 * j, :4 * j].reshape(hat.shape[:-2] + (j, 4, j, 4))
        c = lambda a, b: q[..., :, a, :, b]
        w = c(0, 0) + c(1, 1) + c(2, 2) + c(3, 3)
        x = c(0, 1) - c(1, 0) - c(2, 3) + c(3, 2)
        y = c(0, 2) + c(1, 3) - c(2, 0) - c(3, 1)
        z = c(0, 3) - c(1, 2) + c(2, 1) - c(3, 0)
        tr2 = fro2(w) + fro2(x) + fro2(y) + fro2(z)
    else:
        npair = num
        xx = hat[..., :npair, :npair]
        yy = hat[..., npair:2 * npair, npair:2 * npair]
        xy = hat[..., :npair, npair:2 * npair]
        tr2 = fro2(xx + yy) + fro2(xy - np.swapaxes(xy, -1, -2))
    if rotated < R:
        tr2 = tr2 + 2.0 * fro2(hat[..., :rotated, rotated:]) + fro2(hat[..., rotated:, rotated:])
    tr2 = np.maximum(tr2, DIV_EPS)
    return tr1 * tr1 / tr2
