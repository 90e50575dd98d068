"""Pins of the Mamba-3 oracle (oracle/mamba3.py) against facts it does not
restate: the quaternion algebra's defining rules, rotation composition by an
independent library (scipy), rotations about one axis (angles add), central
finite differences of every gradient, brute-force loops on tiny inputs, and
the page's statement that its closed-form backward is exact for unit
quaternions (and, as a check that the test can fail, not otherwise)."""
import itertools

import numpy as np
import pytest

from oracle import mamba3 as m3

Rotation = pytest.importorskip("scipy.spatial.transform").Rotation

E = np.eye(4)  # 1, i, j, k as (w, x, y, z)
ONE, I, J, K = E


def rand_unit(rng, shape):
    q = rng.standard_normal(shape + (4,))
    return q / np.linalg.norm(q, axis=-1, keepdims=True)


# ---------------------------------------------------------------- the algebra
def test_hamilton_rules():
    assert np.allclose(m3.qmul(I, J), K) and np.allclose(m3.qmul(J, K), I) and np.allclose(m3.qmul(K, I), J)
    assert np.allclose(m3.qmul(J, I), -K)  # not commutative
    for u in (I, J, K):
        assert np.allclose(m3.qmul(u, u), -ONE)
    assert np.allclose(m3.qmul(m3.qmul(I, J), K), -ONE)  # ijk = -1


def test_norm_multiplies_and_conjugate():
    rng = np.random.default_rng(1)
    a, b = rng.standard_normal((2, 50, 4))
    assert np.allclose(np.linalg.norm(m3.qmul(a, b), axis=-1),
                       np.linalg.norm(a, axis=-1) * np.linalg.norm(b, axis=-1))
    n2 = np.sum(a * a, axis=-1)
    assert np.allclose(m3.qmul(a, m3.qconj(a)), n2[:, None] * ONE)


def test_product_composes_rotations_like_scipy():
    # for unit q, v -> q v conj(q) is the rotation R(q); R(a (x) b) = R(a) R(b)
    rng = np.random.default_rng(2)
    a, b = rand_unit(rng, (20,)), rand_unit(rng, (20,))
    to_scipy = lambda q: Rotation.from_quat(np.concatenate([q[..., 1:], q[..., :1]], axis=-1))  # scalar last
    Rab = to_scipy(m3.qmul(a, b)).as_matrix()
    assert np.allclose(Rab, to_scipy(a).as_matrix() @ to_scipy(b).as_matrix())
    v = rng.standard_normal((20, 3))
    vq = np.concatenate([np.zeros((20, 1)), v], axis=-1)
    rot = m3.qmul(m3.qmul(a, vq), m3.qconj(a))[:, 1:]
    assert np.allclose(rot, to_scipy(a).apply(v))


# ---------------------------------------------------------------- the scan
def test_cumprod_about_one_axis_adds_angles():
    rng = np.random.default_rng(3)
    b, L, H, Jn = 2, 37, 3, 2
    axis = rng.standard_normal((b, 1, H, Jn, 3))
    axis /= np.linalg.norm(axis, axis=-1, keepdims=True)
    theta = rng.uniform(-1.0, 1.0, (b, L, H, Jn))
    q = np.concatenate([np.cos(theta / 2)[..., None], np.sin(theta / 2)[..., None] * axis], axis=-1)
    init = rand_unit(rng, (b, H, Jn))
    cum = m3.quat_cumprod(q, init)
    tot = np.cumsum(theta, axis=1)
    rot = np.concatenate([np.cos(tot / 2)[..., None], np.sin(tot / 2)[..., None] * axis], axis=-1)
    assert np.allclose(cum, m3.qmul(rot, init[:, None]))


def test_cumprod_matches_scipy_composition():
    rng = np.random.default_rng(4)
    q, init = rand_unit(rng, (1, 9, 1, 1)), rand_unit(rng, (1, 1, 1))
    cum = m3.quat_cumprod(q, init)
    to_scipy = lambda x: Rotation.from_quat(np.concatenate([x[..., 1:], x[..., :1]], axis=-1))
    R = to_scipy(init[0, 0, 0])
    for t in range(9):
        R = to_scipy(q[0, t, 0, 0]) * R
        assert np.allclose(to_scipy(cum[0, t, 0, 0]).as_matrix(), R.as_matrix())


def _fd_check(f, args, grads, eps=1e-6, rtol=1e-6):
    for idx, (arr, g) in enumerate(zip(args, grads)):
        for pos in itertools.islice(np.ndindex(arr.shape), 0, None):
            old = arr[pos]
            arr[pos] = old + eps
            fp = f(*args)
            arr[pos] = old - eps
            fm = f(*args)
            arr[pos] = old
            num = (fp - fm) / (2 * eps)
            assert abs(num - g[pos]) <= rtol * max(1.0, abs(num)), (idx, pos, num, g[pos])


def test_cumprod_vjp_finite_differences():
    # non-unit quaternions: the reverse recurrence is the derivative for any input
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 5, 2, 1, 4)) * 0.7
    init = rng.standard_normal((1, 2, 1, 4))
    w = rng.standard_normal((1, 5, 2, 1, 4))
    loss = lambda q_, i_: float(np.sum(w * m3.quat_cumprod(q_, i_)))
    d_q, d_init = m3.quat_cumprod_vjp(q, init, w)
    _fd_check(loss, [q, init], [d_q, d_init])


def test_closed_form_equals_vjp_for_unit_quaternions_only():
    rng = np.random.default_rng(6)
    q = rand_unit(rng, (2, 23, 3, 2))
    init = rng.standard_normal((2, 3, 2, 4))
    d_cum = rng.standard_normal(q.shape)
    a = m3.quat_cumprod_vjp(q, init, d_cum)
    b = m3.quat_cumprod_backward_closed(q, init, d_cum)
    for x, y in zip(a, b):
        assert np.allclose(x, y, atol=1e-10)
    qn = q * rng.uniform(0.5, 1.5, q.shape[:-1] + (1,))  # not unit: the closed form no longer holds
    a = m3.quat_cumprod_vjp(qn, init, d_cum)
    b = m3.quat_cumprod_backward_closed(qn, init, d_cum)
    assert not np.allclose(a[0], b[0], atol=1e-3)


# ---------------------------------------------------------------- gamma correction
def _brute_y(V, B, C, gamma):
    T, m, H, P = V.shape
    N = B.shape[-1]
    y = np.zeros((T, m, H, P))
    for t, o, h, p in itertools.product(range(T), range(m), range(H), range(P)):
        acc = 0.0
        for i in range(m):
            qk = sum(C[t, o, h, r] * B[t, i, h, r] for r in range(N))
            acc += qk * V[t, i, h, p]
        y[t, o, h, p] = gamma[t, h] * acc
    return y


@pytest.mark.parametrize("m", [1, 2, 3])
def test_y_diag_brute_force(m):
    rng = np.random.default_rng(10 + m)
    T, H, P, N = 3, 2, 3, 4
    V = rng.standard_normal((T, m, H, P))
    B, C = rng.standard_normal((2, T, m, H, N))
    g = rng.standard_normal((T, H))
    assert np.allclose(m3.y_diag(V, B, C, g), _brute_y(V, B, C, g))


def test_y_diag_siso_is_the_mimo_case_of_rank_one():
    rng = np.random.default_rng(20)
    V = rng.standard_normal((7, 1, 3, 5))
    B, C = rng.standard_normal((2, 7, 1, 3, 6))
    g = rng.standard_normal((7, 3))
    assert np.allclose(m3.y_diag_siso(V, B, C, g), m3.y_diag(V, B, C, g))


@pytest.mark.parametrize("m", [1, 3])
def test_y_diag_vjp_finite_differences(m):
    rng = np.random.default_rng(30 + m)
    T, H, P, N = 2, 2, 3, 4
    V = rng.standard_normal((T, m, H, P))
    B, C = rng.standard_normal((2, T, m, H, N))
    g = rng.standard_normal((T, H))
    w = rng.standard_normal((T, m, H, P))
    loss = lambda V_, B_, C_, g_: float(np.sum(w * m3.y_diag(V_, B_, C_, g_)))
    dV, dB, dC, dg = m3.y_diag_vjp(w, V, B, C, g)
    _fd_check(loss, [V, B, C, g], [dV, dB, dC, dg])
