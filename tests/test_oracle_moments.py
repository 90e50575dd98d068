"""Pins of the state-moment oracle (oracle.state_moments, oracle/moments.py)
against facts it does not restate: every per-token state read back out of the
already-pinned forward oracle (one-hot C and D = 0 make y_t = S_t[:, r]),
the dt = 0 closed form, additivity over a split of the sequence, and the
participation ratio's textbook values (identity, rank one, a known spectrum
under a random rotation) and the pages' statements about the complex and
quaternionic forms (the real pairing is the real PR; one complex or quaternion
direction counts as one)."""
import numpy as np
import pytest

import oracle
from oracle import moments as om
from state_space_model_mamba_gb300.inputs import generate_small


def all_states(inp):
    """S_t for every token from the forward oracle: [b, L, H, P, N]."""
    b, L, H, P = inp["x"].shape
    N, G = inp["B"].shape[-1], inp["B"].shape[2]
    S = np.zeros((b, L, H, P, N))
    D0 = np.zeros_like(inp["D"])
    for r in range(N):
        C = np.zeros((b, L, G, N))
        C[..., r] = 1.0
        y, _ = oracle.forward(inp["x"], inp["dt"], inp["A"], inp["B"], C, D0, inp["init"], inp["valid_len"])
        S[..., r] = y
    return S


@pytest.mark.parametrize("G,vl", [(1, None), (2, [13, 20])])
def test_moments_match_states_read_from_forward_oracle(G, vl):
    inp = generate_small(2, 20, 4, 3, 5, G, seed=11 + G, init_std=0.4, valid_len=vl)
    S = all_states(inp)
    b, L = 2, 20
    V = np.full(b, L) if vl is None else np.asarray(vl)
    mask = (np.arange(L)[None, :] < V[:, None]).astype(np.float64)
    m2_ref = np.einsum("bt,bthpr,bthps->bhrs", mask, S, S)
    m1_ref = np.einsum("bt,bthpr->bhr", mask, S)
    m2, m1, n = oracle.state_moments(inp["x"], inp["dt"], inp["A"], inp["B"], inp["init"], inp["valid_len"])
    assert np.allclose(m2, m2_ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(m1, m1_ref, rtol=1e-12, atol=1e-12)
    assert list(n) == list(V * 3)


def test_moments_dt_zero_keep_the_initial_state():
    inp = generate_small(1, 9, 2, 3, 4, 1, seed=5, init_std=1.0)
    inp["dt"][:] = 0.0
    m2, m1, _ = oracle.state_moments(inp["x"], inp["dt"], inp["A"], inp["B"], inp["init"])
    h0 = inp["init"].astype(np.float64)
    assert np.allclose(m2, 9 * np.einsum("bhpr,bhps->bhrs", h0, h0))
    assert np.allclose(m1, 9 * h0.sum(axis=2))


def test_moments_add_over_a_split_sequence():
    inp = generate_small(1, 30, 2, 3, 4, 1, seed=6, init_std=0.5)
    cut = 11
    m2, m1, _ = oracle.state_moments(inp["x"], inp["dt"], inp["A"], inp["B"], inp["init"])
    first = {k: (v[:, :cut] if k in ("x", "B", "C") else v[..., :cut] if k == "dt" else v) for k, v in inp.items()}
    second = {k: (v[:, cut:] if k in ("x", "B", "C") else v[..., cut:] if k == "dt" else v) for k, v in inp.items()}
    a2, a1, _ = oracle.state_moments(first["x"], first["dt"], inp["A"], first["B"], inp["init"])
    _, fin = oracle.forward(first["x"], first["dt"], inp["A"], first["B"], first["C"], inp["D"], inp["init"])
    b2, b1, _ = oracle.state_moments(second["x"], second["dt"], inp["A"], second["B"], fin)
    assert np.allclose(m2, a2 + b2) and np.allclose(m1, a1 + b1)


# ---------------------------------------------------------------- participation ratio
def spd(rng, eig):
    Q, _ = np.linalg.qr(rng.standard_normal((len(eig), len(eig))))
    return Q @ np.diag(eig) @ Q.T


def test_pr_textbook_values():
    rng = np.random.default_rng(0)
    n = np.array([7])
    N = 6
    assert np.allclose(om.pr(np.eye(N)[None, None] * 7, None, n), N)
    v = rng.standard_normal(N)
    assert np.allclose(om.pr(np.outer(v, v)[None, None] * 7, None, n), 1.0)
    eig = np.array([3.0, 1.0, 0.5, 0.25, 0.0, 0.0])
    assert np.allclose(om.pr(spd(rng, eig)[None, None], None, np.array([1])), eig.sum() ** 2 / (eig ** 2).sum())
    # scale invariance, and the page's trace
    m = spd(rng, eig)[None, None] * 5.0
    assert np.allclose(om.pr(m, None, n), om.pr(m * 1e-20, None, n))
    assert np.allclose(om.trace(m, n), np.trace(m[0, 0]) / 7)


def test_pr_centred_uses_the_sample_covariance():
    rng = np.random.default_rng(1)
    X = rng.standard_normal((500, 5)) @ rng.standard_normal((5, 5)) + 3.0
    m2 = (X.T @ X)[None, None]
    m1 = X.sum(axis=0)[None, None]
    cov = np.cov(X.T, bias=True)
    ev = np.linalg.eigvalsh(cov)
    assert np.allclose(om.pr(m2, m1, np.array([500]), center=True), ev.sum() ** 2 / (ev ** 2).sum())


def test_pr_complex_real_pairing_is_pr_and_one_direction_counts_once():
    rng = np.random.default_rng(2)
    m2 = spd(rng, rng.uniform(0.1, 2.0, 8))[None, None]
    n = np.array([3])
    assert np.allclose(om.pr_complex(m2, None, n, om.REAL, 0), om.pr(m2, None, n))
    # a single rotating complex direction: (cos th, sin th) samples; real PR 2, complex PR 1
    th = rng.uniform(0, 2 * np.pi, 4000)
    X = np.stack([np.cos(th), np.sin(th)], axis=1) * 2.0
    m2c = (X.T @ X)[None, None]
    n2 = np.array([4000])
    assert om.pr(m2c, None, n2)[0, 0] == pytest.approx(2.0, abs=0.05)
    assert np.allclose(om.pr_complex(m2c, None, n2, om.COMPLEX_INTERLEAVED, 1), 1.0)
    # one quaternion block: the Hermitian moment is a 1 x 1 real number whatever the samples
    q = rng.standard_normal((3000, 4))
    m2q = (q.T @ q)[None, None]
    assert om.pr(m2q, None, np.array([3000]))[0, 0] > 3.5
    assert np.allclose(om.pr_complex(m2q, None, np.array([3000]), om.QUATERNION_BLOCKS, 1), 1.0)


def test_pr_complex_half_half_is_interleaved_after_the_permutation():
    rng = np.random.default_rng(3)
    R, npair = 10, 3
    m2 = spd(rng, rng.uniform(0.1, 2.0, R))
    perm = list(range(R))  # interleaved index of each half-half coordinate
    half = R // 2
    order = [None] * R
    for a in range(npair):
        order[2 * a] = a
        order[2 * a + 1] = half + a
    rest = [k for k in perm if k not in order[:2 * npair]]
    order[2 * npair:] = rest
    m2_inter = m2[np.ix_(order, order)]
    a = om.pr_complex(m2[None, None], None, np.array([1]), om.COMPLEX_HALF_HALF, npair)
    b = om.pr_complex(m2_inter[None, None], None, np.array([1]), om.COMPLEX_INTERLEAVED, npair)
    assert np.allclose(a, b)


def test_pr_complex_two_equal_directions_count_two():
    rng = np.random.default_rng(4)
    th1, th2 = rng.uniform(0, 2 * np.pi, (2, 6000))
    z = np.stack([np.cos(th1), np.cos(th2), np.sin(th1), np.sin(th2)], axis=1)  # half-half: x0, x1, y0, y1
    m2 = (z.T @ z)[None, None]
    assert om.pr_complex(m2, None, np.array([6000]), om.COMPLEX_HALF_HALF, 2)[0, 0] == pytest.approx(2.0, abs=0.05)
