"""Pins of the CPU oracle to things other than itself (no GPU needed).

The serial recurrence (oracle/ssd_oracle.c) is checked against:
  * central finite differences of its own forward (every input entry),
  * the pages' chunked five-kernel formulation (oracle/chunked.py, written
    from burn-mamba's "combined_backward.rs" page) for several chunk lengths,
  * closed forms: one token, no decay (A = 0: causal linear attention), dt = 0,
  * linearity in (x, init), padding invariance past valid_len, and group
    invariance (G < H equals G = H with B/C replicated),
  * the page's own identities: the reverse-cumsum K1 backward, the
    ``out_x . dout - ddt . dt`` same-chunk identity, and the BLUE d_da identity,
  * a hand-worked example stored under tests/golden/.
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import chunked
from state_space_model_mamba_gb300.inputs import generate_small

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f64(d):
    return {k: (None if v is None else np.asarray(v, np.float64) if k != "valid_len" else v)
            for k, v in d.items()}


def fwd(d, **kw):
    return oracle.forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d.get("init"),
                          d.get("valid_len"), **kw)


def bwd(d, **kw):
    return oracle.backward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d.get("init"),
                           d.get("valid_len"), d["dy"], d.get("d_final"), **kw)


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def case(b=1, L=32, H=2, P=4, N=4, G=1, seed=0, init_std=0.5, valid_len=None, dt_mu=-1.0):
    d = generate_small(b, L, H, P, N, G, seed=seed, dt_mu=dt_mu, init_std=init_std,
                       d_final_std=1.0, valid_len=valid_len)
    if d["init"] is None:
        d["init"] = np.zeros((b, H, P, N), np.float32)
    return f64(d)


# ---------------------------------------------------------------- finite differences
FD_CASES = [
    dict(b=1, L=24, H=2, P=3, N=4, G=1, seed=1),
    dict(b=2, L=20, H=4, P=2, N=3, G=2, seed=2, valid_len=[13, 20]),
]


@pytest.mark.parametrize("spec", FD_CASES)
def test_backward_matches_central_differences(spec):
    d = case(**spec)
    g = bwd(d)
    names = {"x": "dx", "dt": "ddt", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "init": "d_init"}
    eps = 1e-6

    def L_of(dd):
        y, fin = fwd(dd)
        return oracle.loss(y, fin, dd["dy"], dd["d_final"])

    for inp, gname in names.items():
        base = d[inp]
        fd = np.empty(base.size)
        for i in range(base.size):
            dd = dict(d)
            pert = base.copy().reshape(-1)
            pert[i] += eps
            dd[inp] = pert.reshape(base.shape)
            lp = L_of(dd)
            pert[i] -= 2 * eps
            dd[inp] = pert.reshape(base.shape)
            lm = L_of(dd)
            fd[i] = (lp - lm) / (2 * eps)
        an = g[gname].reshape(-1)
        scale = max(np.max(np.abs(fd)), 1e-3)
        err = np.max(np.abs(an - fd)) / scale
        assert err < 1e-6, f"d{inp}: max err {err:.3e} (scale {scale:.3e})"


# ---------------------------------------------------------------- chunked == serial
@pytest.mark.parametrize("Q", [1, 2, 4, 16, 48])
@pytest.mark.parametrize("spec", [
    dict(b=1, L=48, H=2, P=3, N=5, G=1, seed=3),
    dict(b=2, L=45, H=4, P=4, N=3, G=2, seed=4, valid_len=[30, 45]),
])
def test_chunked_equals_serial(Q, spec):
    d = case(**spec)
    y_s, f_s = fwd(d)
    y_c, f_c = chunked.forward_chunked(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"],
                                       d["init"], d["valid_len"], Q=Q)
    assert rel(y_c, y_s) < 1e-11
    assert rel(f_c, f_s) < 1e-11
    g_s = bwd(d)
    g_c = chunked.backward_chunked(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"],
                                   d["valid_len"], d["dy"], d["d_final"], Q=Q)
    for k in ("dx", "ddt", "dA", "dB", "dC", "dD", "d_init"):
        assert rel(g_c[k], g_s[k]) < 1e-10, k


# ---------------------------------------------------------------- closed forms
def test_single_token_closed_form():
    d = case(b=2, L=1, H=3, P=4, N=5, G=1, seed=5)
    y, fin = fwd(d)
    a = np.exp(d["dt"][:, :, 0] * d["A"][None, :])                  # [b,H]
    S = a[..., None, None] * d["init"] + (d["dt"][:, :, 0][..., None, None]
                                         * d["x"][:, 0][..., None] * d["B"][:, 0, 0][:, None, None, :])
    y_ref = np.einsum("bhpr,br->bhp", S, d["C"][:, 0, 0]) + d["D"][None, :, None] * d["x"][:, 0]
    assert rel(fin, S) < 1e-14
    assert rel(y[:, 0], y_ref) < 1e-14


def test_no_decay_is_causal_linear_attention():
    d = case(b=1, L=40, H=2, P=3, N=4, G=1, seed=6)
    d["A"] = np.zeros_like(d["A"])
    y, fin = fwd(d)
    x, dt, B, C, D, h0 = d["x"][0], d["dt"][0], d["B"][0, :, 0], d["C"][0, :, 0], d["D"], d["init"][0]
    L = x.shape[0]
    CBt = C @ B.T                                               # [t, s]
    mask = np.tril(np.ones((L, L)))
    for h in range(2):
        M = CBt * mask * dt[h][None, :]
        y_ref = M @ x[:, h] + C @ h0[h].T + D[h] * x[:, h]
        assert rel(y[0, :, h], y_ref) < 1e-12
        fin_ref = h0[h] + (x[:, h] * dt[h][:, None]).T @ B
        assert rel(fin[0, h], fin_ref) < 1e-12


def test_zero_step_keeps_state():
    d = case(b=1, L=10, H=2, P=3, N=4, G=1, seed=7)
    d["dt"] = np.zeros_like(d["dt"])
    y, fin = fwd(d)
    y_ref = np.einsum("hpr,tr->thp", d["init"][0], d["C"][0, :, 0]) + d["D"][None, :, None] * d["x"][0]
    assert rel(fin, d["init"]) == 0.0
    assert rel(y[0], y_ref) < 1e-14


def test_hand_worked_golden():
    with open(os.path.join(GOLDEN, "hand_worked.json")) as f:
        g = json.load(f)
    inp = {k: np.asarray(v, np.float64) for k, v in g["inputs"].items()}
    y, fin = oracle.forward(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                            inp["init"], None)
    np.testing.assert_allclose(y.reshape(-1), np.asarray(g["y"]), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(fin.reshape(-1), np.asarray(g["final_state"]), rtol=1e-14)


# ---------------------------------------------------------------- invariants
def test_linear_in_x_and_init():
    d = case(b=2, L=30, H=2, P=3, N=4, G=1, seed=8)
    y1, f1 = fwd(d)
    d2 = dict(d, x=2.5 * d["x"], init=2.5 * d["init"])
    y2, f2 = fwd(d2)
    assert rel(y2, 2.5 * y1) < 1e-13 and rel(f2, 2.5 * f1) < 1e-13


def test_padding_invariance():
    V = np.array([17, 30], np.int32)
    d = case(b=2, L=30, H=2, P=3, N=4, G=1, seed=9, valid_len=V)
    y, fin = fwd(d)
    g = bwd(d)
    for bi in range(2):
        v = int(V[bi])
        t = {k: d[k][bi:bi + 1] for k in ("x", "B", "C", "dy")}
        dd = dict(d, x=t["x"][:, :v], B=t["B"][:, :v], C=t["C"][:, :v], dy=t["dy"][:, :v],
                  dt=d["dt"][bi:bi + 1, :, :v], init=d["init"][bi:bi + 1],
                  d_final=d["d_final"][bi:bi + 1], valid_len=None)
        yt, ft = fwd(dd)
        gt = bwd(dd)
        assert rel(y[bi:bi + 1, :v], yt) < 1e-14 and rel(fin[bi:bi + 1], ft) < 1e-14
        assert np.all(y[bi, v:] == 0)
        assert rel(g["dx"][bi:bi + 1, :v], gt["dx"]) < 1e-13
        assert rel(g["ddt"][bi:bi + 1, :, :v], gt["ddt"]) < 1e-13
        assert rel(g["d_init"][bi:bi + 1], gt["d_init"]) < 1e-13
        for k in ("dx", "dB", "dC"):
            assert np.all(g[k][bi, v:] == 0), k
        assert np.all(g["ddt"][bi, :, v:] == 0)
    # tail values do not matter
    d3 = dict(d)
    for k in ("x", "B", "C", "dy"):
        a = d[k].copy()
        a[0, V[0]:] = 123.0
        d3[k] = a
    dt3 = d["dt"].copy()
    dt3[0, :, V[0]:] = 7.0
    d3["dt"] = dt3
    y3, f3 = fwd(d3)
    g3 = bwd(d3)
    assert np.array_equal(y3, y) and np.array_equal(f3, fin)
    for k in ("dx", "ddt", "dA", "dB", "dC", "dD", "d_init"):
        assert rel(g3[k], g[k]) < 1e-14, k


def test_group_invariance():
    d = case(b=2, L=24, H=4, P=3, N=4, G=2, seed=10)
    y, fin = fwd(d)
    g = bwd(d)
    rep = dict(d, B=np.repeat(d["B"], 2, axis=2), C=np.repeat(d["C"], 2, axis=2))
    y2, f2 = fwd(rep)
    g2 = bwd(rep)
    assert rel(y, y2) < 1e-14 and rel(fin, f2) < 1e-14
    for k in ("dx", "ddt", "dA", "dD", "d_init"):
        assert rel(g[k], g2[k]) < 1e-13, k
    assert rel(g["dB"], g2["dB"].reshape(2, 24, 2, 2, 4).sum(3)) < 1e-13
    assert rel(g["dC"], g2["dC"].reshape(2, 24, 2, 2, 4).sum(3)) < 1e-13


# ---------------------------------------------------------------- the page's identities
def _chunked_case(Q=8):
    d = case(b=2, L=32, H=2, P=3, N=4, G=1, seed=11)
    g = chunked.backward_chunked(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"],
                                 None, d["dy"], d["d_final"], Q=Q)
    return d, g


def test_reverse_cumsum_identity():
    _, g = _chunked_case()
    assert rel(g["d_da"], g["d_da_suffix"]) < 1e-13


def test_out_x_dout_minus_ddt_dt_identity():
    d, g = _chunked_case()
    y, _ = fwd(d)
    lhs = g["d_da_local"]                                             # [b,H,L]
    rhs = (np.einsum("blhp,blhp->bhl", y - d["D"][None, None, :, None] * d["x"], d["dy"])
           - g["d_dt_orange"] * d["dt"])
    assert rel(lhs, rhs) < 1e-11


def test_blue_d_da_identity():
    d, g = _chunked_case()
    nb, L, H, P = d["x"].shape
    Q = 8
    Ch = np.repeat(d["C"], H, axis=2).reshape(nb, L // Q, Q, H, 4)
    lhs = g["d_da_blue"]                                              # [b,H,n,Q]
    rhs = np.einsum("bnlhr,bnlhr->bhnl", g["dC_blue_h"], Ch)
    assert rel(lhs, rhs) < 1e-12
