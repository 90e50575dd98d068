"""Plant plausible mistakes in a copy of the CPU oracle and check that the pins
(finite differences, chunked == serial, closed forms) catch every one.

Each mutation is a one-line edit of ``oracle/ssd_oracle.c`` compiled into a
temporary library; the shipped oracle is never modified.
"""
import numpy as np
import pytest

import oracle
from oracle import chunked
from state_space_model_mamba_gb300.inputs import generate_small

MUTATIONS = {
    "ddt_decay_sign": ("ddt[(bi * H + h) * L + t] = s_w + Ah * a * s_a;",
                       "ddt[(bi * H + h) * L + t] = s_w - Ah * a * s_a;"),
    "dx_drops_skip": ("dxt[p] = Dh * dyt[p] + dtt * gb[p];", "dxt[p] = dtt * gb[p];"),
    "dA_drops_decay": ("dA_acc += dtt * a * s_a;", "dA_acc += dtt * s_a;"),
    "dC_uses_prev_state": ("acc += dyt[p] * Scur[p * N + r];", "acc += dyt[p] * Sprev[p * N + r];"),
    "dB_drops_dt": ("dBt[r] += dtt * acc;", "dBt[r] += acc;"),
    "carry_not_decayed": ("for (int64_t i = 0; i < PN; ++i) Gs[i] *= a;", ""),
    "group_index_modulo": ("g = h / hpg;", "g = h % G;"),
    "forward_B_C_swapped": ("step_state(S, P, N, a, dtt, xt, Bt);", "step_state(S, P, N, a, dtt, xt, Ct);"),
    "forward_skip_dropped": ("yt[p] = acc + D[h] * xt[p];", "yt[p] = acc;"),
    "valid_len_off_by_one": ("if (v > L) v = L;", "if (v > L) v = L;\n    if (v > 0) v -= 1;"),
}


def _case():
    d = generate_small(2, 12, 4, 2, 3, 2, seed=21, dt_mu=-1.0, init_std=0.5, d_final_std=1.0,
                       valid_len=[7, 12])
    return {k: (v if v is None or k == "valid_len" else np.asarray(v, np.float64))
            for k, v in d.items()}


def _pins_hold(lib) -> bool:
    d = _case()
    args = (d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], d["valid_len"])
    y, fin = oracle.forward(*args, lib=lib)
    # (1) chunked restatement of the pages' kernels
    yc, fc = chunked.forward_chunked(*args, Q=4)
    if not (np.allclose(y, yc, rtol=1e-10, atol=1e-12) and np.allclose(fin, fc, rtol=1e-10)):
        return False
    g = oracle.backward(*args, d["dy"], d["d_final"], lib=lib)
    gc = chunked.backward_chunked(*args, d["dy"], d["d_final"], Q=4)
    for k in g:
        if not np.allclose(g[k], gc[k], rtol=1e-9, atol=1e-11):
            return False
    # (2) central differences on a few entries of every input
    eps = 1e-6
    rng = np.random.default_rng(0)
    names = {"x": "dx", "dt": "ddt", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "init": "d_init"}
    for inp, gname in names.items():
        base = d[inp]
        for i in rng.choice(base.size, size=min(6, base.size), replace=False):
            vals = []
            for s in (+1, -1):
                pert = base.copy().reshape(-1)
                pert[i] += s * eps
                dd = dict(d)
                dd[inp] = pert.reshape(base.shape)
                yy, ff = oracle.forward(dd["x"], dd["dt"], dd["A"], dd["B"], dd["C"], dd["D"],
                                        dd["init"], dd["valid_len"], lib=lib)
                vals.append(oracle.loss(yy, ff, d["dy"], d["d_final"]))
            fd = (vals[0] - vals[1]) / (2 * eps)
            if abs(fd - g[gname].reshape(-1)[i]) > 1e-6 * max(1.0, abs(fd)):
                return False
    return True


def test_unmodified_oracle_passes_the_pins():
    assert _pins_hold(None)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = oracle.source_text()
    assert old in src, f"mutation anchor for {name} not found"
    lib = oracle.compile_variant(src.replace(old, new), str(tmp_path))
    assert not _pins_hold(lib), f"planted mistake {name} was not caught"
