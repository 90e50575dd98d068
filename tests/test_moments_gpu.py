"""GPU parity of the state-moment path (ssd_state_moments, ssd_state_pr) through
the C ABI against the oracle: the per-token definition in the C oracle for
m2 / m1 / count, NumPy for the participation ratio.  Bars: normwise relative
error <= 2e-2 for m2 and m1 (bf16 operands), over the whole tensor and over
each (b, h) slice (the slice norm floored at a tenth of the RMS slice norm);
counts exact; PR and trace within 1e-4 of the oracle evaluated on the GPU's
own moments (fp32 arithmetic)."""
import numpy as np
import pytest

import oracle
from oracle import moments as om
from state_space_model_mamba_gb300.inputs import WORKLOADS, generate, generate_small
from parity_util import to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def slicewise(gpu, ref, tol, what):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(gpu).all(), what
    whole = np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-30)
    k = ref.shape[0] * ref.shape[1]
    d = (gpu - ref).reshape(k, -1)
    rn = np.linalg.norm(ref.reshape(k, -1), axis=1)
    floor = 0.1 * np.sqrt(np.mean(rn ** 2))
    worst = float(np.max(np.linalg.norm(d, axis=1) / np.maximum(rn, max(floor, 1e-30))))
    assert whole <= tol and worst <= tol, f"{what}: whole {whole:.3e}, worst slice {worst:.3e} (bar {tol})"
    return whole, worst


def gpu_moments(inp, split=False):
    from state_space_model_mamba_gb300 import ssd
    d = to_device(inp, "bf16")
    m2, m1, n = ssd.state_moments(d["x"], d["dt"], d["A"], d["B"], init_state=d["init"],
                                  valid_len=d["valid_len"], check_status=True, split_scan=split)
    torch.cuda.synchronize()
    return m2.cpu().numpy(), m1.cpu().numpy(), n.cpu().numpy()


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("b,L,H,G,vl", [(2, 300, 3, 1, [300, 129]), (2, 700, 40, 2, [700, 1]),
                                        (1, 128, 2, 1, None), (3, 200, 2, 2, [0, 77, 200])])
def test_state_moments_match_oracle(b, L, H, G, vl, split):
    inp = generate_small(b, L, H, 64, 128, G, seed=200 + L + H, init_std=0.3, valid_len=vl, bf16=True)
    m2, m1, n = gpu_moments(inp, split)
    r2, r1, rn = oracle.state_moments(inp["x"], inp["dt"], inp["A"], inp["B"], inp["init"], inp["valid_len"])
    assert list(n) == list(rn)
    e2 = slicewise(m2, r2, 2e-2, "m2")
    e1 = slicewise(m1, r1, 2e-2, "m1")
    assert np.allclose(m2, np.swapaxes(m2, -1, -2), rtol=1e-6, atol=1e-6 * np.abs(m2).max())  # symmetric
    print(f"b={b} L={L} H={H} split={split}", f"m2 {e2[0]:.2e}/{e2[1]:.2e}", f"m1 {e1[0]:.2e}/{e1[1]:.2e}")


def test_state_moments_strong_decay_and_tiny_steps():
    # fast decay (sigma, tau near 1, F nearly diagonal) and exact zeros of dt
    inp = generate_small(2, 400, 4, 64, 128, 1, seed=230, init_std=0.3, valid_len=[400, 257], bf16=True,
                         dt_mu=0.5)
    inp["dt"][:, :, ::7] = 0.0
    m2, m1, _ = gpu_moments(inp)
    r2, r1, _ = oracle.state_moments(inp["x"], inp["dt"], inp["A"], inp["B"], inp["init"], inp["valid_len"])
    slicewise(m2, r2, 2e-2, "m2")
    slicewise(m1, r1, 2e-2, "m1")


def test_state_moments_full_size_head_sample():
    # the 2.7B layer on the GPU; the oracle (about a teraflop per head-set in fp64)
    # on the first four heads, which do not depend on the others (one group)
    w = WORKLOADS["mamba2_2p7b"]
    inp = generate(w)
    m2, m1, n = gpu_moments(inp)
    hs = 4
    r2, r1, rn = oracle.state_moments(inp["x"][:, :, :hs], inp["dt"][:, :hs], inp["A"][:hs], inp["B"],
                                      None, None)
    assert list(n) == list(rn)
    e2 = slicewise(m2[:, :hs], r2, 2e-2, "m2")
    e1 = slicewise(m1[:, :hs], r1, 2e-2, "m1")
    print("mamba2_2p7b heads 0-3", f"m2 {e2[0]:.2e}/{e2[1]:.2e}", f"m1 {e1[0]:.2e}/{e1[1]:.2e}")


@pytest.mark.parametrize("i", range(8))
def test_state_moments_random_shapes(i):
    """Random batch, length, groups, heads and ragged valid lengths; both chunk-state paths."""
    rng = np.random.default_rng(9500 + i)
    b, L, G = int(rng.integers(1, 4)), int(rng.integers(1, 1200)), int(rng.choice([1, 2]))
    H = G * int(rng.integers(1, 24))
    vl = [int(v) for v in rng.integers(0, L + 1, size=b)] if rng.random() < 0.6 else None
    inp = generate_small(b, L, H, 64, 128, G, seed=9600 + i, init_std=0.3, valid_len=vl, bf16=True)
    m2, m1, n = gpu_moments(inp, split=bool(i % 2))
    r2, r1, rn = oracle.state_moments(inp["x"], inp["dt"], inp["A"], inp["B"], inp["init"], inp["valid_len"])
    assert list(n) == list(rn)
    slicewise(m2, r2, 2e-2, "m2")
    slicewise(m1, r1, 2e-2, "m1")


PAIRINGS = [(0, 0), (1, 40), (1, 64), (2, 16), (2, 64), (3, 8), (3, 32)]


@pytest.mark.parametrize("pairing,num", PAIRINGS)
@pytest.mark.parametrize("center", [False, True])
@pytest.mark.parametrize("pool", [False, True])
def test_state_pr_matches_oracle(pairing, num, center, pool):
    from state_space_model_mamba_gb300 import ssd
    inp = generate_small(3, 300, 4, 64, 128, 1, seed=240, init_std=0.5, valid_len=[300, 100, 257], bf16=True)
    d = to_device(inp, "bf16")
    m2, m1, n = ssd.state_moments(d["x"], d["dt"], d["A"], d["B"], init_state=d["init"], valid_len=d["valid_len"])
    pr, tr = ssd.state_pr(m2, m1, n, center=center, pairing=pairing, num=num, pool_batch=pool)
    torch.cuda.synchronize()
    M2, M1, N_ = (t.cpu().numpy().astype(np.float64) for t in (m2, m1, n))
    if pool:
        M2, M1, N_ = M2.sum(0, keepdims=True), M1.sum(0, keepdims=True), N_.sum(keepdims=True)
    ref = om.pr_complex(M2, M1, N_, pairing, num, center=center)
    assert np.allclose(pr.cpu().numpy(), ref, rtol=1e-4, atol=0), (pr.cpu().numpy(), ref)
    assert np.allclose(tr.cpu().numpy(), om.trace(M2, N_), rtol=1e-4)


def test_state_pr_rejects_bad_pairings():
    from state_space_model_mamba_gb300 import ssd
    m2 = torch.zeros(1, 1, 8, 8, device="cuda")
    m1 = torch.zeros(1, 1, 8, device="cuda")
    n = torch.ones(1, device="cuda", dtype=torch.int64)
    for pairing, num in ((1, 5), (2, 5), (3, 3), (7, 1)):
        with pytest.raises(ssd.SsdError):
            ssd.state_pr(m2, m1, n, pairing=pairing, num=num)
