"""GPU parity of the Mamba-3 entry points (include/mamba3.h), through the C ABI,
against the fp64 oracle (oracle/mamba3.py) on seeded inputs.  Bars: normwise
relative error <= 1e-4 for fp32 storage and <= 2e-2 for bf16 storage, over each
whole tensor and over every slice of it along the leading (chain or token)
axes, the slice's reference norm floored at a tenth of the tensor's RMS slice
norm (so a wholly wrong chain or token cannot hide in a large tensor)."""
import numpy as np
import pytest

from oracle import mamba3 as om3
from state_space_model_mamba_gb300.inputs import (MAMBA3_WORKLOADS, DiagWorkload, QuatWorkload, generate_diag,
                                                  generate_quat)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def check(gpu, ref, tol, what, slice_axes):
    """Whole-tensor and per-slice normwise errors; slice_axes: leading axes that index a slice."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, what
    assert np.isfinite(gpu).all(), what
    whole = np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-30)
    assert whole <= tol, f"{what}: {whole:.3e} > {tol}"
    k = int(np.prod(ref.shape[:slice_axes]))
    d = (gpu - ref).reshape(k, -1)
    r = ref.reshape(k, -1)
    rn = np.linalg.norm(r, axis=1)
    floor = 0.1 * np.sqrt(np.mean(rn ** 2))
    worst = float(np.max(np.linalg.norm(d, axis=1) / np.maximum(rn, max(floor, 1e-30))))
    assert worst <= tol, f"{what} (worst slice): {worst:.3e} > {tol}"
    return whole, worst


def dev(a, dt=torch.float32):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda().to(dt)


@pytest.fixture(scope="module")
def m3():
    from state_space_model_mamba_gb300 import mamba3
    return mamba3


# ---------------------------------------------------------------- quaternion scan
# ragged segment tails, one segment, many; 9000 steps give a lane more than
# eight segments in the per-chain carry kernels (their batched path)
QUAT_SHAPES = [(1, 1, 1, 1), (2, 127, 3, 2), (2, 128, 2, 3), (1, 129, 4, 1), (3, 700, 5, 2), (1, 2049, 2, 8),
               (1, 9000, 1, 2)]


@pytest.mark.parametrize("shape", QUAT_SHAPES)
@pytest.mark.parametrize("with_init", [True, False])
def test_quat_scan_forward_backward(m3, shape, with_init):
    b, L, H, J = shape
    inp = generate_quat(QuatWorkload("t", b, L, H, J, seed=7 + L + H), seed=None)
    init = inp["init"] if with_init else None
    q, d_cum = dev(inp["q"]), dev(inp["d_cum"])
    cum = m3.quat_cumprod(q, dev(init))
    d_q, d_init = m3.quat_cumprod_backward(q, dev(init), d_cum)
    torch.cuda.synchronize()
    i64 = init if with_init else np.tile(np.array([1.0, 0, 0, 0]), (b, H, J, 1))
    check(cum.cpu().numpy(), om3.quat_cumprod(inp["q"], i64), 1e-4, "cum", 4)
    rq, ri = om3.quat_cumprod_backward_closed(inp["q"], i64, inp["d_cum"])
    check(d_q.cpu().numpy(), rq, 1e-4, "d_q", 4)
    check(d_init.cpu().numpy(), ri, 1e-4, "d_init", 3)
    # the page's closed form is the derivative itself on (near-)unit inputs
    vq, _ = om3.quat_cumprod_vjp(inp["q"], i64, inp["d_cum"])
    check(d_q.cpu().numpy(), vq, 1e-4, "d_q vs derivative", 4)


def test_quat_scan_full_size(m3):
    w = MAMBA3_WORKLOADS["quat_scan_2p7b"]
    inp = generate_quat(w)
    q, init, d_cum = dev(inp["q"]), dev(inp["init"]), dev(inp["d_cum"])
    cum = m3.quat_cumprod(q, init)
    d_q, d_init = m3.quat_cumprod_backward(q, init, d_cum)
    torch.cuda.synchronize()
    e1 = check(cum.cpu().numpy(), om3.quat_cumprod(inp["q"], inp["init"]), 1e-4, "cum", 4)
    rq, ri = om3.quat_cumprod_backward_closed(inp["q"], inp["init"], inp["d_cum"])
    e2 = check(d_q.cpu().numpy(), rq, 1e-4, "d_q", 4)
    e3 = check(d_init.cpu().numpy(), ri, 1e-4, "d_init", 3)
    print("quat_scan_2p7b", {k: f"{v[0]:.2e}/{v[1]:.2e}" for k, v in zip(("cum", "d_q", "d_init"), (e1, e2, e3))})


# ---------------------------------------------------------------- gamma correction
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("m", [1, 2, 3, 4])
@pytest.mark.parametrize("P,N", [(64, 128), (6, 10), (130, 66)])
def test_y_diag_forward_backward(m3, dtype, m, P, N):
    w = DiagWorkload("t", 37, m, 5, P, N, dtype=dtype, seed=40 + m + P)
    inp = generate_diag(w)
    td = torch.float32 if dtype == "f32" else torch.bfloat16
    V, B, C, dY = (dev(inp[k], td) for k in ("V", "B", "C", "dY"))
    g = dev(inp["gamma"])
    y = m3.y_diag(V, B, C, g)
    dV, dB, dC, dg = m3.y_diag_backward(dY, V, B, C, g)
    torch.cuda.synchronize()
    tol = 1e-4 if dtype == "f32" else 2e-2
    ref_y = om3.y_diag(inp["V"], inp["B"], inp["C"], inp["gamma"])
    check(y.float().cpu().numpy(), ref_y, tol, "y", 3)
    rV, rB, rC, rg = om3.y_diag_vjp(inp["dY"], inp["V"], inp["B"], inp["C"], inp["gamma"])
    check(dV.float().cpu().numpy(), rV, tol, "dV", 3)
    check(dB.float().cpu().numpy(), rB, tol, "dB", 3)
    check(dC.float().cpu().numpy(), rC, tol, "dC", 3)
    check(dg.cpu().numpy(), rg, tol, "d_gamma", 1)


@pytest.mark.parametrize("name", ["ydiag_siso_2p7b", "ydiag_mimo4"])
def test_y_diag_full_size(m3, name):
    w = MAMBA3_WORKLOADS[name]
    inp = generate_diag(w)
    V, B, C, dY = (dev(inp[k], torch.bfloat16) for k in ("V", "B", "C", "dY"))
    g = dev(inp["gamma"])
    y = m3.y_diag(V, B, C, g)
    dV, dB, dC, dg = m3.y_diag_backward(dY, V, B, C, g)
    torch.cuda.synchronize()
    errs = {"y": check(y.float().cpu().numpy(), om3.y_diag(inp["V"], inp["B"], inp["C"], inp["gamma"]),
                       2e-2, "y", 3)}
    rV, rB, rC, rg = om3.y_diag_vjp(inp["dY"], inp["V"], inp["B"], inp["C"], inp["gamma"])
    for nm, a, r in (("dV", dV, rV), ("dB", dB, rB), ("dC", dC, rC)):
        errs[nm] = check(a.float().cpu().numpy(), r, 2e-2, nm, 3)
    errs["d_gamma"] = check(dg.cpu().numpy(), rg, 2e-2, "d_gamma", 1)
    print(name, {k: f"{v[0]:.2e}/{v[1]:.2e}" for k, v in errs.items()})



def host(t):
    return t.float().cpu().numpy()


@pytest.mark.parametrize("i", range(6))
def test_quat_scan_random_shapes(m3, i):
    """Random batch, length (up to ~19k steps: several carry batches per lane), heads, blocks."""
    rng = np.random.default_rng(9700 + i)
    b, L, H, J = int(rng.integers(1, 4)), int(rng.integers(1, 20000)), int(rng.integers(1, 5)), int(rng.integers(1, 5))
    qi = generate_quat(QuatWorkload("r", b, L, H, J, seed=9710 + i), seed=None)
    with_init = bool(i % 2)
    init = qi["init"] if with_init else np.tile(np.array([1, 0, 0, 0], np.float32), (b, H, J, 1))
    gin = dev(qi["init"]) if with_init else None
    cum = m3.quat_cumprod(dev(qi["q"]), gin)
    d_q, d_init = m3.quat_cumprod_backward(dev(qi["q"]), gin, dev(qi["d_cum"]))
    torch.cuda.synchronize()
    rq, ri = om3.quat_cumprod_backward_closed(qi["q"], init, qi["d_cum"])
    check(host(cum), om3.quat_cumprod(qi["q"], init), 1e-4, "cum", 2)
    check(host(d_q), rq, 1e-4, "d_q", 2)
    check(host(d_init), ri, 1e-4, "d_init", 1)


@pytest.mark.parametrize("i", range(8))
def test_y_diag_random_shapes(m3, i):
    """Random token count, rank, heads and (P, N): the one-piece-per-lane kernels and the looping ones."""
    rng = np.random.default_rng(9800 + i)
    T, m, H = int(rng.integers(1, 3000)), int(rng.integers(1, 5)), int(rng.integers(1, 9))
    P, N = int(rng.choice([2, 6, 32, 64, 66, 130])), int(rng.choice([4, 10, 64, 128, 132]))
    dtype = "bf16" if i % 2 == 0 else "f32"
    di = generate_diag(DiagWorkload("r", T, m, H, P, N, dtype=dtype, seed=9810 + i))
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    V, B, C, dY = (dev(di[k], tdt) for k in ("V", "B", "C", "dY"))
    g = dev(di["gamma"])
    y = m3.y_diag(V, B, C, g)
    grads = m3.y_diag_backward(dY, V, B, C, g)
    torch.cuda.synchronize()
    tol = 2e-2 if dtype == "bf16" else 1e-4
    check(host(y), om3.y_diag(di["V"], di["B"], di["C"], di["gamma"]), tol, "y", 1)
    for name, a, r in zip(("dV", "dB", "dC", "d_gamma"), grads,
                          om3.y_diag_vjp(di["dY"], di["V"], di["B"], di["C"], di["gamma"])):
        check(host(a), r, tol, name, 1)
