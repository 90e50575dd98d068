"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
binding and the CPU oracle on the same seeded inputs, and compare."""
import numpy as np
import torch

import oracle
from state_space_model_mamba_gb300 import ssd

OUT_KEYS = ("y", "final_state", "dx", "ddt", "dA", "dB", "dC", "dD", "d_init")
TOL = {"f32": 1e-4, "bf16": 2e-2}


def to_device(inp, dtype: str, device="cuda"):
    T = torch.float32 if dtype == "f32" else torch.bfloat16

    def t(a, dt=torch.float32):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dt)

    return dict(x=t(inp["x"], T), dt=t(inp["dt"]), A=t(inp["A"]), B=t(inp["B"], T), C=t(inp["C"], T),
                D=t(inp["D"]), init=t(inp["init"]), dy=t(inp["dy"], T), d_final=t(inp["d_final"]),
                valid_len=None if inp["valid_len"] is None else
                torch.from_numpy(np.asarray(inp["valid_len"], np.int32)).to(device))


def run_gpu(inp, dtype: str, chunk_len: int, simt=False, backward=True):
    d = to_device(inp, dtype)
    y, fin = ssd.ssd_forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], chunk_len,
                             init_state=d["init"], valid_len=d["valid_len"], simt=simt)
    out = {"y": y, "final_state": fin}
    if backward:
        g = ssd.ssd_backward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], chunk_len, d["dy"],
                             d_final_state=d["d_final"], init_state=d["init"],
                             valid_len=d["valid_len"], simt=simt)
        out.update(g)
    torch.cuda.synchronize()
    return {k: v.double().cpu().numpy() for k, v in out.items() if v is not None}


def run_oracle(inp, backward=True):
    y, fin = oracle.forward(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                            inp["init"], inp["valid_len"])
    out = {"y": y, "final_state": fin}
    if backward:
        g = oracle.backward(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                            inp["init"], inp["valid_len"], inp["dy"], inp["d_final"])
        out.update(g)
    return out


def normrel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def compare(gpu, ref, tol, label=""):
    errs = {k: normrel(gpu[k], ref[k]) for k in OUT_KEYS if k in gpu and k in ref}
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{label}: normwise rel. error above {tol}: {bad} (all: {errs})"
    return errs


def padded_grads_zero(gpu, valid_len):
    if valid_len is None:
        return
    for bi, v in enumerate(np.asarray(valid_len)):
        for k in ("y", "dx", "dB", "dC"):
            assert np.all(gpu[k][bi, v:] == 0), k
        assert np.all(gpu["ddt"][bi, :, v:] == 0)
