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


def run_gpu(inp, dtype: str, chunk_len: int, simt=False, backward=True, split_scan=False, check_status=False):
    d = to_device(inp, dtype)
    y, fin = ssd.ssd_forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], chunk_len,
                             init_state=d["init"], valid_len=d["valid_len"], simt=simt,
                             split_scan=split_scan, check_status=check_status)
    out = {"y": y, "final_state": fin}
    if backward:
        g = ssd.ssd_backward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], chunk_len, d["dy"],
                             d_final_state=d["d_final"], init_state=d["init"],
                             valid_len=d["valid_len"], simt=simt, split_scan=split_scan,
                             check_status=check_status)
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


# A tile's normwise error is taken against max(its own reference norm, this
# fraction of the root-mean-square reference norm of the tensor's tiles), so a
# tile whose reference is nearly zero is judged against a typical tile's size
# instead of its own.
TILE_FLOOR = 0.1


# Outputs checked tile by tile.  dA and dD are not: each entry is a sum over
# the whole batch and sequence of terms that largely cancel (the two sides of
# the d cumA identity), so one entry's relative error reflects that
# cancellation, not a local mistake; a wholly wrong entry still moves the
# whole-tensor norm of these [H] vectors far past the bar.
TILED_KEYS = ("y", "final_state", "dx", "ddt", "dB", "dC", "d_init")


def _tile_view(key, a, chunk):
    """Reshape one output into (tiles, elements per tile) without copying where
    the sequence length is a multiple of the chunk.  Tiles: (b, chunk, head) of
    y and dx; (b, head, chunk) of ddt; (b, chunk, group) of dB and dC; (b, head)
    of final_state and d_init."""
    a = np.asarray(a, np.float64)
    if key in ("final_state", "d_init"):
        return a.reshape(a.shape[0] * a.shape[1], -1), None
    seq_axis = 2 if key == "ddt" else 1
    L = a.shape[seq_axis]
    n = -(-L // chunk)
    if n * chunk != L:
        pad = [(0, 0)] * a.ndim
        pad[seq_axis] = (0, n * chunk - L)
        a = np.pad(a, pad)
    if key == "ddt":                          # [b, H, L] -> (b, H, n) tiles of Q
        b, H = a.shape[:2]
        return a.reshape(b * H * n, chunk), None
    b, _, X, Y = a.shape                      # [b, L, X, Y] -> tiles (b, n, X) of Q x Y
    return a.reshape(b, n, chunk, X, Y), (2, 4)


def tile_errors(gpu_a, ref_a, key, chunk):
    """Normwise relative error of every tile (see _tile_view), each against
    max(tile reference norm, TILE_FLOOR x RMS tile reference norm)."""
    g, axes = _tile_view(key, gpu_a, chunk)
    r, _ = _tile_view(key, ref_a, chunk)
    if axes is None:
        num = np.sum((g - r) ** 2, axis=1)
        den = np.sum(r ** 2, axis=1)
    else:                                     # per batch entry, to bound the temporaries
        num = np.stack([np.sum((g[i] - r[i]) ** 2, axis=(1, 3)) for i in range(g.shape[0])])
        den = np.stack([np.sum(r[i] ** 2, axis=(1, 3)) for i in range(r.shape[0])])
    num, den = num.ravel(), den.ravel()
    floor = TILE_FLOOR ** 2 * max(float(np.mean(den)), 1e-60)
    return np.sqrt(num / np.maximum(den, floor))


def compare(gpu, ref, tol, label="", chunk=None):
    """Normwise relative error of every output against the bar; with `chunk`,
    also the normwise error of every tile (tile_errors) against the same bar,
    so that one wrong tile of a large tensor cannot hide in the whole norm.
    Returns {key: whole-tensor error} and, with `chunk`, {key + "/tile": worst
    tile error}."""
    errs = {k: normrel(gpu[k], ref[k]) for k in OUT_KEYS if k in gpu and k in ref}
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{label}: normwise rel. error above {tol}: {bad} (all: {errs})"
    if chunk is not None:
        worst = {}
        for k in TILED_KEYS:
            if k in gpu and k in ref:
                te = tile_errors(gpu[k], ref[k], k, chunk)
                i = int(np.argmax(te))
                worst[k] = (float(te[i]), i)
        bad = {k: v for k, v in worst.items() if not v[0] <= tol}
        assert not bad, f"{label}: tile error above {tol} (key: (error, tile index)): {bad}"
        errs.update({k + "/tile": v[0] for k, v in worst.items()})
    return errs


def padded_grads_zero(gpu, valid_len):
    if valid_len is None:
        return
    for bi, v in enumerate(np.asarray(valid_len)):
        for k in ("y", "dx", "dB", "dC"):
            assert np.all(gpu[k][bi, v:] == 0), k
        assert np.all(gpu["ddt"][bi, :, v:] == 0)
