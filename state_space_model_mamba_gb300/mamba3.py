"""Thin Python binding of the Mamba-3 entry points of ``libssd.so``
(``include/mamba3.h``): the quaternion cumulative-product scan and its
backward, and the same-step gamma correction and its backward.

Argument marshalling only, as :mod:`ssd`: torch CUDA tensors supply memory
and streams, every step runs in the library's kernels, and a missing library
or a failed call raises.
"""
from __future__ import annotations

import ctypes
import threading

import torch

from . import ssd

EXPORTED = ("m3_quat_workspace_bytes", "m3_quat_cumprod", "m3_quat_cumprod_backward", "m3_y_diag",
            "m3_y_diag_backward")

_lock = threading.Lock()
_bound = None


def _lib():
    global _bound
    with _lock:
        if _bound is None:
            lib = ssd.load_library()
            vp, sz, i32, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int64
            lib.m3_quat_workspace_bytes.argtypes = [i64] * 4 + [i32]
            lib.m3_quat_workspace_bytes.restype = sz
            lib.m3_quat_cumprod.argtypes = [vp] * 3 + [i64] * 4 + [vp, sz, vp]
            lib.m3_quat_cumprod.restype = i32
            lib.m3_quat_cumprod_backward.argtypes = [vp] * 5 + [i64] * 4 + [vp, sz, vp]
            lib.m3_quat_cumprod_backward.restype = i32
            lib.m3_y_diag.argtypes = [i32] + [vp] * 5 + [i64] * 5 + [vp]
            lib.m3_y_diag.restype = i32
            lib.m3_y_diag_backward.argtypes = [i32] + [vp] * 9 + [i64] * 5 + [vp]
            lib.m3_y_diag_backward.restype = i32
            _bound = lib
    return _bound


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _quat_check(q, init):
    if q.dim() != 5 or q.shape[-1] != 4 or q.dtype != torch.float32 or not q.is_contiguous() or not q.is_cuda:
        raise ValueError("q must be a contiguous CUDA float32 tensor [b, L, H, J, 4]")
    if init is not None:
        b, _, H, J, _ = q.shape
        if tuple(init.shape) != (b, H, J, 4) or init.dtype != torch.float32 or not init.is_contiguous():
            raise ValueError("init must be a contiguous float32 tensor [b, H, J, 4]")


def quat_workspace(q: torch.Tensor, backward: bool) -> torch.Tensor:
    b, L, H, J, _ = q.shape
    n = _lib().m3_quat_workspace_bytes(b, L, H, J, int(backward))
    return torch.empty(n, dtype=torch.uint8, device=q.device)


def quat_cumprod(q: torch.Tensor, init: torch.Tensor | None = None) -> torch.Tensor:
    """cum[:, t] = q[:, t] (x) cum[:, t-1] (Hamilton product), cum[:, -1] = init."""
    _quat_check(q, init)
    b, L, H, J, _ = q.shape
    cum = torch.empty_like(q)
    ws = quat_workspace(q, False)
    ssd._check(_lib().m3_quat_cumprod(_ptr(q), _ptr(init), _ptr(cum), b, L, H, J, _ptr(ws), ws.numel(),
                                      _stream(q.device)))
    return cum


def quat_cumprod_backward(q, init, d_cum, want_d_init=True):
    """The closed-form recompute backward; returns (d_q, d_init or None)."""
    _quat_check(q, init)
    if tuple(d_cum.shape) != tuple(q.shape) or d_cum.dtype != torch.float32 or not d_cum.is_contiguous():
        raise ValueError("d_cum must match q")
    b, L, H, J, _ = q.shape
    d_q = torch.empty_like(q)
    d_init = torch.empty(b, H, J, 4, device=q.device, dtype=torch.float32) if want_d_init else None
    ws = quat_workspace(q, True)
    ssd._check(_lib().m3_quat_cumprod_backward(_ptr(q), _ptr(init), _ptr(d_cum), _ptr(d_q), _ptr(d_init),
                                               b, L, H, J, _ptr(ws), ws.numel(), _stream(q.device)))
    return d_q, d_init


def _y_check(V, B, C, gamma):
    if V.dim() != 4 or B.dim() != 4 or tuple(B.shape[:3]) != tuple(V.shape[:3]) or B.shape != C.shape:
        raise ValueError("V [T, m, H, P], B and C [T, m, H, N]")
    if B.dtype != V.dtype or C.dtype != V.dtype or V.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("V, B, C must share a float32 or bfloat16 dtype")
    T, m, H, _ = V.shape
    if tuple(gamma.shape) != (T, H) or gamma.dtype != torch.float32:
        raise ValueError("gamma must be float32 [T, H]")
    for t in (V, B, C, gamma):
        if not t.is_contiguous() or not t.is_cuda:
            raise ValueError("tensors must be contiguous CUDA tensors")
    return ssd.SSD_F32 if V.dtype == torch.float32 else ssd.SSD_BF16


def y_diag(V, B, C, gamma):
    """y = gamma * (C B^T) V per token and head (MIMO rank m = V.shape[1])."""
    code = _y_check(V, B, C, gamma)
    T, m, H, P = V.shape
    N = B.shape[3]
    y = torch.empty_like(V)
    ssd._check(_lib().m3_y_diag(code, _ptr(V), _ptr(B), _ptr(C), _ptr(gamma), _ptr(y), T, m, H, P, N,
                                _stream(V.device)))
    return y


def y_diag_backward(dY, V, B, C, gamma):
    """Returns (dV, dB, dC, d_gamma)."""
    code = _y_check(V, B, C, gamma)
    if dY.shape != V.shape or dY.dtype != V.dtype or not dY.is_contiguous():
        raise ValueError("dY must match V")
    T, m, H, P = V.shape
    N = B.shape[3]
    dV, dB, dC = torch.empty_like(V), torch.empty_like(B), torch.empty_like(C)
    dg = torch.empty_like(gamma)
    ssd._check(_lib().m3_y_diag_backward(code, _ptr(dY), _ptr(V), _ptr(B), _ptr(C), _ptr(gamma), _ptr(dV),
                                         _ptr(dB), _ptr(dC), _ptr(dg), T, m, H, P, N, _stream(V.device)))
    return dV, dB, dC, dg
