"""Thin Python binding of ``libssd.so`` (the C ABI in ``include/ssd.h``).

Argument marshalling only: every step of the selective scan runs in the CUDA
kernels behind the ABI.  Tensors are torch CUDA tensors (PyTorch supplies
device memory and streams); the binding checks dtypes and shapes, allocates
outputs and workspace with torch, and passes raw device pointers plus the
current CUDA stream.  There is no fallback: if the library is missing or a
call fails, a RuntimeError is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libssd.so")

SSD_F32, SSD_BF16 = 0, 1
SSD_FLAG_SIMT = 1
SSD_FLAG_CHECK_FINITE = 2
SSD_FLAG_SPLIT_SCAN = 4
SSD_OK, SSD_ERR_INVALID_ARG, SSD_ERR_UNSUPPORTED, SSD_ERR_WORKSPACE = 0, 1, 2, 3
SSD_ERR_CUDA, SSD_ERR_TIMEOUT, SSD_ERR_NONFINITE = 4, 5, 6
STATUS = {0: "SSD_OK", 1: "SSD_ERR_INVALID_ARG", 2: "SSD_ERR_UNSUPPORTED",
          3: "SSD_ERR_WORKSPACE", 4: "SSD_ERR_CUDA", 5: "SSD_ERR_TIMEOUT", 6: "SSD_ERR_NONFINITE"}
EXPORTED = ("ssd_supported", "ssd_workspace_bytes", "ssd_forward", "ssd_backward",
            "ssd_workspace_status", "ssd_status_str", "ssd_last_error", "ssd_version",
            "ssd_last_launch_count", "ssd_profile_begin", "ssd_profile_end", "ssd_profile_name",
            "ssd_profile_only", "ssd_forward_noalloc", "ssd_noalloc_status",
            "ssd_moments_workspace_bytes", "ssd_state_moments", "ssd_state_pr", "ssd_wait_selftest")
SSD_PAIR_REAL, SSD_PAIR_COMPLEX_INTERLEAVED, SSD_PAIR_COMPLEX_HALF_HALF, SSD_PAIR_QUATERNION = 0, 1, 2, 3


class SsdDims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64),
                ("nheads", ctypes.c_int64), ("headdim", ctypes.c_int64),
                ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64),
                ("chunk_len", ctypes.c_int64), ("flags", ctypes.c_uint32),
                ("reserved", ctypes.c_uint32)]


class SsdError(RuntimeError):
    def __init__(self, code: int, detail: str):
        super().__init__(f"{STATUS.get(code, code)}: {detail}")
        self.code = code


_lock = threading.Lock()
_lib = None


def load_library(path: str | None = None):
    """Open libssd.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with "
                               "`python -m state_space_model_mamba_gb300.build`")
        import torch.cuda  # noqa: F401  (makes the CUDA runtime PyTorch uses resident first)
        lib = ctypes.CDLL(p)
        vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        dims_p = ctypes.POINTER(SsdDims)
        lib.ssd_supported.argtypes = [dims_p, i32]
        lib.ssd_supported.restype = i32
        lib.ssd_workspace_bytes.argtypes = [dims_p, i32, i32]
        lib.ssd_workspace_bytes.restype = sz
        lib.ssd_forward.argtypes = [dims_p, i32] + [vp] * 10 + [vp, sz, vp]
        lib.ssd_forward.restype = i32
        lib.ssd_backward.argtypes = [dims_p, i32] + [vp] * 17 + [vp, sz, vp]
        lib.ssd_backward.restype = i32
        lib.ssd_workspace_status.argtypes = [vp, sz, vp]
        lib.ssd_workspace_status.restype = i32
        lib.ssd_wait_selftest.argtypes = [vp, sz, ctypes.c_uint32, i32, vp]
        lib.ssd_wait_selftest.restype = i32
        lib.ssd_status_str.argtypes = [i32]
        lib.ssd_status_str.restype = ctypes.c_char_p
        lib.ssd_last_error.restype = ctypes.c_char_p
        lib.ssd_version.restype = i32
        lib.ssd_last_launch_count.restype = i32
        lib.ssd_profile_begin.argtypes = [vp, i32]
        lib.ssd_profile_begin.restype = i32
        lib.ssd_profile_end.restype = i32
        lib.ssd_profile_name.argtypes = [i32]
        lib.ssd_profile_name.restype = ctypes.c_char_p
        lib.ssd_profile_only.argtypes = [ctypes.c_char_p]
        lib.ssd_profile_only.restype = None
        lib.ssd_forward_noalloc.argtypes = [dims_p, i32] + [vp] * 10 + [vp]
        lib.ssd_forward_noalloc.restype = i32
        lib.ssd_noalloc_status.argtypes = [vp]
        lib.ssd_noalloc_status.restype = i32
        lib.ssd_moments_workspace_bytes.argtypes = [dims_p, i32]
        lib.ssd_moments_workspace_bytes.restype = sz
        lib.ssd_state_moments.argtypes = [dims_p, i32] + [vp] * 9 + [vp, sz, vp]
        lib.ssd_state_moments.restype = i32
        i64 = ctypes.c_int64
        lib.ssd_state_pr.argtypes = [vp] * 3 + [i64] * 3 + [i32, i32, i64, i32, vp, vp, vp]
        lib.ssd_state_pr.restype = i32
        if path is None:
            _lib = lib
        return lib


def _check(code: int):
    if code != 0:
        raise SsdError(code, load_library().ssd_last_error().decode())


@dataclass(frozen=True)
class Dims:
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk_len: int
    simt: bool = False
    check_finite: bool = False
    split_scan: bool = False

    def c(self) -> SsdDims:
        flags = ((SSD_FLAG_SIMT if self.simt else 0) | (SSD_FLAG_CHECK_FINITE if self.check_finite else 0)
                 | (SSD_FLAG_SPLIT_SCAN if self.split_scan else 0))
        return SsdDims(self.batch, self.seqlen, self.nheads, self.headdim, self.dstate,
                       self.ngroups, self.chunk_len, flags, 0)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SSD_F32
    if t.dtype == torch.bfloat16:
        return SSD_BF16
    raise TypeError(f"x must be float32 or bfloat16, got {t.dtype}")


def dims_of(x: torch.Tensor, B: torch.Tensor, chunk_len: int, simt: bool = False,
            check_finite: bool = False, split_scan: bool = False) -> Dims:
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    return Dims(b, L, H, P, N, G, int(chunk_len), simt, check_finite, split_scan)


def supported(dims: Dims, dtype_code: int) -> bool:
    return load_library().ssd_supported(ctypes.byref(dims.c()), dtype_code) == 0


def workspace_bytes(dims: Dims, dtype_code: int, backward: bool) -> int:
    n = load_library().ssd_workspace_bytes(ctypes.byref(dims.c()), dtype_code, int(backward))
    if n == 0:
        _check(load_library().ssd_supported(ctypes.byref(dims.c()), dtype_code) or 1)
    return int(n)


def alloc_workspace(dims: Dims, dtype_code: int, backward: bool, device) -> torch.Tensor:
    return torch.empty(workspace_bytes(dims, dtype_code, backward), dtype=torch.uint8, device=device)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check_inputs(x, dt, A, B, C, D, init_state, valid_len, T):
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    exp = {"dt": (dt, (b, H, L), torch.float32), "A": (A, (H,), torch.float32),
           "B": (B, (b, L, G, N), T), "C": (C, (b, L, G, N), T), "D": (D, (H,), torch.float32)}
    if init_state is not None:
        exp["init_state"] = (init_state, (b, H, P, N), torch.float32)
    for name, (t, shape, dtype) in exp.items():
        if tuple(t.shape) != shape or t.dtype != dtype:
            raise ValueError(f"{name}: expected {shape} {dtype}, got {tuple(t.shape)} {t.dtype}")
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor")
    if valid_len is not None and (valid_len.dtype != torch.int32 or tuple(valid_len.shape) != (b,)
                                  or not valid_len.is_cuda):
        raise ValueError("valid_len must be a CUDA int32 tensor of shape [batch]")


def forward_into(dims: Dims, x, dt, A, B, C, D, init_state, valid_len, y, final_state,
                 workspace: torch.Tensor):
    """ssd_forward on caller-provided outputs and workspace (no allocation)."""
    code = _dtype_code(x)
    _check(load_library().ssd_forward(
        ctypes.byref(dims.c()), code, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
        _ptr(init_state), _ptr(valid_len), _ptr(y), _ptr(final_state), _ptr(workspace),
        workspace.numel(), _stream_ptr(x.device)))


def backward_into(dims: Dims, x, dt, A, B, C, D, init_state, valid_len, dy, d_final, dx, ddt,
                  dA, dB, dC, dD, d_init, workspace: torch.Tensor):
    """ssd_backward on caller-provided gradients and workspace (no allocation)."""
    code = _dtype_code(x)
    _check(load_library().ssd_backward(
        ctypes.byref(dims.c()), code, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
        _ptr(init_state), _ptr(valid_len), _ptr(dy), _ptr(d_final), _ptr(dx), _ptr(ddt), _ptr(dA),
        _ptr(dB), _ptr(dC), _ptr(dD), _ptr(d_init), _ptr(workspace), workspace.numel(),
        _stream_ptr(x.device)))


def ssd_forward(x, dt, A, B, C, D, chunk_len, init_state=None, valid_len=None,
                return_final_state=True, simt=False, check_finite=False, check_status=False,
                split_scan=False):
    """Forward of the chunked selective scan.  Returns ``(y, final_state)``.

    x [b,L,H,P] (fp32 or bf16), dt [b,H,L] fp32, A [H] fp32, B/C [b,L,G,N]
    (x's dtype), D [H] fp32, init_state [b,H,P,N] fp32 or None,
    valid_len int32 [b] or None.  ``check_finite`` sets SSD_FLAG_CHECK_FINITE;
    with it or ``check_status`` the call synchronises and raises SsdError when
    the device reported a condition (timeout, non-finite values, clamped
    valid_len entries).  ``split_scan`` sets SSD_FLAG_SPLIT_SCAN (chunk states by
    the chunk-parallel K3 and a separate K4 pass instead of the fused scan).
    """
    _check_inputs(x, dt, A, B, C, D, init_state, valid_len, x.dtype)
    dims = dims_of(x, B, chunk_len, simt, check_finite, split_scan)
    code = _dtype_code(x)
    y = torch.empty_like(x)
    fin = (torch.empty(x.shape[0], x.shape[2], x.shape[3], B.shape[3], device=x.device,
                       dtype=torch.float32) if return_final_state else None)
    ws = alloc_workspace(dims, code, False, x.device)
    forward_into(dims, x, dt, A, B, C, D, init_state, valid_len, y, fin, ws)
    if check_finite or check_status:
        workspace_status(ws)
    return y, fin


def ssd_backward(x, dt, A, B, C, D, chunk_len, dy, d_final_state=None, init_state=None,
                 valid_len=None, want_d_init=True, simt=False, check_finite=False, split_scan=False,
                 check_status=False):
    """Recompute backward.  Returns a dict with dx, ddt, dA, dB, dC, dD, d_init.
    ``check_finite`` / ``check_status`` as in :func:`ssd_forward`."""
    _check_inputs(x, dt, A, B, C, D, init_state, valid_len, x.dtype)
    if tuple(dy.shape) != tuple(x.shape) or dy.dtype != x.dtype or not dy.is_contiguous():
        raise ValueError("dy must match x in shape and dtype and be contiguous")
    dims = dims_of(x, B, chunk_len, simt, check_finite, split_scan)
    code = _dtype_code(x)
    b, L, H, P = x.shape
    N = B.shape[3]
    dev = x.device
    out = dict(dx=torch.empty_like(x), ddt=torch.empty_like(dt), dA=torch.empty_like(A),
               dB=torch.empty_like(B), dC=torch.empty_like(C), dD=torch.empty_like(D),
               d_init=(torch.empty(b, H, P, N, device=dev, dtype=torch.float32)
                       if want_d_init else None))
    ws = alloc_workspace(dims, code, True, dev)
    backward_into(dims, x, dt, A, B, C, D, init_state, valid_len, dy, d_final_state, out["dx"],
                  out["ddt"], out["dA"], out["dB"], out["dC"], out["dD"], out["d_init"], ws)
    if check_finite or check_status:
        workspace_status(ws)
    return out


def state_moments(x, dt, A, B, init_state=None, valid_len=None, check_status=False, split_scan=False):
    """Raw moments of the per-token states: returns (m2 [b,H,N,N], m1 [b,H,N],
    count int64 [b]).  x, B bf16; dt, A, init fp32 (as ssd_forward)."""
    _check_inputs(x, dt, A, B, B, A, init_state, valid_len, x.dtype)
    dims = dims_of(x, B, 128, split_scan=split_scan)
    code = _dtype_code(x)
    b, L, H, P = x.shape
    N = B.shape[3]
    dev = x.device
    m2 = torch.empty(b, H, N, N, device=dev, dtype=torch.float32)
    m1 = torch.empty(b, H, N, device=dev, dtype=torch.float32)
    count = torch.empty(b, device=dev, dtype=torch.int64)
    lib = load_library()
    n = lib.ssd_moments_workspace_bytes(ctypes.byref(dims.c()), code)
    if n == 0:
        _check(lib.ssd_supported(ctypes.byref(dims.c()), code) or SSD_ERR_UNSUPPORTED)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    _check(lib.ssd_state_moments(ctypes.byref(dims.c()), code, _ptr(x), _ptr(dt), _ptr(A), _ptr(B),
                                 _ptr(init_state), _ptr(valid_len), _ptr(m2), _ptr(m1), _ptr(count),
                                 _ptr(ws), ws.numel(), _stream_ptr(dev)))
    if check_status:
        workspace_status(ws)
    return m2, m1, count


def state_pr(m2, m1, count, center=False, pairing=SSD_PAIR_REAL, num=0, pool_batch=False):
    """Participation ratio [b or 1, H] and trace of pooled state moments."""
    b, H, N, _ = m2.shape
    nb = 1 if pool_batch else b
    pr = torch.empty(nb, H, device=m2.device, dtype=torch.float32)
    tr = torch.empty(nb, H, device=m2.device, dtype=torch.float32)
    _check(load_library().ssd_state_pr(_ptr(m2), _ptr(m1), _ptr(count), b, H, N, int(center), int(pairing),
                                       int(num), int(pool_batch), _ptr(pr), _ptr(tr), _stream_ptr(m2.device)))
    return pr, tr


def workspace_status(workspace: torch.Tensor) -> None:
    """Raise SsdError if the last call on ``workspace`` recorded a device-side
    condition: a timeout, non-finite values (SSD_FLAG_CHECK_FINITE) or clamped
    valid_len entries.  Synchronises the current stream."""
    _check(load_library().ssd_workspace_status(_ptr(workspace), workspace.numel(),
                                               _stream_ptr(workspace.device)))


def wait_selftest(workspace: torch.Tensor, limit_us: int, arrive: bool) -> None:
    """Run the kernels' bounded device wait on a barrier that one arrival
    completes (``arrive``) or that nothing completes, giving up after
    ``limit_us`` microseconds; :func:`workspace_status` then reports the
    timeout (ssd_wait_selftest)."""
    _check(load_library().ssd_wait_selftest(_ptr(workspace), workspace.numel(), int(limit_us), int(arrive),
                                            _stream_ptr(workspace.device)))


def noalloc_status(device=None) -> None:
    """Raise SsdError if the last ssd_forward_noalloc call on the current
    device recorded a device-side condition (as :func:`workspace_status`)."""
    _check(load_library().ssd_noalloc_status(_stream_ptr(device)))


def last_launch_count() -> int:
    """Kernels enqueued by the most recent forward/backward call on this thread."""
    return int(load_library().ssd_last_launch_count())


class KernelTimer:
    """Records a CUDA-event pair around every kernel the library launches while
    active (on the launching stream).  ``durations()`` returns a list of
    (kernel name, milliseconds) in launch order after a synchronize."""

    def __init__(self, capacity_kernels: int, only: str | None = None):
        self.only = only  # record only the kernel of this name (None: every kernel)
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * capacity_kernels)]
        for e in self.events:
            e.record()  # materialise the underlying cudaEvent_t
        torch.cuda.synchronize()
        self._arr = (ctypes.c_void_p * len(self.events))(*[e.cuda_event for e in self.events])
        self.n = 0

    def __enter__(self):
        lib = load_library()
        lib.ssd_profile_only(self.only.encode() if self.only else None)
        _check(lib.ssd_profile_begin(self._arr, len(self.events)))
        return self

    def __exit__(self, *exc):
        lib = load_library()
        self.n = int(lib.ssd_profile_end())
        lib.ssd_profile_only(None)
        return False

    def names(self, count: int) -> list:
        lib = load_library()
        return [lib.ssd_profile_name(i).decode() for i in range(min(count, 4096))]

    def durations(self, pattern: list | None = None) -> list:
        """(name, ms) per recorded kernel.  Names past the library's 4096-entry
        name table are taken from ``pattern`` (the per-step launch sequence)."""
        torch.cuda.synchronize()
        k = self.n // 2
        names = self.names(k)
        out = []
        for i in range(k):
            if self.only:
                nm = self.only
            elif pattern:
                nm = pattern[i % len(pattern)]
            else:
                nm = names[i] if i < len(names) else ""
            out.append((nm, self.events[2 * i].elapsed_time(self.events[2 * i + 1])))
        return out
