"""CPU oracle for the Mamba-2 SSD selective scan -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never imports, links
or calls it, and it imports nothing from the CUDA package.

Two independent CPU implementations live here:

* :func:`forward` / :func:`backward` -- the plain token-by-token recurrence in
  fp64 C (``ssd_oracle.c``), the definition that the GPU path must match.
* :mod:`oracle.chunked` -- a NumPy fp64 restatement of the pages' chunked
  five-kernel forward and recompute backward (burn-mamba,
  ``combined_backward.rs``), used only to pin the serial oracle to the pages'
  structure and to check the pages' identities.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libssd_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc + OpenMP into ``oracle/_build``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    i64, dp, ip = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
    lib.ssd_oracle_forward.argtypes = [i64] * 6 + [dp] * 7 + [ip, dp, dp, ctypes.c_int]
    lib.ssd_oracle_forward.restype = ctypes.c_int
    lib.ssd_oracle_backward.argtypes = ([i64] * 6 + [dp] * 7 + [ip] + [dp] * 2
                                        + [dp] * 7 + [ctypes.c_int])
    lib.ssd_oracle_backward.restype = ctypes.c_int
    lib.ssd_oracle_num_threads.restype = ctypes.c_int
    lib.ssd_oracle_state_moments.argtypes = [i64] * 6 + [dp] * 5 + [ip, dp, dp, ctypes.c_int]
    lib.ssd_oracle_state_moments.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def compile_variant(source_text: str, out_dir: str) -> "ctypes.CDLL":
    """Compile an edited copy of the oracle's C source (used by the tests that
    plant a mistake in the oracle to show that its pins catch it)."""
    os.makedirs(out_dir, exist_ok=True)
    src = os.path.join(out_dir, "variant.c")
    lib = os.path.join(out_dir, "libvariant.so")
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", lib, src,
                    "-lm"], check=True)
    return _bind(ctypes.CDLL(lib))


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def num_threads() -> int:
    """Threads the oracle uses by default (OpenMP's default team size)."""
    return int(_load().ssd_oracle_num_threads())


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dims(x, B, ngroups):
    nb, L, H, P = x.shape
    N = B.shape[-1]
    G = ngroups if ngroups is not None else B.shape[2]
    return nb, L, H, P, N, G


def forward(x, dt, A, B, C, D, init=None, valid_len=None, nthreads=0, lib=None):
    """Serial recurrence forward.  Returns ``(y, final_state)`` as fp64 arrays.

    Shapes: x [b,L,H,P], dt [b,H,L], A [H], B/C [b,L,G,N], D [H],
    init [b,H,P,N] or None (zeros), valid_len int [b] or None (= L).
    """
    x, dt, A, B, C, D, init = map(_f64, (x, dt, A, B, C, D, init))
    nb, L, H, P, N, G = _dims(x, B, None)
    vl = None if valid_len is None else np.ascontiguousarray(valid_len, dtype=np.int32)
    y = np.empty((nb, L, H, P), np.float64)
    fin = np.empty((nb, H, P, N), np.float64)
    rc = (lib or _load()).ssd_oracle_forward(nb, L, H, P, N, G, _ptr(x), _ptr(dt), _ptr(A), _ptr(B),
                                    _ptr(C), _ptr(D), _ptr(init), _ptr(vl), _ptr(y), _ptr(fin),
                                    int(nthreads))
    if rc != 0:
        raise RuntimeError(f"ssd_oracle_forward failed with code {rc}")
    return y, fin


def backward(x, dt, A, B, C, D, init, valid_len, dy, d_final=None, nthreads=0, lib=None):
    """Reverse mode of the serial recurrence for Loss = <dy, y> + <d_final, final>.

    Returns a dict with dx, ddt, dA, dB, dC, dD, d_init (fp64).
    """
    x, dt, A, B, C, D, init, dy, d_final = map(_f64, (x, dt, A, B, C, D, init, dy, d_final))
    nb, L, H, P, N, G = _dims(x, B, None)
    vl = None if valid_len is None else np.ascontiguousarray(valid_len, dtype=np.int32)
    out = {
        "dx": np.empty((nb, L, H, P)), "ddt": np.empty((nb, H, L)), "dA": np.empty(H),
        "dB": np.empty((nb, L, G, N)), "dC": np.empty((nb, L, G, N)), "dD": np.empty(H),
        "d_init": np.empty((nb, H, P, N)),
    }
    rc = (lib or _load()).ssd_oracle_backward(
        nb, L, H, P, N, G, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init),
        _ptr(vl), _ptr(dy), _ptr(d_final), _ptr(out["dx"]), _ptr(out["ddt"]), _ptr(out["dA"]),
        _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]), _ptr(out["d_init"]), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"ssd_oracle_backward failed with code {rc}")
    return out


def state_moments(x, dt, A, B, init=None, valid_len=None, nthreads=0, lib=None):
    """Raw moments of the per-token states (the states after each valid token):
    m2 [b,H,N,N] = sum_t S_t^T S_t, m1 [b,H,N] = sum_t sum_p S_t[p,:], and the
    sample count per sample, valid_len * P (int64 [b])."""
    x, dt, A, B, init = map(_f64, (x, dt, A, B, init))
    nb, L, H, P, N, G = _dims(x, B, None)
    vl = None if valid_len is None else np.ascontiguousarray(valid_len, dtype=np.int32)
    m2 = np.empty((nb, H, N, N), np.float64)
    m1 = np.empty((nb, H, N), np.float64)
    rc = (lib or _load()).ssd_oracle_state_moments(nb, L, H, P, N, G, _ptr(x), _ptr(dt), _ptr(A), _ptr(B),
                                                   _ptr(init), _ptr(vl), _ptr(m2), _ptr(m1), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"ssd_oracle_state_moments failed with code {rc}")
    V = np.full(nb, L, np.int64) if vl is None else np.clip(vl.astype(np.int64), 0, L)
    return m2, m1, V * P


def loss(y, final, dy, d_final):
    """Scalar whose gradient :func:`backward` returns."""
    s = float(np.sum(np.asarray(dy, np.float64) * y))
    if d_final is not None:
        s += float(np.sum(np.asarray(d_final, np.float64) * final))
    return s
