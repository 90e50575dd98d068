"""Seeded synthetic inputs for the SSD selective scan.

This module holds no arithmetic of the method: it only draws random numbers
with the shapes and distributions of the five workloads the library is
measured on, so that the CUDA path, the CPU oracle, the tests and the
benchmark all consume identical inputs.  It imports numpy only.

Draw order (NumPy PCG64, ``default_rng(seed)``): x, B, C, dt_raw, A_raw, D,
init, dy, d_final, valid_len.  Every array is drawn in fp32; the tensors the
workload stores in bf16 (x, B, C, dy) are rounded to bf16 values here, so the
oracle and the GPU see the same numbers.

Distributions:  x, B, C, dy ~ N(0, 1);  dt = softplus(N(mu, 1)) with mu = -2
(mu = -3 for the long-sequence workload);  A = -exp(U(0, ln 16));  D ~ N(0, 1);
init = 0, or N(0, 0.1^2) for the grouped workload;  d_final ~ N(0, 1) for the
tiny and grouped workloads, 0 otherwise;  valid_len = L, or U{1024..4096} per
sample for the grouped workload, whose x, B, C, dy tails past valid_len are
zeroed (the dt tail is left as drawn).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk_len: int
    dtype: str            # "f32" or "bf16": storage type of x, B, C, dy, y, dx, dB, dC
    dt_mu: float = -2.0
    init_std: float = 0.0
    d_final_std: float = 0.0
    ragged: bool = False  # per-sample valid_len ~ U{1024..seqlen}, tails zeroed
    seed: int = 1000

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen

    def dims(self) -> dict:
        return dict(batch=self.batch, seqlen=self.seqlen, nheads=self.nheads,
                    headdim=self.headdim, dstate=self.dstate, ngroups=self.ngroups,
                    chunk_len=self.chunk_len)

    def scaled(self, **kw) -> "Workload":
        d = {k: getattr(self, k) for k in self.__dataclass_fields__}
        d.update(kw)
        return Workload(**d)


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 1, 64, 2, 8, 8, 1, 16, "f32", d_final_std=1.0, seed=1000),
    "mamba2_130m": Workload("mamba2_130m", 4, 2048, 24, 64, 128, 1, 256, "bf16", seed=1001),
    "mamba2_2p7b": Workload("mamba2_2p7b", 2, 8192, 80, 64, 128, 1, 256, "bf16", seed=1002),
    "grouped_padded": Workload("grouped_padded", 8, 4096, 64, 64, 128, 8, 256, "bf16",
                               init_std=0.1, d_final_std=1.0, ragged=True, seed=1003),
    "long_seq": Workload("long_seq", 1, 131072, 32, 64, 128, 1, 256, "bf16", dt_mu=-3.0,
                         seed=1004),
}


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 value (ties to even), kept in fp32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _softplus(z: np.ndarray) -> np.ndarray:
    return np.logaddexp(np.float32(0.0), z).astype(np.float32)


def generate(w: Workload, seed: int | None = None) -> dict:
    """Draw one set of inputs (and upstream gradients) for workload ``w``.

    Returns fp32 numpy arrays in the library's layouts: x, dy [b,L,H,P];
    dt [b,H,L]; A, D [H]; B, C [b,L,G,N]; init, d_final [b,H,P,N] (or None when
    identically zero); valid_len int32 [b] (or None when every sample is full).
    """
    rng = np.random.default_rng(w.seed if seed is None else seed)
    b, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    f32 = np.float32
    x = rng.standard_normal((b, L, H, P), dtype=f32)
    B = rng.standard_normal((b, L, G, N), dtype=f32)
    C = rng.standard_normal((b, L, G, N), dtype=f32)
    dt = _softplus(rng.standard_normal((b, H, L), dtype=f32) + f32(w.dt_mu))
    A = (-np.exp(rng.uniform(0.0, np.log(16.0), H))).astype(f32)
    D = rng.standard_normal(H, dtype=f32)
    init = rng.standard_normal((b, H, P, N), dtype=f32) * f32(w.init_std)
    dy = rng.standard_normal((b, L, H, P), dtype=f32)
    d_final = rng.standard_normal((b, H, P, N), dtype=f32) * f32(w.d_final_std)
    valid_len = None
    if w.ragged:
        lo = min(1024, L)
        valid_len = rng.integers(lo, L, size=b, endpoint=True).astype(np.int32)
        tail = np.arange(L)[None, :] >= valid_len[:, None]
        for a in (x, dy):
            a[tail] = 0.0
        for a in (B, C):
            a[tail] = 0.0
    if w.dtype == "bf16":
        x, B, C, dy = (round_to_bf16(a) for a in (x, B, C, dy))
    return dict(x=x, dt=dt, A=A, B=B, C=C, D=D,
                init=init if w.init_std != 0.0 else None,
                dy=dy, d_final=d_final if w.d_final_std != 0.0 else None,
                valid_len=valid_len)


def generate_small(b, L, H, P, N, G, seed=0, dt_mu=-2.0, init_std=0.0, d_final_std=1.0,
                   valid_len=None, bf16=False) -> dict:
    """Same distributions at an arbitrary small shape (for unit tests)."""
    w = Workload("custom", b, L, H, P, N, G, 16, "bf16" if bf16 else "f32", dt_mu=dt_mu,
                 init_std=init_std, d_final_std=d_final_std, seed=seed)
    out = generate(w)
    if valid_len is not None:
        out["valid_len"] = np.asarray(valid_len, np.int32)
    return out


# ---------------------------------------------------------------- Mamba-3 pieces
# Quaternion scan: per step a unit quaternion (cos(phi/2), sin(phi/2) u) with a
# uniformly random axis u and phi ~ N(0, angle_std^2), drawn in fp64 and stored
# in fp32; init a random unit quaternion; d_cum ~ N(0, 1).  Draw order: axis,
# phi, init axis, init angle, d_cum.
# Gamma correction: V, B, C, dY ~ N(0, 1) (rounded to bf16 values when the
# workload stores bf16), gamma ~ U(0, 1).  Draw order: V, B, C, gamma, dY.
@dataclass(frozen=True)
class QuatWorkload:
    name: str
    batch: int
    seqlen: int
    nheads: int
    nblocks: int           # quaternion blocks per head (J)
    angle_std: float = 0.3
    seed: int = 2000

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen


@dataclass(frozen=True)
class DiagWorkload:
    name: str
    tokens: int            # the page's (b, n, l) axes flattened
    mimo: int              # m
    nheads: int
    headdim: int
    dstate: int
    dtype: str = "bf16"
    seed: int = 3000


# at the Mamba-2 2.7B layer's token count (2 x 8192) and head count
MAMBA3_WORKLOADS = {
    "quat_scan_2p7b": QuatWorkload("quat_scan_2p7b", 2, 8192, 80, 8, seed=2001),
    "ydiag_siso_2p7b": DiagWorkload("ydiag_siso_2p7b", 16384, 1, 80, 64, 128, seed=3001),
    "ydiag_mimo4": DiagWorkload("ydiag_mimo4", 16384, 4, 16, 64, 128, seed=3002),
}


def _unit_quaternions(rng, shape, angle_std):
    axis = rng.standard_normal(shape + (3,))
    axis /= np.linalg.norm(axis, axis=-1, keepdims=True)
    phi = rng.standard_normal(shape) * angle_std
    q = np.concatenate([np.cos(phi / 2)[..., None], np.sin(phi / 2)[..., None] * axis], axis=-1)
    return q.astype(np.float32)


def generate_quat(w: QuatWorkload, seed: int | None = None) -> dict:
    """q, d_cum [b, L, H, J, 4] and init [b, H, J, 4], fp32."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    b, L, H, J = w.batch, w.seqlen, w.nheads, w.nblocks
    q = _unit_quaternions(rng, (b, L, H, J), w.angle_std)
    init = _unit_quaternions(rng, (b, H, J), 1.0)
    d_cum = rng.standard_normal((b, L, H, J, 4), dtype=np.float32)
    return dict(q=q, init=init, d_cum=d_cum)


def generate_diag(w: DiagWorkload, seed: int | None = None) -> dict:
    """V, dY [T, m, H, P]; B, C [T, m, H, N]; gamma [T, H]; fp32 arrays."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    T, m, H, P, N = w.tokens, w.mimo, w.nheads, w.headdim, w.dstate
    f32 = np.float32
    V = rng.standard_normal((T, m, H, P), dtype=f32)
    B = rng.standard_normal((T, m, H, N), dtype=f32)
    C = rng.standard_normal((T, m, H, N), dtype=f32)
    gamma = rng.uniform(0.0, 1.0, (T, H)).astype(f32)
    dY = rng.standard_normal((T, m, H, P), dtype=f32)
    if w.dtype == "bf16":
        V, B, C, dY = (round_to_bf16(a) for a in (V, B, C, dY))
    return dict(V=V, B=B, C=C, gamma=gamma, dY=dY)
