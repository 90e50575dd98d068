"""Host-side checks of the C ABI (no GPU): the library loads, exports every
function that include/ssd.h declares, sizes workspaces, and rejects bad
arguments before enqueuing any device work."""
import ctypes
import os
import re

import pytest

from state_space_model_mamba_gb300 import build as ssd_build
from state_space_model_mamba_gb300 import ssd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    ssd_build.build()
    return ssd.load_library()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b((?:ssd|m3)_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(ssd.EXPORTED) <= set(names)
    from state_space_model_mamba_gb300 import mamba3
    assert set(mamba3.EXPORTED) <= set(names)


def test_mamba3_calls_reject_bad_arguments_before_launch(lib):
    from state_space_model_mamba_gb300 import mamba3
    m = mamba3._lib()
    buf = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails validation first
    # one quaternion per (sample, 32-step segment, chain); three arrays of them for the backward
    assert m.m3_quat_workspace_bytes(2, 300, 3, 2, 0) == 2 * 10 * 6 * 16
    assert m.m3_quat_workspace_bytes(2, 300, 3, 2, 1) == 3 * 2 * 10 * 6 * 16
    assert m.m3_quat_workspace_bytes(0, 300, 3, 2, 0) == 0
    assert m.m3_quat_cumprod(None, None, buf, 1, 8, 1, 1, buf, 1 << 20, None) == ssd.SSD_ERR_INVALID_ARG
    assert m.m3_quat_cumprod(buf, None, buf, 1, 0, 1, 1, buf, 1 << 20, None) == ssd.SSD_ERR_INVALID_ARG
    assert m.m3_quat_cumprod(buf, None, buf, 1, 300, 1, 1, buf, 16, None) == ssd.SSD_ERR_WORKSPACE
    assert m.m3_quat_cumprod_backward(buf, None, ctypes.c_void_p((1 << 20) + 4), buf, None, 1, 8, 1, 1, buf,
                                      1 << 20, None) == ssd.SSD_ERR_INVALID_ARG
    args = [buf] * 5
    assert m.m3_y_diag(ssd.SSD_BF16, *args, 4, 5, 2, 64, 128, None) == ssd.SSD_ERR_UNSUPPORTED
    assert m.m3_y_diag(ssd.SSD_BF16, *args, 4, 1, 2, 63, 128, None) == ssd.SSD_ERR_UNSUPPORTED
    assert m.m3_y_diag(7, *args, 4, 1, 2, 64, 128, None) == ssd.SSD_ERR_INVALID_ARG
    assert m.m3_y_diag_backward(ssd.SSD_F32, *([buf] * 8), None, 4, 1, 2, 64, 128, None) == ssd.SSD_ERR_INVALID_ARG
    assert b"NULL" in lib.ssd_last_error()


def test_version_and_status_strings(lib):
    assert lib.ssd_version() >= 10000
    for code in range(7):
        assert lib.ssd_status_str(code) and lib.ssd_status_str(code) != b"unknown status"
    assert lib.ssd_status_str(99) == b"unknown status"


def _dims(**kw):
    base = dict(batch=2, seqlen=8192, nheads=80, headdim=64, dstate=128, ngroups=1, chunk_len=256)
    base.update(kw)
    return ssd.SsdDims(base["batch"], base["seqlen"], base["nheads"], base["headdim"],
                       base["dstate"], base["ngroups"], base["chunk_len"],
                       base.get("flags", 0), base.get("reserved", 0))


def test_workspace_sizes(lib):
    d = _dims()
    f = lib.ssd_workspace_bytes(ctypes.byref(d), ssd.SSD_BF16, 0)
    b = lib.ssd_workspace_bytes(ctypes.byref(d), ssd.SSD_BF16, 1)
    states_bf16 = 2 * 32 * 80 * 64 * 128 * 2       # tensor-core path stores chunk states in bf16
    assert f >= states_bf16 and b >= 2 * states_bf16 and b > f
    simt = _dims(flags=ssd.SSD_FLAG_SIMT)          # CUDA-core path keeps them in fp32
    assert lib.ssd_workspace_bytes(ctypes.byref(simt), ssd.SSD_BF16, 1) >= 4 * states_bf16
    assert lib.ssd_workspace_bytes(ctypes.byref(_dims(ngroups=3)), ssd.SSD_BF16, 0) == 0
    # ragged sequence length rounds the chunk count up
    r = lib.ssd_workspace_bytes(ctypes.byref(_dims(seqlen=8193)), ssd.SSD_BF16, 0)
    assert r > f


def _forward_workspace(b, L, H, P, N, Q, fp32_states):
    """The forward's workspace as documented: 256-byte aligned regions for the
    status words, (segmented state passing only) its ticket counter and ready
    flags, per-segment reductions, group carries and decays, then cumA, endA,
    the CB region (CUDA-core path only) and the chunk states."""
    al = lambda v: (v + 255) // 256 * 256
    n = -(-L // Q)
    slices = -(-(P * N // 16) // 128)
    pairs = b * H * slices
    T = 4 if fp32_states else 8
    K = -(-n // T)
    KG = -(-K // 8)
    seg = (P * N) % 2048 == 0 and pairs <= 304 and K >= 2
    total = al(16)
    if seg:
        total += al(4 * (64 + pairs * (K + KG))) + al(4 * pairs * K * 2048) + al(4 * pairs * KG * 2048) + al(4 * pairs * K)
    total += al(4 * b * H * n * Q) + al(4 * b * H * n)
    if fp32_states:
        total += al(4 * b * n * Q * Q)                       # fp32 CB, one group
    total += al((4 if fp32_states else 2) * b * n * H * P * N)
    return total, seg


@pytest.mark.parametrize("shape", [
    dict(batch=1, seqlen=131072, nheads=32),                 # 32 chains of 512 chunks: segmented
    dict(batch=1, seqlen=131072, nheads=32, flags=ssd.SSD_FLAG_SIMT),  # fp32 states: segmented
    dict(batch=1, seqlen=131072, nheads=76),                 # 304 blocks: segmented
    dict(batch=1, seqlen=131072, nheads=80),                 # 320 blocks: chunk-serial
    dict(batch=1, seqlen=2048, nheads=2),                    # one segment per chain: chunk-serial
    # P * N below one slice (and outside the tensor-core shapes: fp32 states): chunk-serial
    dict(batch=1, seqlen=8192, nheads=2, headdim=32, dstate=32),
])
def test_forward_workspace_layout_and_segmented_state_passing(lib, shape):
    kw = dict(shape)
    d = _dims(**kw)
    simt = bool(kw.get("flags", 0) & ssd.SSD_FLAG_SIMT) or (d.headdim, d.dstate) != (64, 128)
    want, seg = _forward_workspace(d.batch, d.seqlen, d.nheads, d.headdim, d.dstate, d.chunk_len, simt)
    assert lib.ssd_workspace_bytes(ctypes.byref(d), ssd.SSD_BF16, 0) == want
    expect_seg = {(32, 131072): True, (76, 131072): True}.get((d.nheads, d.seqlen), False)
    assert seg == expect_seg


@pytest.mark.parametrize("kw,code", [
    (dict(ngroups=3), ssd.SSD_BF16 and 1),
    (dict(chunk_len=100), 2),
    (dict(chunk_len=512), 2),
    (dict(headdim=130), 2),
    (dict(dstate=6), 2),
    (dict(batch=0), 1),
    (dict(reserved=1), 1),
    (dict(flags=8), 1),
])
def test_supported_rejects(lib, kw, code):
    assert lib.ssd_supported(ctypes.byref(_dims(**kw)), ssd.SSD_BF16) == code
    assert lib.ssd_last_error()


def test_flags_accepted(lib):
    for flags in (ssd.SSD_FLAG_SIMT, ssd.SSD_FLAG_CHECK_FINITE, ssd.SSD_FLAG_SIMT | ssd.SSD_FLAG_CHECK_FINITE):
        assert lib.ssd_supported(ctypes.byref(_dims(flags=flags)), ssd.SSD_BF16) == 0
    # the check adds no workspace
    base = lib.ssd_workspace_bytes(ctypes.byref(_dims()), ssd.SSD_BF16, 1)
    chk = lib.ssd_workspace_bytes(ctypes.byref(_dims(flags=ssd.SSD_FLAG_CHECK_FINITE)), ssd.SSD_BF16, 1)
    assert base == chk


def test_status_query_arguments(lib):
    assert lib.ssd_workspace_status(None, 1 << 20, None) == 1
    assert lib.ssd_workspace_status(ctypes.c_void_p(0x10000), 8, None) == 1
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    assert lib.ssd_wait_selftest(None, 64, 1000, 0, None) == 1
    assert lib.ssd_wait_selftest(fake, 8, 1000, 0, None) == 1
    for limit_us, arrive in ((0, 0), (2000001, 0), (1000, 2), (1000, -1)):
        assert lib.ssd_wait_selftest(fake, 64, limit_us, arrive, None) == 1


def test_supported_accepts_workloads(lib):
    from state_space_model_mamba_gb300.inputs import WORKLOADS
    for w in WORKLOADS.values():
        d = _dims(**w.dims())
        assert lib.ssd_supported(ctypes.byref(d), 0 if w.dtype == "f32" else 1) == 0


def test_calls_reject_bad_arguments_before_launch(lib):
    d = _dims(batch=1, seqlen=64, nheads=2, headdim=8, dstate=8, chunk_len=16)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    args = [fake] * 10
    # NULL x
    rc = lib.ssd_forward(ctypes.byref(d), 0, None, *args[1:], fake, 1 << 20, None)
    assert rc == 1 and b"x is NULL" in lib.ssd_last_error()
    # misaligned B
    bad = ctypes.c_void_p(0x10004)
    rc = lib.ssd_forward(ctypes.byref(d), 0, fake, fake, fake, bad, fake, fake, None, None, fake,
                         None, fake, 1 << 20, None)
    assert rc == 1 and b"aligned" in lib.ssd_last_error()
    # workspace too small
    rc = lib.ssd_forward(ctypes.byref(d), 0, fake, fake, fake, fake, fake, fake, None, None, fake,
                         None, fake, 16, None)
    assert rc == 3
    # backward: NULL dB
    rc = lib.ssd_backward(ctypes.byref(d), 0, fake, fake, fake, fake, fake, fake, None, None, fake,
                          None, fake, fake, fake, None, fake, fake, None, fake, 1 << 30, None)
    assert rc == 1 and b"dB is NULL" in lib.ssd_last_error()
    # bad dtype
    rc = lib.ssd_forward(ctypes.byref(d), 7, *([fake] * 6), None, None, fake, None, fake, 1 << 20, None)
    assert rc == 1


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        ssd.load_library(str(tmp_path / "nope.so"))
