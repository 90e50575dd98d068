"""ssd_forward_noalloc: the forward for callers that cannot allocate device
memory (an arena-owned or pool-owned process, a plug-in whose host framework
forbids allocation on the hot path, code running while another component
captures work).  Its scratch is a fixed array inside the library, so the
check here is that two calls in a row, sharing that array, give what
ssd_forward gives with a caller-allocated workspace, and that shapes needing
more scratch than the array holds are refused before any work is enqueued.

This file is named to be collected last."""
import ctypes

import numpy as np
import pytest

from state_space_model_mamba_gb300 import ssd
from state_space_model_mamba_gb300.inputs import generate_small

SSD_ERR_UNSUPPORTED = 2


def _noalloc_fn():
    lib = ssd.load_library()
    fn = lib.ssd_forward_noalloc
    fn.argtypes = [ctypes.POINTER(ssd.SsdDims), ctypes.c_int] + [ctypes.c_void_p] * 10 + [ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return lib, fn


def test_noalloc_refuses_shapes_beyond_the_static_scratch():
    from state_space_model_mamba_gb300 import build as ssd_build
    ssd_build.build()
    lib, fn = _noalloc_fn()
    # the 2.7B-layer forward needs several hundred MB of scratch
    dims = ssd.Dims(2, 8192, 80, 64, 128, 1, 256).c()
    need = lib.ssd_workspace_bytes(ctypes.byref(dims), ssd.SSD_BF16, 0)
    assert need > 64 * 1024 * 1024
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the size check comes first
    rc = fn(ctypes.byref(dims), ssd.SSD_BF16, fake, fake, fake, fake, fake, fake, None, None, fake, None, None)
    assert rc == SSD_ERR_UNSUPPORTED
    msg = lib.ssd_last_error().decode()
    assert "scratch" in msg and str(need) in msg


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,shape,Q,valid", [
    ("bf16", (2, 700, 4, 64, 128, 2), 256, [517, 700]),   # tensor-core path
    ("f32", (2, 200, 4, 16, 32, 2), 32, [150, 200]),      # CUDA-core path
])
def test_noalloc_forward_matches_ssd_forward_twice(dtype, shape, Q, valid):
    torch = pytest.importorskip("torch")
    from parity_util import TOL, normrel, to_device
    b, L, H, P, N, G = shape
    inp = generate_small(b, L, H, P, N, G, seed=91, init_std=0.3, d_final_std=1.0, valid_len=valid,
                         bf16=dtype == "bf16")
    d = to_device(inp, dtype)
    y_ref, f_ref = ssd.ssd_forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], Q,
                                   init_state=d["init"], valid_len=d["valid_len"])
    torch.cuda.synchronize()
    lib, fn = _noalloc_fn()
    dims = ssd.dims_of(d["x"], d["B"], Q).c()
    code = ssd.SSD_BF16 if dtype == "bf16" else ssd.SSD_F32
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        y = torch.full_like(y_ref, float("nan"))
        fin = torch.full_like(f_ref, float("nan"))
        rc = fn(ctypes.byref(dims), code, ptr(d["x"]), ptr(d["dt"]), ptr(d["A"]), ptr(d["B"]),
                ptr(d["C"]), ptr(d["D"]), ptr(d["init"]), ptr(d["valid_len"]), ptr(y), ptr(fin), stream)
        assert rc == 0, lib.ssd_last_error().decode()
        ssd.noalloc_status()                     # the call's status words: nothing recorded
        torch.cuda.synchronize()
        ey = normrel(y.double().cpu().numpy(), y_ref.double().cpu().numpy())
        ef = normrel(fin.double().cpu().numpy(), f_ref.double().cpu().numpy())
        assert ey <= TOL[dtype] and ef <= TOL[dtype], f"call {call}: y {ey:.2e}, final {ef:.2e}"
        assert np.isfinite(y.float().cpu().numpy()).all()
