"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle,
element by element, on seeded inputs.  Bars: normwise relative error <= 1e-4
on the fp32 path and <= 2e-2 on the bf16 path, for y, final_state and every
gradient; padded positions exactly 0."""
import numpy as np
import pytest

from state_space_model_mamba_gb300.inputs import WORKLOADS, generate, generate_small
from parity_util import TOL, compare, padded_grads_zero, run_gpu, run_oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def small(b, L, H, P, N, G, seed, valid_len=None, bf16=False, init_std=0.3, dt_mu=-2.0):
    return generate_small(b, L, H, P, N, G, seed=seed, init_std=init_std, d_final_std=1.0,
                          valid_len=valid_len, bf16=bf16, dt_mu=dt_mu)


# ---------------------------------------------------------------- fp32 path
@pytest.mark.parametrize("Q", [16, 32, 64])
def test_fp32_small_ragged_grouped(Q):
    inp = small(2, 200, 4, 16, 32, 2, seed=40 + Q, valid_len=[150, 200])
    gpu = run_gpu(inp, "f32", Q)
    compare(gpu, run_oracle(inp), TOL["f32"], f"f32 Q={Q}")
    padded_grads_zero(gpu, inp["valid_len"])


def test_fp32_tiny_workload():
    w = WORKLOADS["tiny_f32"]
    inp = generate(w)
    compare(run_gpu(inp, "f32", w.chunk_len), run_oracle(inp), TOL["f32"], "tiny")


# ---------------------------------------------------------------- bf16 path
@pytest.mark.parametrize("simt", [False, True])
@pytest.mark.parametrize("Q", [64, 128, 256])
def test_bf16_small_ragged_grouped(Q, simt):
    inp = small(2, 700, 4, 64, 128, 2, seed=50 + Q, valid_len=[517, 700], bf16=True)
    gpu = run_gpu(inp, "bf16", Q, simt=simt)
    compare(gpu, run_oracle(inp), TOL["bf16"], f"bf16 Q={Q} simt={simt}")
    padded_grads_zero(gpu, inp["valid_len"])


def test_bf16_q128_several_heads_per_cta():
    # chunk 128 with enough chunks that every per-group kernel gives a CTA several
    # heads (the small cases above give each CTA one head), ragged and grouped
    inp = small(2, 8192, 8, 64, 128, 2, seed=58, valid_len=[8192, 5000], bf16=True)
    gpu = run_gpu(inp, "bf16", 128)
    compare(gpu, run_oracle(inp), TOL["bf16"], "bf16 Q=128 multi-head")
    padded_grads_zero(gpu, inp["valid_len"])


@pytest.mark.parametrize("Q", [128, 256])
def test_bf16_strong_decay(Q):
    # dt ~ softplus(N(0.5, 1)) with |A| up to 16: with these seeds 32 % (Q = 128) and
    # 75 % (Q = 256) of the 16-token blocks decay by more than e^64 (the tensor-core
    # kernels then take one exponential per element on the diagonal sub-blocks), the
    # rest stay below it (factored path), mixed within single heads
    inp = small(2, 700, 4, 64, 128, 2, seed=70 + Q, valid_len=[517, 700], bf16=True, dt_mu=0.5)
    gpu = run_gpu(inp, "bf16", Q)
    compare(gpu, run_oracle(inp), TOL["bf16"], f"bf16 strong decay Q={Q}")
    padded_grads_zero(gpu, inp["valid_len"])


def test_chunk_length_independence():
    # the same inputs at chunk 64 (CUDA-core path), 128 and 256 (tensor-core path):
    # chunking regroups the recurrence exactly, so each result meets the bar against
    # the oracle and any two agree within the sum of their bars (triangle inequality)
    inp = small(2, 700, 4, 64, 128, 2, seed=80, valid_len=[517, 700], bf16=True)
    ref = run_oracle(inp)
    outs = {Q: run_gpu(inp, "bf16", Q) for Q in (64, 128, 256)}
    for Q, o in outs.items():
        compare(o, ref, TOL["bf16"], f"Q={Q}")
    compare(outs[128], outs[256], 2 * TOL["bf16"], "Q=128 vs Q=256")
    compare(outs[64], outs[256], 2 * TOL["bf16"], "Q=64 vs Q=256")


@pytest.mark.parametrize("N", [64, 128])
def test_bf16_dstate(N):
    inp = small(1, 512, 2, 64, N, 1, seed=60 + N, bf16=True)
    compare(run_gpu(inp, "bf16", 256), run_oracle(inp), TOL["bf16"], f"bf16 N={N}")


# ---------------------------------------------------------------- edge cases
def test_edge_single_token_and_empty_sample():
    inp = small(3, 1, 2, 8, 8, 1, seed=70, valid_len=[1, 0, 1])
    gpu = run_gpu(inp, "f32", 16)
    compare(gpu, run_oracle(inp), TOL["f32"], "L=1")
    assert np.all(gpu["y"][1] == 0) and np.all(gpu["dx"][1] == 0)
    # an empty sample passes the initial state through and its gradient back
    np.testing.assert_allclose(gpu["final_state"][1], inp["init"][1], rtol=0, atol=0)
    np.testing.assert_allclose(gpu["d_init"][1], inp["d_final"][1], rtol=1e-6)


def test_edge_seqlen_below_chunk():
    inp = small(2, 37, 2, 64, 64, 1, seed=71, bf16=True)
    compare(run_gpu(inp, "bf16", 256), run_oracle(inp), TOL["bf16"], "L<Q")


def test_edge_all_padding_chunks_skipped():
    # second sample valid for one token: whole chunks past valid_len
    inp = small(2, 1024, 2, 64, 128, 1, seed=72, valid_len=[1024, 1], bf16=True)
    gpu = run_gpu(inp, "bf16", 256)
    compare(gpu, run_oracle(inp), TOL["bf16"], "valid_len=1")
    padded_grads_zero(gpu, inp["valid_len"])


def test_backward_is_deterministic():
    inp = small(2, 512, 4, 64, 128, 2, seed=73, bf16=True)
    a = run_gpu(inp, "bf16", 256)
    b = run_gpu(inp, "bf16", 256)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


# ---------------------------------------------------------------- full-size workloads
@pytest.mark.parametrize("name", ["mamba2_130m", "mamba2_2p7b", "grouped_padded", "long_seq"])
def test_workload_full_size(name):
    w = WORKLOADS[name]
    inp = generate(w)
    gpu = run_gpu(inp, w.dtype, w.chunk_len)
    errs = compare(gpu, run_oracle(inp), TOL[w.dtype], name)
    padded_grads_zero(gpu, inp["valid_len"])
    print(name, {k: f"{v:.2e}" for k, v in errs.items()})
