"""The comparison the GPU parity tests use, checked on the CPU: the per-tile
bound catches one wrong tile that the whole-tensor bound lets through, tiles
follow the documented layouts, and near-zero tiles are judged against the
floor, not against their own size."""
import numpy as np
import pytest

from parity_util import TILE_FLOOR, compare, normrel, tile_errors


def test_one_wrong_tile_passes_whole_norm_but_fails_tile_bound():
    rng = np.random.default_rng(0)
    b, L, H, P, Q = 1, 16384, 64, 4, 256          # 64 chunks x 64 heads = 4096 tiles
    ref = rng.standard_normal((b, L, H, P))
    gpu = ref.copy()
    gpu[0, 5 * Q:6 * Q, 17, :] = 0.0               # tile (b=0, chunk 5, head 17) wholly wrong
    assert normrel(gpu, ref) < 2e-2                # the whole norm cannot see it
    te = tile_errors(gpu, ref, "y", Q)
    assert te.shape == (b * (L // Q) * H,)
    assert int(np.argmax(te)) == 5 * H + 17 and te.max() == pytest.approx(1.0)
    assert np.count_nonzero(te) == 1
    with pytest.raises(AssertionError, match="tile error"):
        compare({"y": gpu}, {"y": ref}, 2e-2, chunk=Q)


@pytest.mark.parametrize("key,shape,tile", [
    ("ddt", (2, 3, 600), (1, 2, 1)),              # (b, head, chunk): chunk 2 of [b=1, h=2]
    ("dB", (2, 600, 3, 8), (1, 2, 1)),            # (b, chunk, group)
    ("final_state", (2, 3, 4, 8), (1, 2)),        # (b, head)
])
def test_tile_layouts(key, shape, tile):
    rng = np.random.default_rng(1)
    Q = 256                                        # 600 tokens: a ragged third chunk
    ref = rng.standard_normal(shape)
    gpu = ref.copy()
    if key == "ddt":
        gpu[tile[0], tile[1], 256 * tile[2]:256 * tile[2] + 7] += 5.0
        flat = (tile[0] * shape[1] + tile[1]) * 3 + tile[2]
    elif key == "dB":
        gpu[tile[0], 256 * tile[1]:256 * tile[1] + 7, tile[2]] += 5.0
        flat = (tile[0] * 3 + tile[1]) * shape[2] + tile[2]
    else:
        gpu[tile[0], tile[1]] += 5.0
        flat = tile[0] * shape[1] + tile[1]
    te = tile_errors(gpu, ref, key, Q)
    assert int(np.argmax(te)) == flat and np.count_nonzero(te) == 1


def test_near_zero_tile_judged_against_floor():
    rng = np.random.default_rng(2)
    ref = rng.standard_normal((1, 512, 2, 4))
    ref[0, :256, 0] *= 1e-9                        # one tile 1e-9 the size of the others
    gpu = ref.copy()
    gpu[0, :256, 0] *= 2.0                         # 100 % wrong relative to itself ...
    te = tile_errors(gpu, ref, "y", 256)
    assert te.max() < 1e-6                         # ... but negligible against the floor
    rms = np.sqrt(np.mean([np.sum(ref[0, q * 256:(q + 1) * 256, h] ** 2) for q in range(2) for h in range(2)]))
    assert TILE_FLOOR * rms > 1e-8 * np.linalg.norm(ref[0, :256, 0])
