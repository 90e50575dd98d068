"""Host-side arithmetic of bench.py (no GPU): the per-kernel table of the
benchmark line and the cost model's coverage of every kernel the library
launches."""
import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from state_space_model_mamba_gb300.inputs import WORKLOADS  # noqa: E402


def launch_names():
    with open(os.path.join(ROOT, "state_space_model_mamba_gb300", "csrc", "ssd_api.cu")) as f:
        return set(re.findall(r'SSD_LAUNCH\("([a-z0-9_]+)"', f.read()))


def test_kernel_table_arithmetic():
    per = {"bwd_orange_tc": [0.2, 0.2], "bwd_dcb_tc": [0.1, 0.3], "k1_chunk_cumsum": [0.01, 0.01]}
    costs = {"bwd_orange": (0.0, 1_000_000_000), "bwd_dcb": (0.0, 500_000_000)}
    live = [0.25] * 4
    t = bench.kernel_table(per, "bwd_orange_tc", live, steps=4, prof_steps=2, costs=costs,
                           hbm_gbs=8000.0)
    o, g, k1 = t["bwd_orange_tc"], t["bwd_dcb_tc"], t["k1_chunk_cumsum"]
    assert o["launches"] == 4 and o["timed_live"] and "second_stream" not in o
    assert o["avg_us"] == pytest.approx(250.0)
    assert o["hbm_frac"] == pytest.approx(0.5)          # 1 GB in 250 us = 4000 GB/s of 8000
    assert g["avg_us"] == pytest.approx(200.0) and g["second_stream"] and "timed_live" not in g
    assert g["hbm_frac"] == pytest.approx(0.5e9 / 200e-6 / 1e9 / 8000.0)
    assert "hbm_frac" not in k1                          # no cost entry given
    assert sum(e["share"] for e in t.values()) == pytest.approx(1.0)
    assert o["share"] == pytest.approx(0.4 / 0.82)       # profiled time, not the live one


def test_every_launched_kernel_has_a_cost():
    names = launch_names()
    assert {"k1_chunk_cumsum", "k5_scan_tc", "bwd_orange_tc", "bwd_dcb_tc"} <= names
    for w in ("mamba2_2p7b", "tiny_f32"):
        for tc in (True, False):
            costs = bench.kernel_costs(WORKLOADS[w], tc=tc)
            missing = {n for n in names if bench.cost_key(n) not in costs}
            assert not missing, missing
            assert all(b > 0 for _, b in costs.values())


def test_second_stream_names_are_launched_kernels():
    assert set(bench.SECOND_STREAM) <= launch_names()


PEAKS = {"hbm_gbs": 6789.0, "bf16_tflops_sustained": 1691.0, "sm_max_mhz": 2070.0}


def test_roofline_hbm_bound_live_and_alone():
    # the ORANGE backward at the 2.7B layer: 528.5 MB and 43.1 GF per launch (below the
    # ridge of ~249 flop/B), 219 us live beside the group chain, 176 us alone
    r = bench.roofline_entry("bwd_orange_tc", 43.1e9, 528.5e6, 0.219, 0.176, PEAKS)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6789.0
    assert r["achieved"] == pytest.approx(528.5e6 / 219e-6 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6789.0)
    assert r["alone"]["avg_us"] == pytest.approx(176.0)
    assert r["alone"]["frac"] == pytest.approx(528.5e6 / 176e-6 / 1e9 / 6789.0)
    assert r["kernel"] == "bwd_orange_tc" and r["algorithmic_bytes_per_launch"] == 528.5e6


def test_roofline_tensor_and_alu_bounds():
    r = bench.roofline_entry("k_tc", 1e12, 1e9, 1.0, 0.5, PEAKS)       # 1000 flop/B > ridge
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(1000.0) and r["alone"]["achieved"] == pytest.approx(2000.0)
    assert r["frac"] == pytest.approx(1000.0 / 1691.0)
    r = bench.roofline_entry("k_simt", 1e9, 1e9, 1.0, 1.0, PEAKS)     # CUDA-core kernel
    assert r["bound"] == "alu" and r["peak"] == pytest.approx(152 * 128 * 2 * 2070e6 / 1e12)
    r = bench.roofline_entry("k1_chunk_cumsum", 0.0, 1e7, 0.01, 0.01, PEAKS)
    assert r["bound"] == "hbm" and r["achieved"] == pytest.approx(1000.0)
