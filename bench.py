#!/usr/bin/env python
"""Benchmark of the SSD chunked selective scan: forward + backward tokens/s.

One step = ssd_forward + ssd_backward (the backward recomputes every forward
intermediate) over one batch of the Mamba-2 2.7B-layer shape (batch 2,
seqlen 8192, nheads 80, headdim 64, dstate 128, ngroups 1, chunk 256; bf16
x/B/C/dy, fp32 dt/A/D), synthetic seeded inputs resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--profile-case forward|step]
                    [--op quat_scan|ydiag_siso|ydiag_mimo4|state_moments]

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs an
independent replica of the workload (the scan has no data-path exchange) and
`value` is the tokens all ranks processed divided by the slowest rank's time.
`--impl reference` times the CPU oracle (plain fp64 recurrence) on the host
cores on a bounded sample of the same workload.  `--profile-case` is the
light run that ncu captures are taken on: W + K forward calls (or whole
steps) on resident inputs, then a short line; no per-kernel pass, no end-to-end
leg, no CPU baseline.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from state_space_model_mamba_gb300.inputs import WORKLOADS, generate  # noqa: E402

METRIC = "SSD fwd+bwd tokens/sec (2.7B-layer shape, 1 GB300); % of tensor/HBM roofline"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "mamba2_2p7b"
L2_BYTES = 129 * 1024 * 1024
# kernels the library launches on its second stream, beside the caller's chain
SECOND_STREAM = ("k2_cb_tc", "bwd_dcb_tc", "bwd_dbc_tc", "bwd_dbc_reduce_tc")
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))


def kernel_table(per: dict, top: str, live: list, steps: int, prof_steps: int, costs: dict,
                 hbm_gbs: float) -> dict:
    """Per-kernel entries of the benchmark line.  `per` maps a kernel name to its
    event durations (ms) over `prof_steps` profiled steps, `live` holds the
    dominant kernel's durations inside the timed region of `steps` steps.  Each
    entry: launches in the timed region, mean duration (the live one for `top`),
    share of the summed profiled time, the fraction of the HBM peak its
    algorithmic bytes per launch reach at that duration, and whether it runs on
    the library's second stream."""
    tot = sum(sum(v) for v in per.values())
    out = {}
    for k, v in per.items():
        e = {"launches": len(v) * steps // prof_steps, "avg_us": 1e3 * sum(v) / len(v),
             "share": sum(v) / tot if tot else None}
        if k == top:
            e["avg_us"] = 1e3 * sum(live) / len(live)
            e["timed_live"] = True
        byts = costs.get(cost_key(k), (0.0, 0))[1]
        if byts and e["avg_us"] > 0:
            e["hbm_frac"] = byts / (e["avg_us"] * 1e-6) / 1e9 / hbm_gbs
        if k in SECOND_STREAM:
            e["second_stream"] = True
        out[k] = e
    return out


def roofline_entry(kernel: str, flops: float, byts: float, live_ms: float, alone_ms: float,
                   peaks: dict) -> dict:
    """The roofline object of the benchmark line for one kernel: its algorithmic
    work per launch over its mean live launch time in the timed region
    (`achieved`, `frac`), against the HBM peak, the sustained bf16 tensor peak
    (when its flops per byte exceed the ridge) or the fp32 FFMA peak (CUDA-core
    kernels); and the same over its mean time when it runs alone (`alone`)."""
    ridge = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if kernel.endswith("_simt") and flops > 0:
        sm_mhz = peaks.get("sm_max_mhz", 2070.0)
        bound, unit, work = "alu", "TFLOP/s", flops / 1e12
        peak = 152 * 128 * 2 * sm_mhz * 1e6 / 1e12                    # fp32 FFMA TFLOP/s
    elif flops > 0 and flops / max(byts, 1) > ridge:
        bound, unit, work, peak = "tensor", "TFLOP/s", flops / 1e12, peaks["bf16_tflops_sustained"]
    else:
        bound, unit, work, peak = "hbm", "GB/s", byts / 1e9, peaks["hbm_gbs"]
    achieved = work / (live_ms * 1e-3)
    alone = work / (alone_ms * 1e-3)
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "kernel": kernel,
            "algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": byts,
            "alone": {"avg_us": 1e3 * alone_ms, "achieved": alone, "frac": alone / peak}}


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest `x` over all ranks (the slowest rank's time); `x` itself on
    one rank.  `device` holds the reduction tensor: the rank's GPU under NCCL,
    the CPU under gloo."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def kernel_costs(w, tc: bool) -> dict:
    """Algorithmic work of each kernel per launch: (flops, bytes).  Flops count
    the causal half of the Q x Q blocks (and K2 / its backward per group, not per
    head); bytes count every input of the kernel read once and every output
    written once, intermediates at the precision the path stores them (chunk
    states and CB in bf16 on the tensor-core path, fp32 on the CUDA-core path)."""
    b, L, H, P, N, G, Q = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk_len
    n = -(-L // Q)
    Lp = n * Q
    s = 2 if w.dtype == "bf16" else 4
    st = b * n * H * P * N                       # chunk-state elements
    tri = Q * (Q + 1) // 2                       # causal pairs per chunk
    tok_h = b * H * L
    x_b = s * b * L * H * P                      # one [b,L,H,P] tensor
    bc_b = s * b * L * G * N                     # one [b,L,G,N] tensor
    cum_b = 4 * b * H * Lp                       # one per-token fp32 [b,H,n,Q] array
    sts = 2 if tc else 4                         # bytes per stored chunk-state element
    cbs = 2 if tc else 4                         # bytes per stored CB element
    cb_b = cbs * b * n * G * tri                 # causal CB of every (chunk, group)
    c = {
        "k1_chunk_cumsum": (0.0, 4 * tok_h + cum_b + 4 * b * H * n),
        "k2_cb": (2.0 * b * n * G * tri * N, 2 * bc_b + cb_b * (2 if tc else 1)),   # CB and CB^T on tc
        "k3_state": (2.0 * b * n * H * Q * P * N, x_b + bc_b + 4 * tok_h + cum_b + sts * st),
        "k4_state_passing": (2.0 * st, 2 * sts * st + 4 * b * H * n),
        # fused K1 + K3 + K4 (tensor-core path): reads x, B, dt (and init), writes cumA, endA,
        # the bf16 chunk-input states (and the final state); the intra states stay on chip
        "state_scan": (2.0 * b * n * H * Q * P * N + 2.0 * st,
                       x_b + bc_b + 4 * tok_h + cum_b + 4 * b * H * n + sts * st + 2 * 4 * b * H * P * N),
        # K5; on the tensor-core path it computes CB itself (K2's flops, B read instead of CB)
        "k5_scan": (b * n * H * (2.0 * Q * P * N + 2.0 * tri * P) + (2.0 * b * n * G * tri * N if tc else 0.0),
                    2 * x_b + bc_b + (bc_b if tc else cb_b) + sts * st + cum_b + 4 * tok_h),
        "bwd_blue": (b * n * H * 4.0 * Q * P * N, x_b + bc_b + 2 * sts * st + 2 * cum_b),
        "bwd_k4_state_passing": (4.0 * st, 3 * sts * st + 4 * b * H * n),
        "bwd_main": (b * n * H * (4.0 * tri * P + 2.0 * Q * P * N),
                     3 * x_b + bc_b + cb_b + sts * st + 6 * cum_b),
        # ORANGE backward: dx' = M^T dy and yo = M (dt x) per head; writes dx and two per-token arrays
        "bwd_orange": (b * n * H * 4.0 * tri * P, 3 * x_b + cb_b + 2 * cum_b + 2 * cum_b),
        # K3 backward: U = B d_intra^T per head; adds into dx, ddt_main, d cumA (read + write)
        "bwd_k3": (b * n * H * 2.0 * Q * P * N, 3 * x_b + bc_b + sts * st + 2 * cum_b + 5 * cum_b),
        # G1: d_cb = sum over the group's heads of dW o decay o dt (dW causal per head)
        "bwd_dcb": (b * n * H * 2.0 * tri * P, 2 * x_b + 2 * cum_b + cbs * b * n * G * Q * Q),
        # G2: dC = d_cb B + sum_h (dy exp cumA) s_in, dB = d_cb^T C + sum_h (x bbs) d_intra
        "bwd_dbc": (b * n * G * 4.0 * tri * N + b * n * H * 4.0 * Q * P * N,
                    2 * x_b + 2 * sts * st + 2 * bc_b + cbs * b * n * G * Q * Q + 2 * cum_b + 2 * 4 * b * L * G * N),
        "bwd_dbc_reduce": (0.0, 2 * 4 * b * L * G * N + 2 * bc_b),
        "bwd_group": (b * n * G * 4.0 * tri * N + b * n * H * 4.0 * Q * P * N,
                      2 * x_b + 2 * sts * st + 4 * bc_b + 2 * cum_b),
        "bwd_k1_chunk_cumsum": (0.0, 4 * cum_b + 8 * tok_h),
        # state moments (128-token chunks): G = X X^T, Y = F B + (2 alpha X) s, A += B^T Y + c0 s^T s;
        # reads x, B, the bf16 chunk-input states, cumA and dt, writes the fp32 range partials
        "moments": (b * -(-L // 128) * H * 2.0 * 128 * 128 * (64 + 2 * (128 + 64)) * (P * N / (64 * 128)),
                    x_b + bc_b + 2 * b * -(-L // 128) * H * P * N + 8 * b * H * -(-L // 128) * 128
                    + 4 * b * H * (N * N + N)),
        "moments_reduce": (0.0, 2 * 4 * b * H * (N * N + N)),
        # debug check (SSD_FLAG_CHECK_FINITE, never timed): reads the backward's outputs,
        # cumA, endA and the chunk states and their gradients once
        "check_finite": (0.0, x_b + 4 * tok_h + 2 * bc_b + cum_b + 4 * b * H * n + 2 * sts * st),
    }
    return c


def cost_key(name: str) -> str:
    for suffix in ("_simt", "_tc"):
        if name.endswith(suffix):
            return name[: -len(suffix)]
    return name


def source_digest() -> str:
    """Digest of the sources the SSD kernels are built from (every csrc file but
    the Mamba-3 kernels', which no SSD launch uses): `traffic.json` figures
    apply while it matches."""
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "state_space_model_mamba_gb300", "csrc", "*"))):
        if os.path.basename(f) == "mamba3.cu":
            continue
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if it
    was taken on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(kernel)
    if not e or e.get("source_digest") != source_digest():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"ssd_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "50"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()
        return False

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        pw = [float(r[4]) for r in rows if r[4].replace(".", "").isdigit()]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            for nm, v in zip(names, r[6:10]):
                if v.lower() == "active":
                    reasons.add(nm)
        load = sorted(sm)[len(sm) // 4:] if len(sm) >= 4 else sm  # drop the idle ramp samples
        return {"sm_mhz": statistics.median(load) if load else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "samples": len(rows), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample(inp, w, heads: int, seqlen: int):
    """Run the oracle forward + backward on batch 0, the first `heads` heads and
    the first `seqlen` tokens.  Returns (seconds, head_tokens, threads)."""
    import oracle
    G = w.ngroups
    hpg = w.nheads // G
    heads = max(1, min(heads, w.nheads))
    hsel = slice(0, heads)
    gcount = -(-heads // hpg)
    sub = dict(
        x=inp["x"][:1, :seqlen, hsel], dt=inp["dt"][:1, hsel, :seqlen], A=inp["A"][hsel],
        B=inp["B"][:1, :seqlen, :gcount], C=inp["C"][:1, :seqlen, :gcount], D=inp["D"][hsel],
        init=None if inp["init"] is None else inp["init"][:1, hsel],
        dy=inp["dy"][:1, :seqlen, hsel],
        d_final=None if inp["d_final"] is None else inp["d_final"][:1, hsel])
    if heads % hpg != 0 or gcount * hpg != heads:
        # keep whole groups: use one group per head for the sample
        sub["B"] = np.repeat(sub["B"][:, :, :1], heads, axis=2)
        sub["C"] = np.repeat(sub["C"][:, :, :1], heads, axis=2)
    vl = None
    if inp["valid_len"] is not None:
        vl = np.minimum(inp["valid_len"][:1], seqlen).astype(np.int32)
    t0 = time.perf_counter()
    oracle.forward(sub["x"], sub["dt"], sub["A"], sub["B"], sub["C"], sub["D"], sub["init"], vl)
    oracle.backward(sub["x"], sub["dt"], sub["A"], sub["B"], sub["C"], sub["D"], sub["init"], vl,
                    sub["dy"], sub["d_final"])
    dt = time.perf_counter() - t0
    return dt, heads * seqlen, oracle.num_threads()


def cpu_baseline(inp, w, target_s: float = 15.0):
    """Time the oracle on a bounded sample of about `target_s` seconds: the
    first heads of batch 0 over the whole sequence, repeated until the time is
    reached (one repetition when the sample alone is that long)."""
    import oracle
    cores = oracle.num_threads()
    heads = min(w.nheads, max(2 * cores, 1))
    probe_len = min(w.seqlen, 512)
    t, ht, thr = oracle_sample(inp, w, heads, probe_len)
    rate = ht / max(t, 1e-9)                                   # head-tokens / s
    seqlen = int(min(w.seqlen, max(probe_len, rate * target_s / heads)))
    tot, reps, done = 0.0, 0, 0
    while tot < 0.8 * target_s or reps == 0:
        t, ht, thr = oracle_sample(inp, w, heads, seqlen)
        tot += t
        reps += 1
        done += ht
    value = done / tot / w.nheads                              # tokens/s of the full-head workload
    return {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle",
            "sample": f"fp64 serial recurrence fwd+bwd on batch 0, heads 0..{heads - 1} of "
                      f"{w.nheads}, first {seqlen} of {w.seqlen} tokens, {reps} repetition(s), "
                      f"{tot:.1f} s; scaled to tokens/s of all {w.nheads} heads"}


# ----------------------------------------------------------------------------- arms
def run_reference(args, w, rank, world):
    if rank != 0:
        return None
    inp = generate(w)
    import oracle
    cores = oracle.num_threads()
    heads = min(w.nheads, cores)
    total_steps = args.steps + args.warmup
    budget = 120.0 / max(total_steps, 1)                       # seconds per step
    t, ht, _ = oracle_sample(inp, w, heads, min(w.seqlen, 256))
    rate = ht / max(t, 1e-9)
    seqlen = int(min(w.seqlen, max(64, rate * budget / heads)))
    for _ in range(args.warmup):
        oracle_sample(inp, w, heads, seqlen)
    times = []
    for _ in range(args.steps):
        t, ht, thr = oracle_sample(inp, w, heads, seqlen)
        times.append(t)
    tot = sum(times)
    value = ht * args.steps / tot / w.nheads
    sample = (f"each step: fp64 oracle fwd+bwd on batch 0, heads 0..{heads - 1} of {w.nheads}, "
              f"first {seqlen} of {w.seqlen} tokens; value scaled to tokens/s of all heads")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, **w.dims()},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_profile_case(args, w, local_rank):
    """W warm-up and K timed forward calls (or fwd + bwd steps) on resident
    inputs, for ncu captures: nothing else is launched."""
    import torch

    from state_space_model_mamba_gb300 import ssd
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    inp = generate(w)
    bf = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    def up(a, dt=torch.float32):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)

    x, B, C, dy = up(inp["x"], bf), up(inp["B"], bf), up(inp["C"], bf), up(inp["dy"], bf)
    dt, A, D, init, dfin = up(inp["dt"]), up(inp["A"]), up(inp["D"]), up(inp["init"]), up(inp["d_final"])
    vl = None if inp["valid_len"] is None else torch.from_numpy(inp["valid_len"]).to(dev)
    dims = ssd.dims_of(x, B, w.chunk_len, split_scan=args.split_scan)
    code = ssd.SSD_BF16 if w.dtype == "bf16" else ssd.SSD_F32
    bwd = args.profile_case == "step"
    ws = ssd.alloc_workspace(dims, code, bwd, dev)
    y = torch.empty_like(x)
    fin = torch.empty(w.batch, w.nheads, w.headdim, w.dstate, device=dev)
    g = dict(dx=torch.empty_like(x), ddt=torch.empty_like(dt), dA=torch.empty_like(A),
             dB=torch.empty_like(B), dC=torch.empty_like(C), dD=torch.empty_like(D),
             d_init=torch.empty_like(fin))

    def one():
        ssd.forward_into(dims, x, dt, A, B, C, D, init, vl, y, fin, ws)
        if bwd:
            ssd.backward_into(dims, x, dt, A, B, C, D, init, vl, dy, dfin, g["dx"], g["ddt"], g["dA"],
                              g["dB"], g["dC"], g["dD"], g["d_init"], ws)

    for _ in range(args.warmup):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        one()
    e1.record()
    torch.cuda.synchronize()
    ssd.workspace_status(ws)
    ms = e0.elapsed_time(e1) / args.steps
    return {"profile_case": args.profile_case, "workload": w.name, "steps": args.steps,
            "warmup": args.warmup, "ms_per_call": ms, "device_bytes": torch.cuda.max_memory_allocated(dev)}


def run_ours(args, w, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from state_space_model_mamba_gb300 import ssd

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    inp = generate(w)
    bf = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    def up(a, dt=torch.float32):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)

    x, B, C, dy = up(inp["x"], bf), up(inp["B"], bf), up(inp["C"], bf), up(inp["dy"], bf)
    dt, A, D = up(inp["dt"]), up(inp["A"]), up(inp["D"])
    init, dfin = up(inp["init"]), up(inp["d_final"])
    vl = None if inp["valid_len"] is None else torch.from_numpy(inp["valid_len"]).to(dev)
    dims = ssd.dims_of(x, B, w.chunk_len, split_scan=args.split_scan)
    code = ssd.SSD_BF16 if w.dtype == "bf16" else ssd.SSD_F32
    ws = torch.empty(max(ssd.workspace_bytes(dims, code, True),
                         ssd.workspace_bytes(dims, code, False)), dtype=torch.uint8, device=dev)
    y = torch.empty_like(x)
    fin = torch.empty(w.batch, w.nheads, w.headdim, w.dstate, device=dev)
    g = dict(dx=torch.empty_like(x), ddt=torch.empty_like(dt), dA=torch.empty_like(A),
             dB=torch.empty_like(B), dC=torch.empty_like(C), dD=torch.empty_like(D),
             d_init=torch.empty_like(fin))

    def fwd():
        ssd.forward_into(dims, x, dt, A, B, C, D, init, vl, y, fin, ws)

    def step():
        fwd()
        n1 = ssd.last_launch_count()
        ssd.backward_into(dims, x, dt, A, B, C, D, init, vl, dy, dfin, g["dx"], g["ddt"], g["dA"],
                          g["dB"], g["dC"], g["dD"], g["d_init"], ws)
        return n1 + ssd.last_launch_count()

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        launches_per_step = step()
    # launch sequence of one step (names of the timed kernel units)
    probe = ssd.KernelTimer(capacity_kernels=64)
    with probe:
        step()
    pattern = [nm for nm, _ in probe.durations()]
    torch.cuda.synchronize()
    ssd.workspace_status(ws)

    # per-kernel durations from an untimed pass (an event pair around every
    # kernel); the timed region below brackets only the dominant kernel, so that
    # the step time carries no per-kernel instrumentation
    prof_steps = max(3, min(args.steps, 20))
    ptimer = ssd.KernelTimer(capacity_kernels=len(pattern) * prof_steps + 8)
    with ptimer:
        for _ in range(prof_steps):
            step()
    per = {}
    for name, ms in ptimer.durations(pattern):
        per.setdefault(name, []).append(ms)
    # (while every kernel is timed the library runs its second-stream kernels on the
    # caller's stream, so these are standalone durations.)  The dominant kernel is taken
    # among the caller's-stream kernels: in the timed region below the second-stream
    # kernels run beside them, and their event spans would include that overlap
    top = max((k for k in per if k not in SECOND_STREAM), key=lambda k: sum(per[k]))

    # ---------------- timed region (device time, CUDA events on the launching stream)
    stream = torch.cuda.current_stream(dev)
    timer = ssd.KernelTimer(capacity_kernels=args.steps * pattern.count(top) + 8, only=top)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    barrier()
    torch.cuda.synchronize()
    with clocks:
        ev0.record(stream)
        with timer:
            for _ in range(args.steps):
                step()
        ev1.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    ms_step = ms_total / args.steps
    value = w.tokens * world / (ms_step * 1e-3)
    ssd.workspace_status(ws)

    # ---------------- the forward alone, same inputs and timing
    for _ in range(3):
        fwd()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    f0.record(stream)
    for _ in range(args.steps):
        fwd()
    f1.record(stream)
    torch.cuda.synchronize()
    barrier()
    fwd_ms = max_over_ranks(f0.elapsed_time(f1) / args.steps, world, dev)
    ssd.workspace_status(ws)

    # the dominant kernel's live durations (timed region); the others from the pass above
    live = [ms for _, ms in timer.durations()]
    peaks, peak_src = load_peaks()
    shares = kernel_table(per, top, live, args.steps, prof_steps,
                          kernel_costs(w, tc=not any(k.endswith("_simt") for k in pattern)),
                          peaks["hbm_gbs"])
    costs = kernel_costs(w, tc=not top.endswith("_simt"))
    flops, byts = costs[cost_key(top)]
    roof = roofline_entry(top, flops, byts, statistics.mean(live), statistics.mean(per[top]), peaks)
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback"
    roof["traffic"] = ncu_traffic(top, w.name)

    # the whole step against HBM: the kernels' algorithmic bytes summed over one
    # step's launches, and the minimum (every leaf, dy and d_final read once per
    # call, every output written once)
    step_costs = kernel_costs(w, tc=not any(k.endswith("_simt") for k in pattern))
    step_bytes = sum(step_costs.get(cost_key(k), (0.0, 0))[1] for k in pattern)
    nb = lambda *ts: sum(t.numel() * t.element_size() for t in ts if t is not None)
    leaves = nb(x, dt, A, B, C, D, init, vl)
    min_bytes = (leaves + nb(y, fin)) + (leaves + nb(dy, dfin) + nb(*g.values()))
    step_s = ms_step * 1e-3
    step_roof = {"unit": "GB/s", "peak": peaks["hbm_gbs"],
                 "algorithmic_bytes": step_bytes, "achieved": step_bytes / step_s / 1e9,
                 "frac": step_bytes / step_s / 1e9 / peaks["hbm_gbs"],
                 "minimum_bytes": min_bytes,
                 "frac_of_minimum": min_bytes / step_s / 1e9 / peaks["hbm_gbs"]}

    # ---------------- end to end: pinned host buffers -> device -> host every step.
    # Every step's inputs cross to the device and its results cross back inside the
    # timed region; the copies of step i + 1's inputs (one copy stream) and of step
    # i - 1's results (another) run while step i computes, on two device buffer sets.
    host_in = {k: torch.from_numpy(np.ascontiguousarray(inp[k])).to(
        dtype=(bf if k in ("x", "B", "C", "dy") else torch.float32)).pin_memory()
        for k in ("x", "dt", "A", "B", "C", "D", "dy")}
    if inp["init"] is not None:
        host_in["init"] = torch.from_numpy(inp["init"]).pin_memory()
    if inp["d_final"] is not None:
        host_in["d_final"] = torch.from_numpy(inp["d_final"]).pin_memory()
    dev_in = {"x": x, "dt": dt, "A": A, "B": B, "C": C, "D": D, "dy": dy, "init": init,
              "d_final": dfin}
    outs = {"y": y, "final_state": fin, **g}
    host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in outs.items()}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    e2e_steps = max(3, min(args.steps, 20))
    sets = []
    for _ in range(2):
        din = {k: (None if v is None else torch.empty_like(v)) for k, v in dev_in.items()}
        din["valid_len"] = vl
        sets.append((din, {k: torch.empty_like(v) for k, v in outs.items()}))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # set j's inputs are on the device
    ev_done = [torch.cuda.Event() for _ in range(2)]  # set j's step has finished
    ev_out = [torch.cuda.Event() for _ in range(2)]   # set j's results are on the host
    for j in range(2):
        ev_done[j].record(stream)
        ev_out[j].record(stream)

    def e2e_h2d(j):
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_done[j])  # the previous step on set j no longer reads its inputs
            for k, t in host_in.items():
                sets[j][0][k].copy_(t, non_blocking=True)
            ev_in[j].record(s_in)

    def e2e_compute(j):
        d, o = sets[j]
        stream.wait_event(ev_in[j])
        stream.wait_event(ev_out[j])  # set j's previous results have left the device
        ssd.forward_into(dims, d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"],
                         d["valid_len"], o["y"], o["final_state"], ws)
        ssd.backward_into(dims, d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"],
                          d["valid_len"], d["dy"], d["d_final"], o["dx"], o["ddt"], o["dA"], o["dB"],
                          o["dC"], o["dD"], o["d_init"], ws)
        ev_done[j].record(stream)

    def e2e_d2h(j):
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[j])
            for k in outs:
                host_out[k].copy_(sets[j][1][k], non_blocking=True)
            ev_out[j].record(s_out)

    def e2e_run(nsteps):
        e2e_h2d(0)
        for i in range(nsteps):
            if i + 1 < nsteps:
                e2e_h2d((i + 1) % 2)
            e2e_compute(i % 2)
            e2e_d2h(i % 2)
        for j in range(2):
            stream.wait_event(ev_out[j])

    e2e_run(2)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)

    if rank != 0:
        return None
    in_bytes = sum(t.numel() * t.element_size() for t in (x, dt, A, B, C, D, dy))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, **w.dims(),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB > {L2_BYTES / 1e6:.0f} MB); no flush",
                   "step": "ssd_forward + ssd_backward (recompute), inputs resident in HBM",
                   "chunk_states": "split (K3 + K4)" if args.split_scan else "library default"},
        "roofline": roof,
        "step_roofline": step_roof,
        "forward": {"value": w.tokens * world / (fwd_ms * 1e-3), "unit": UNIT,
                    "ms_per_step": fwd_ms, "steps": args.steps},
        "valid_tokens": (None if inp["valid_len"] is None else {
            "per_step": int(np.sum(inp["valid_len"])) * world,
            "value": int(np.sum(inp["valid_len"])) * world / (ms_step * 1e-3), "unit": UNIT,
            "forward_value": int(np.sum(inp["valid_len"])) * world / (fwd_ms * 1e-3)}),
        "kernels": {k: {kk: (round(vv, 4) if isinstance(vv, float) else vv) for kk, vv in s.items()}
                    for k, s in sorted(shares.items(), key=lambda kv: -kv[1]["share"])},
        "e2e": {"value": w.tokens * world / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "steps": e2e_steps,
                "overlap": "step i+1 inputs up and step i-1 results down on two copy streams during step i"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, w, args.cpu_seconds)
    return line


# ----------------------------------------------------------------------------- other ops
# `--op NAME` measures one of the library's other entry points on its workload
# (inputs resident in HBM and larger than L2, CUDA events on the launching
# stream, W warm-up and K timed calls of forward and backward each) and prints
# one line with its own metric, the HBM roofline of the op and the oracle
# timed on the host cores on a bounded sample.
OPS = ("quat_scan", "ydiag_siso", "ydiag_mimo4", "state_moments")


def _event_time(fn, warmup: int, steps: int) -> float:
    """Mean milliseconds per call of fn over `steps` calls after `warmup`."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def _wall_rate(fn, units: float, target_s: float) -> tuple:
    """Units per second of the CPU function fn (repeated to about target_s)."""
    t0 = time.perf_counter()
    reps = 0
    while True:
        fn()
        reps += 1
        el = time.perf_counter() - t0
        if el >= target_s or el * (reps + 1) / reps > 3 * target_s:
            return units * reps / el, reps, el


def run_op(args, local_rank):
    import ctypes

    import torch

    from oracle import mamba3 as om3
    from state_space_model_mamba_gb300 import mamba3, ssd
    from state_space_model_mamba_gb300.inputs import MAMBA3_WORKLOADS, generate_diag, generate_quat
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    lib = mamba3._lib()
    stream = lambda: ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    P_ = lambda t: ctypes.c_void_p(t.data_ptr())
    peaks, peak_src = load_peaks()
    clocks = ClockSampler(local_rank)
    up = lambda a, dt=torch.float32: torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
    if args.op == "state_moments":
        return run_moments(args, dev, peaks, peak_src, clocks)
    if args.op == "quat_scan":
        w = MAMBA3_WORKLOADS["quat_scan_2p7b"]
        inp = generate_quat(w)
        q, init, dcum = up(inp["q"]), up(inp["init"]), up(inp["d_cum"])
        cum, dq, dinit = torch.empty_like(q), torch.empty_like(q), torch.empty_like(init)
        wsf, wsb = mamba3.quat_workspace(q, False), mamba3.quat_workspace(q, True)
        b, L, H, J, _ = q.shape

        def fwd():
            ssd._check(lib.m3_quat_cumprod(P_(q), P_(init), P_(cum), b, L, H, J, P_(wsf), wsf.numel(), stream()))

        def bwd():
            ssd._check(lib.m3_quat_cumprod_backward(P_(q), P_(init), P_(dcum), P_(dq), P_(dinit), b, L, H, J,
                                                    P_(wsb), wsb.numel(), stream()))
        bytes_f = 2 * q.nbytes + init.nbytes
        bytes_b = 3 * q.nbytes + 2 * init.nbytes
        tokens = w.tokens
        config = {"workload": w.name, "batch": b, "seqlen": L, "nheads": H, "nblocks": J, "dtype": "f32"}
        kernels = {"forward": "quat_seg_product + quat_seg_scan", "backward": "quat_bwd_segments + quat_bwd_apply"}
        hs = 8  # oracle sample: batch 0, 8 heads

        def cpu():
            om3.quat_cumprod(inp["q"][:1, :, :hs], inp["init"][:1, :hs])
            om3.quat_cumprod_backward_closed(inp["q"][:1, :, :hs], inp["init"][:1, :hs], inp["d_cum"][:1, :, :hs])
        cpu_units, cpu_scale = L * hs / H, 1.0
        sample = f"fp64 NumPy oracle fwd + closed-form bwd on batch 0, heads 0..{hs - 1} of {H}, all {L} steps; scaled to tokens/s of all heads"
        metric = "Mamba-3 quaternion cumprod scan fwd+bwd tokens/sec (2.7B-layer tokens and heads, 1 GB300)"
    else:
        w = MAMBA3_WORKLOADS["ydiag_siso_2p7b" if args.op == "ydiag_siso" else "ydiag_mimo4"]
        inp = generate_diag(w)
        V, B, C, dY = (up(inp[k], torch.bfloat16) for k in ("V", "B", "C", "dY"))
        g = up(inp["gamma"])
        y, dV, dB, dC, dg = torch.empty_like(V), torch.empty_like(V), torch.empty_like(B), torch.empty_like(C), torch.empty_like(g)
        T, m, H, Pd = V.shape
        N = B.shape[3]

        def fwd():
            ssd._check(lib.m3_y_diag(ssd.SSD_BF16, P_(V), P_(B), P_(C), P_(g), P_(y), T, m, H, Pd, N, stream()))

        def bwd():
            ssd._check(lib.m3_y_diag_backward(ssd.SSD_BF16, P_(dY), P_(V), P_(B), P_(C), P_(g), P_(dV), P_(dB),
                                              P_(dC), P_(dg), T, m, H, Pd, N, stream()))
        bytes_f = 2 * V.nbytes + B.nbytes + C.nbytes + g.nbytes
        bytes_b = 3 * V.nbytes + 2 * B.nbytes + 2 * C.nbytes + 2 * g.nbytes
        tokens = T
        config = {"workload": w.name, "tokens": T, "mimo": m, "nheads": H, "headdim": Pd, "dstate": N, "dtype": "bf16"}
        kernels = {"forward": f"y_diag_fwd_fast<bf16, {m}>", "backward": f"y_diag_bwd_fast<bf16, {m}>"}
        ts = 2048

        def cpu():
            sl = lambda a: a[:ts]
            om3.y_diag(sl(inp["V"]), sl(inp["B"]), sl(inp["C"]), sl(inp["gamma"]))
            om3.y_diag_vjp(sl(inp["dY"]), sl(inp["V"]), sl(inp["B"]), sl(inp["C"]), sl(inp["gamma"]))
        cpu_units = ts
        sample = f"fp64 NumPy oracle fwd + bwd on tokens 0..{ts - 1} of {T}, all heads"
        metric = f"Mamba-3 gamma correction ({'SISO' if m == 1 else f'MIMO rank {m}'}) fwd+bwd tokens/sec (1 GB300)"
    with clocks:
        tf = _event_time(fwd, args.warmup, args.steps)
        tb = _event_time(bwd, args.warmup, args.steps)
    hbm = peaks["hbm_gbs"]
    rate_cpu, reps, el = _wall_rate(cpu, cpu_units, min(args.cpu_seconds, 10.0))
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return {
        "metric": metric, "value": tokens / ((tf + tb) * 1e-3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": tf + tb, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": config["dtype"], "data": "synthetic", "op": args.op,
        "config": {**config, "l2": "inputs larger than L2; no flush"},
        "forward": {"ms": tf, "tokens_per_s": tokens / (tf * 1e-3), "algorithmic_bytes": bytes_f,
                    "achieved_gbs": bytes_f / (tf * 1e-3) / 1e9, "kernels": kernels["forward"]},
        "backward": {"ms": tb, "tokens_per_s": tokens / (tb * 1e-3), "algorithmic_bytes": bytes_b,
                     "achieved_gbs": bytes_b / (tb * 1e-3) / 1e9, "kernels": kernels["backward"]},
        "roofline": {"bound": "hbm", "unit": "GB/s", "peak": hbm,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback",
                     "achieved": bytes_b / (tb * 1e-3) / 1e9, "frac": bytes_b / (tb * 1e-3) / 1e9 / hbm,
                     "kernel": "backward (the longer of the two)", "traffic": None},
        "gpu_launches": 4 * args.steps if args.op == "quat_scan" else 2 * args.steps,
        "clocks": clocks.summary(),
        "cpu_baseline": {"value": rate_cpu, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{sample}; {reps} repetition(s), {el:.1f} s; NumPy on one core "
                                   f"({cores} available)"},
    }


def run_moments(args, dev, peaks, peak_src, clocks):
    """ssd_state_moments on the 2.7B layer (chunk states recomputed at chunk 128,
    then the closed-form moments and the fixed-order reduction), one call per
    step; the tensor-core moment kernel also timed alone with its own events."""
    import torch

    import oracle
    from state_space_model_mamba_gb300 import ssd
    w = WORKLOADS["mamba2_2p7b"]
    inp = generate(w)
    up = lambda a, dt=torch.float32: torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
    x, B = up(inp["x"], torch.bfloat16), up(inp["B"], torch.bfloat16)
    dt, A = up(inp["dt"]), up(inp["A"])
    b, L, H, P = x.shape
    N = B.shape[3]
    m2 = torch.empty(b, H, N, N, device=dev)
    m1 = torch.empty(b, H, N, device=dev)
    cnt = torch.empty(b, device=dev, dtype=torch.int64)
    dims = ssd.dims_of(x, B, 128)
    lib = ssd.load_library()
    ws = torch.empty(lib.ssd_moments_workspace_bytes(ctypes_byref(dims), ssd.SSD_BF16), dtype=torch.uint8, device=dev)

    def call():
        ssd._check(lib.ssd_state_moments(ctypes_byref(dims), ssd.SSD_BF16, ssd._ptr(x), ssd._ptr(dt), ssd._ptr(A),
                                         ssd._ptr(B), None, None, ssd._ptr(m2), ssd._ptr(m1), ssd._ptr(cnt),
                                         ssd._ptr(ws), ws.numel(), ssd._stream_ptr(dev)))
    with clocks:
        t = _event_time(call, args.warmup, args.steps)
        timer = ssd.KernelTimer(capacity_kernels=args.steps + 4, only="moments_tc")
        with timer:
            for _ in range(args.steps):
                call()
        live = [ms for _, ms in timer.durations()]
    ssd.workspace_status(ws)
    costs = kernel_costs(w, tc=True)
    flops, byts = costs["moments"]
    km = statistics.mean(live)
    peak = peaks["bf16_tflops_sustained"]
    hs = 2

    def cpu():
        oracle.state_moments(inp["x"][:1, :, :hs], inp["dt"][:1, :hs], inp["A"][:hs], inp["B"][:1])
    rate_cpu, reps, el = _wall_rate(cpu, L * hs / H, min(args.cpu_seconds, 15.0))
    return {
        "metric": "Mamba-2 state moments (m2, m1 of every per-token state) tokens/sec (2.7B-layer shape, 1 GB300)",
        "value": w.tokens / (t * 1e-3), "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "op": args.op,
        "config": {"workload": w.name, **w.dims(), "moment_chunk": 128,
                   "l2": "inputs larger than L2; no flush",
                   "step": "ssd_state_moments: chunk states at chunk 128, closed-form moments, range reduction"},
        "roofline": {"bound": "tensor", "unit": "TFLOP/s", "peak": peak,
                     "peak_source": f"{peak_src} sustained bf16 (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback",
                     "achieved": flops / (km * 1e-3) / 1e12, "frac": flops / (km * 1e-3) / 1e12 / peak,
                     "kernel": "moments_tc", "avg_us": km * 1e3, "algorithmic_flops_per_launch": flops,
                     "algorithmic_bytes_per_launch": byts, "hbm_frac": byts / (km * 1e-3) / 1e9 / peaks["hbm_gbs"],
                     "traffic": None},
        "gpu_launches": (lib.ssd_last_launch_count()) * args.steps,
        "clocks": clocks.summary(),
        "cpu_baseline": {"value": rate_cpu, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"fp64 C oracle (per-token states, OpenMP) on batch 0, heads 0..{hs - 1} of {H}, "
                                   f"all {L} tokens; {reps} repetition(s), {el:.1f} s; scaled to tokens/s of all heads"},
    }


def ctypes_byref(dims):
    import ctypes
    return ctypes.byref(dims.c())


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--split-scan", action="store_true",
                    help="chunk states by the chunk-parallel K3 and a separate K4 pass (SSD_FLAG_SPLIT_SCAN)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--profile-case", choices=("forward", "step"), default=None,
                    help="light run for ncu captures (see the module docstring)")
    ap.add_argument("--op", choices=OPS, default=None,
                    help="measure another entry point of the library (see run_op)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.op:
        print(json.dumps(run_op(args, int(os.environ.get("LOCAL_RANK", "0")))), flush=True)
        return
    rank, world, local_rank = dist_env()
    w = WORKLOADS[args.workload]
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend=backend)
    if args.profile_case:
        if world > 1:
            ap.error("--profile-case runs on one GPU")
        print(json.dumps(run_profile_case(args, w, local_rank)), flush=True)
        return
    if args.impl == "reference":
        line = run_reference(args, w, rank, world)
    else:
        line = run_ours(args, w, rank, world, local_rank)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
