"""Throughput of the K3 LatentMoE layer on GB300 (one JSON line on stdout).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                [--workload decode_t1|decode_t64|prefill_t4096|chain8_t256|decode_t1_tier|...]

A step is one forward of the whole layer (router, permutation, routed
experts, latent norm, up projection and shared experts) over one batch of
synthetic K3-shape input. Default workload: K3 decode, T=1 token per step,
tokens rotating through a seeded pool of 64 so that different experts are
read each step, and the L2 is flushed (256 MB write) between timed steps.

value: tokens/s with inputs resident in HBM (CUDA events around each
forward, summed over K steps); e2e: the same through k3moe_forward_host
with pinned host buffers (copies inside the timed region); roofline: the
dominant kernel's algorithmic bytes per launch over its event-timed average
duration (a second pass of the same K steps with every kernel bracketed by
CUDA events; the first pass, which gives value, has no events between the
kernels) against the measured HBM copy bandwidth; cpu_baseline: the fp64
oracle on the host cores on a bounded sample of the same workload.

With torchrun (N > 1) every rank runs an independent replica of the layer
(the layer does not shard across GPUs); rank 0 prints the line.
--impl reference times the fp64 CPU oracle as the reference arm, on the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import k3synth  # noqa: E402

METRIC = "MoE-layer tokens/s at K3 shape; HBM GB/s (decode) / FP4 TFLOP/s (prefill)"
UNIT = "tokens/s"
POOL = 64
FLUSH_BYTES = 256 << 20

WORKLOADS = {
    "decode_t1": dict(T=1, layers=1, desc="K3-shape single layer, decode T=1 "
                      "(tokens rotate through a seeded pool of 64)"),
    "decode_t64": dict(T=64, layers=1, desc="K3-shape single layer, decode batch T=64, "
                       "covering construction: all 896 experts touched"),
    "prefill_t4096": dict(T=4096, layers=1, desc="K3-shape single layer, prefill T=4096, "
                          "Zipf(1.1) expert popularity via router bias"),
    "chain8_t256": dict(T=256, layers=8, desc="8 stacked K3-shape layers, T=256, RMSNorm "
                        "between layers"),
    # small case for ncu captures: K3 row shapes, 64 experts (1.2 GB), decode T=1
    "decode_t1_e64": dict(T=1, layers=1, desc="K3 row shapes with 64 routed experts, decode T=1 "
                          "(small case for profiler captures)"),
    "batch_t16_e64": dict(T=16, layers=1, desc="K3 row shapes with 64 routed experts, T=16 "
                          "(4 pairs per expert, the 32-pair n-tiles of decode T=64; small case "
                          "for profiler captures)"),
    "batch_t64_e64": dict(T=64, layers=1, desc="K3 row shapes with 64 routed experts, T=64 "
                          "(16 pairs per expert; small case for profiler captures)"),
    "prefill_t512_e64": dict(T=512, layers=1, desc="K3 row shapes with 64 routed experts, T=512 "
                             "(128 pairs per expert; small case for profiler captures)"),
    # the layer fed from the residual stream: the RMSNorm in front of the MoE
    # runs inside the first two decode kernels
    "decode_t1_residual": dict(T=1, layers=1, residual=True,
                               desc="K3-shape single layer, decode T=1 from fp32 residual-stream "
                                    "rows (RMSNorm with the post-norm gain fused into the first "
                                    "kernels; rows rotate through a seeded pool of 64)"),
    # the cumulative-weight cut of the picks (fewer experts read per token)
    "decode_t1_topp": dict(T=1, layers=1, topp=0.8,
                           desc="K3-shape single layer, decode T=1, picks cut to cumulative "
                                "weight 0.8 (renormalised; tokens rotate through a seeded pool of 64)"),
    # the model's dense feed-forward layer 0 (hidden 7168, dense_inter 33792)
    "dense_t1": dict(T=1, layers=1, dense=True,
                     desc="K3 dense feed-forward layer 0 (hidden 7168, dense_inter 33792, bf16), "
                          "decode T=1 (tokens rotate through a seeded pool of 64)"),
    "dense_t4096": dict(T=4096, layers=1, dense=True,
                        desc="K3 dense feed-forward layer 0 (hidden 7168, dense_inter 33792, bf16), "
                             "prefill T=4096"),
    # expert tier: routed experts in pinned host memory, 896 device slots
    # shared by two layers; each step is one forward of one layer (alternating)
    "decode_t1_tier": dict(T=1, layers=2, tier=896, alternate=True,
                           desc="two K3-shape layers with their routed experts in host memory "
                                "and 896 device slots (expert tier); decode T=1, steps alternate "
                                "layers, tokens from a seeded pool of 2048"),
    "decode_t64_tier": dict(T=64, layers=2, tier=896, alternate=True,
                            desc="two K3-shape layers with their routed experts in host memory "
                                 "and 896 device slots (expert tier); T=64 covering construction "
                                 "(all 896 experts per forward), steps alternate layers, so every "
                                 "forward copies in all of its experts"),
}
TIER_POOL = 2048


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]),
                float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured")
    return 6800.0, 1900.0, 1700.0, "fallback"


FP4_NOMINAL_TFLOPS = 13500.0      # dense FP4 tensor peak (nominal), context only


def roofline(kernel, model, avg_ms, hbm_peak, tc_peak, peak_src, workload, mx=False):
    """The dominant kernel against the roof it is closer to: HBM bandwidth for
    its algorithmic bytes, or the tensor peak of its operand types for its
    FLOPs: the measured sustained bf16 rate (the kernel runs inside a long
    step) for the f16/bf16 kernels, twice that (the nominal fp8 : bf16 ratio)
    for the block-scaled expert GEMMs (mx), whose two-term activations run two
    fp8 MMAs per product, so that their useful rate is at most half of it."""
    if mx and kernel in ("expert_w13_gemm", "expert_w2_gemm"):
        tc_peak = 2.0 * tc_peak
        peak_src = f"2 x {peak_src}"
    if not model:
        return {"kernel": kernel, "bound": "hbm", "achieved": None, "peak": hbm_peak,
                "unit": "GB/s", "frac": None, "traffic": None}
    byt, fl = model
    t = avg_ms / 1e3
    gbs = byt / t / 1e9
    tfl = fl / t / 1e12 if fl else 0.0
    f_hbm, f_tc = gbs / hbm_peak, (tfl / tc_peak if fl else 0.0)
    if f_tc > f_hbm:
        roof = {"kernel": kernel, "bound": "tensor", "achieved": round(tfl, 2), "peak": tc_peak,
                "unit": "TFLOP/s", "frac": round(f_tc, 4),
                "peak_source": (f"{peak_src} bf16_tflops_sustained (fp8 rate: e2m1 x e4m3 -> f32, two MMAs "
                                "per product)" if mx and kernel in ("expert_w13_gemm", "expert_w2_gemm")
                                else f"{peak_src} bf16_tflops_sustained (the kernel computes f16 x f16 -> f32)")}
    else:
        roof = {"kernel": kernel, "bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak,
                "unit": "GB/s", "frac": round(f_hbm, 4), "peak_source": f"{peak_src} hbm_gbs"}
    roof.update({"traffic": traffic_for(kernel, workload), "alg_bytes_per_launch": int(byt),
                 "flops_per_launch": int(fl), "avg_launch_ms": round(avg_ms, 5),
                 "hbm_frac": round(f_hbm, 4), "tensor_frac": round(f_tc, 4)})
    if fl:
        # against the attainable roof min(peak, arithmetic intensity x HBM bandwidth)
        ai = fl / byt
        att = min(tc_peak, ai * hbm_peak / 1e3)
        roof["attainable_tflops"] = round(att, 1)
        roof["attainable_frac"] = round(tfl / att, 4)
        roof["fp4_nominal_frac"] = round(tfl / FP4_NOMINAL_TFLOPS, 4)
        roof["fp4_attainable_frac"] = round(tfl / min(FP4_NOMINAL_TFLOPS, ai * hbm_peak / 1e3), 4)
    return roof


# ---- algorithmic traffic and arithmetic per kernel launch -------------------------
# Bytes: every weight byte the launch must read once plus its activation reads
# and result writes (no re-reads). FLOPs: 2 per multiply-add of the
# contraction (tensor-core kernels only).

def kernel_model(shape, T, n_touched):
    H, L, E, I, S, k = (shape.hidden, shape.latent, shape.n_experts, shape.moe_inter,
                        shape.shared_inter, shape.topk)
    P = T * k                                            # (token, expert) pairs
    per_w13 = 2 * (I * L // 2 + I * L // 32)             # packed W1 + W3 and their scales
    per_w2 = L * I // 2 + L * I // 32
    rd = (2 * (E * H + L * H) + 2 * T * H + 4 * T * (E + L), 2 * T * H * (E + L))
    sh = (2 * (2 * S * H) + 2 * T * H + 6 * T * S, 2 * T * H * 2 * S)
    up = (2 * (H * L + H * S) + 2 * T * (L + S) + 2 * T * H, 2 * T * (L + S) * H)
    w13 = (n_touched * per_w13 + 2 * P * L + 2 * P * I, 2 * P * L * 2 * I)
    w2 = (n_touched * per_w2 + 2 * P * I + 8 * T * L, 2 * P * I * L)
    return {
        "router_down_gemv": (rd[0], 0), "router_down_gemm": rd,
        "shared_gate_up_gemv": (sh[0] - 2 * T * S, 0), "shared_gate_up_gemm": sh,
        "route_topk": (4 * T * (E + L) + 2 * T * (L + 16) + 4 * T * L + 8 * T * k, 0),
        "perm_count": (4 * P, 0), "perm_scan": (0, 0), "perm_place": (8 * P + 8 * P, 0),
        "expert_tiles": (0, 0), "gather_latent": (4 * P * (L + 16), 0),
        "expert_w13_gemv": (w13[0] - 2 * P * L + 2 * T * L, 0), "expert_w13_gemm": w13,
        "expert_w2_gemv": (w2[0], 0), "expert_w2_gemm": w2,
        "latent_rmsnorm": (4 * T * L + 2 * T * L + 2 * L, 0),
        "norm_up_shared_gemv": (up[0] - 2 * T * (L + S) + 4 * T * (L + S) + 2 * L, 0),
        "up_shared_gemm": up,
        "chain_glue_rmsnorm": (4 * T * H, 0),
        "tier_plan": (0, 0), "tier_fill": (0, 0),   # set from the tier's counters
        # dense feed-forward layer (no routed part): S is its width; per launch
        "dense_gate_up_gemv": (2 * 2 * S * H + 2 * T * H + 4 * T * S, 0),
        "dense_down_gemv": (2 * H * S + 4 * T * S + 2 * T * H, 0),
        "dense_gate_up_gemm": sh,
        "dense_down_gemm": (2 * H * S + 2 * T * S + 2 * T * H, 2 * T * S * H),
        "residual_rmsnorm": (4 * T * H + 2 * H + 2 * T * H, 0),
    }


def layer_bytes(shape, T, n_touched):
    """Bytes of one layer's minimal traffic: every weight it reads once (the
    dense projections, the shared experts and the touched experts) plus the
    layer input and output."""
    H, L, E, I, S = shape.hidden, shape.latent, shape.n_experts, shape.moe_inter, shape.shared_inter
    if E == 0:   # dense feed-forward layer
        return 2 * 3 * S * H + 4 * T * H
    dense = 2 * (E * H + L * H + 2 * S * H + H * L + H * S)
    experts = n_touched * (3 * (I * L // 2 + I * L // 32))
    return dense + experts + 4 * T * H


# ---- inputs ----------------------------------------------------------------------

def make_inputs(workload, seed=0, layer_index=0):
    T = WORKLOADS[workload]["T"]
    if WORKLOADS[workload].get("dense"):
        shape = k3synth.K3_DENSE
        d = k3synth.make_dense_layer(shape, seed)
        x = k3synth.make_tokens(shape, seed, POOL if T == 1 else T, stream=7 if T == 1 else 13)
        return shape, d, x
    shape = (k3synth.replace(k3synth.K3, n_experts=64) if workload.endswith("_e64")
             else k3synth.K3)
    d = k3synth.make_layer(shape, seed, layer_index, k3synth.K3_RECIPE)
    if workload in ("decode_t1", "decode_t1_e64", "decode_t1_topp"):
        x = k3synth.make_tokens(shape, seed, POOL, stream=7)
    elif workload == "decode_t1_residual":
        x = k3synth.make_residual(shape, seed, POOL, stream=7)   # fp32 residual rows
    elif workload == "decode_t1_tier":
        x = k3synth.make_tokens(shape, seed, TIER_POOL, stream=17)
    elif workload in ("decode_t64", "decode_t64_tier"):
        d = k3synth.with_bias(d, np.zeros(shape.n_experts, np.float32))
        x = k3synth.covering_tokens(shape, d, seed, T)
    elif workload == "prefill_t4096":
        d = k3synth.with_bias(d, k3synth.zipf_bias(shape, seed, layer_index, k3synth.K3_ZIPF_ALPHA))
        x = k3synth.make_tokens(shape, seed, T, stream=11)
    elif workload.endswith("_e64"):
        x = k3synth.make_tokens(shape, seed, T, stream=15)
    else:
        x = k3synth.make_tokens(shape, seed, T, stream=13)
    return shape, d, x


class ClockSampler:
    """Polls nvidia-smi for SM clocks and throttle reasons in a background
    thread; stop() keeps the samples taken inside [start, stop] (widened by one
    polling period so a short region still gets its nearest samples)."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.stop_flag = threading.Event()
        self.t = None

    def _poll(self):
        while not self.stop_flag.is_set():
            try:
                out = subprocess.run(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                      "--format=csv,noheader,nounits"], capture_output=True,
                                     text=True, timeout=10).stdout.strip()
                self.samples.append((time.perf_counter(), out))
            except (OSError, subprocess.TimeoutExpired):
                self.samples.append((time.perf_counter(), ""))
                return
            time.sleep(0.05)

    def start(self):
        self.t = threading.Thread(target=self._poll, daemon=True)
        self.t.start()
        t0 = time.perf_counter()
        while not self.samples and time.perf_counter() - t0 < 10:
            time.sleep(0.01)
        self.t_start = time.perf_counter()

    def stop(self):
        t_end = time.perf_counter()
        time.sleep(0.3)
        self.stop_flag.set()
        self.t.join(timeout=15)
        period = 0.3
        sm, smax, reasons, n = [], None, set(), 0
        for ts, line in self.samples:
            if not (self.t_start - period <= ts <= t_end + period):
                continue
            f = [v.strip() for v in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                smax = float(f[1])
            except ValueError:
                continue
            n += 1
            for name, v in zip(self.NAMES, f[3:7]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": n,
                "window_s": round(t_end - self.t_start, 3)}


def traffic_for(kernel, workload):
    """DRAM bytes per launch of `kernel` from a committed ncu summary, if the
    kernel's source is unchanged since the capture (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        table = json.load(f)
    ent = table.get(f"{kernel}@{workload}")
    if not ent:
        return None
    src = os.path.join(ROOT, "mxfp4_routed_expert_gb300", "csrc", ent["source"])
    if not os.path.exists(src):
        return None
    with open(src, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != ent["sha256"]:
            return None
    return ent["bytes_per_launch"]


def max_over_ranks(value, device="cpu"):
    """The largest `value` over the ranks of the process group (the slowest
    rank sets a whole-job time); the value itself without a group or with one
    rank. `device`: where the reduction runs ("cuda" under NCCL, "cpu" under
    gloo)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, tokens_per_step, steps, seconds):
    """Tokens per second of the whole job: every rank runs `steps` steps of
    `tokens_per_step` tokens on its own replica, timed by the slowest rank."""
    return world * tokens_per_step * steps / seconds


def host_link_gbs():
    """Pinned host -> device copy bandwidth (1 GiB, best of 3, CUDA events)."""
    import torch
    src = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
    dst = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    best = 0.0
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        best = max(best, src.numel() / (a.elapsed_time(b) / 1e3) / 1e9)
    del src, dst
    return round(best, 1)


# ---- oracle timing (CPU baseline and reference arm) ----------------------------------

def oracle_x(workload, shape, x):
    """bf16 bits of the layer input the oracle takes: the workload's tokens, or
    for a residual workload the oracle's own RMSNorm of the residual rows."""
    if not WORKLOADS[workload].get("residual"):
        return x
    import oracle
    return oracle.round_bf16(oracle.residual_input(x, k3synth.post_norm_gain(shape, 0), shape.rms_eps))


def oracle_rows(shape, d, x, rows):
    """The oracle on tokens `rows` of x: the LatentMoE layer, or the dense
    feed-forward layer for a configuration without a routed part."""
    import oracle
    if shape.n_experts == 0:
        return oracle.dense_ffn(x[rows], d["sh_w1"], d["sh_w3"], d["sh_w2"], shape.situ_b1, shape.situ_b2)
    return oracle.layer_forward(shape, d, x, rows=rows)


def time_oracle(shape, d, x, n_tokens):
    import oracle
    oracle.build()
    rows = (np.arange(n_tokens) % x.shape[0]).astype(np.int32)   # the pool repeats when it is smaller
    t0 = time.perf_counter()
    oracle_rows(shape, d, x, rows)
    dt = time.perf_counter() - t0
    return rows.size, dt


def omp_threads(n_rows):
    n = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return max(1, min(n, n_rows))


# ---- native arm ------------------------------------------------------------------------

def run_native(args, rank, world):
    import torch
    import mxfp4_routed_expert_gb300 as km
    from mxfp4_routed_expert_gb300 import tier_trace
    from mxfp4_routed_expert_gb300 import build as kbuild
    kbuild.build()
    dev = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(dev)
    wl = WORKLOADS[args.workload]
    T, n_layers = wl["T"], wl["layers"]

    shape, d0, xpool = make_inputs(args.workload)
    h = km.k3moe_create(km.make_config(shape, max_layers=n_layers, max_tokens=T, device=dev))
    km.k3moe_set_expert_path(h, {"auto": km.K3MOE_EXPERT_AUTO, "gemv": km.K3MOE_EXPERT_GEMV,
                                 "gemm": km.K3MOE_EXPERT_GEMM, "mx": km.K3MOE_EXPERT_MX}[args.expert_path])
    alternate = wl.get("alternate", False)   # one layer per step, layers in turn (else a chain)
    if wl.get("topp"):
        km.k3moe_set_topp(h, wl["topp"])
    if wl.get("tier"):
        km.k3moe_set_expert_tier(h, wl["tier"])
    w, keep = km.layer_weights(d0, shape.n_experts, km.K3MOE_HOST)
    km.k3moe_load_layer(h, 0, w)
    del keep
    oracle_layer = d0
    xpools = [xpool]
    for li in range(1, n_layers):
        _, dl, xl = make_inputs(args.workload, layer_index=li)
        w, keep = km.layer_weights(dl, shape.n_experts, km.K3MOE_HOST)
        km.k3moe_load_layer(h, li, w)
        xpools.append(xl)
        del keep, dl
    if not alternate:
        xpools = xpools[:1]

    residual = wl.get("residual", False)
    if residual:
        km.k3moe_load_post_norm(h, 0, k3synth.post_norm_gain(shape, 0))
        xs = [torch.from_numpy(np.ascontiguousarray(xp, np.float32)).cuda() for xp in xpools]
    else:
        xs = [torch.from_numpy(xp.view(np.int16).copy()).cuda() for xp in xpools]
    npool = xs[0].shape[0] // T
    y = torch.empty((T, shape.hidden), dtype=torch.int16, device="cuda")
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    counts_log = torch.empty((args.steps, shape.n_experts), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def fwd(i):
        if alternate:
            li = i % n_layers
            j = (i // n_layers) % npool
            km.k3moe_forward(h, li, xs[li][j * T:j * T + T], y, T, stream)
            return
        xi = xs[0][(i % npool) * T:(i % npool) * T + T]
        if residual:
            km.k3moe_forward_residual(h, 0, xi, y, T, stream)
        elif n_layers > 1:
            km.k3moe_forward_chain(h, 0, n_layers, xi, y, T, stream)
        else:
            km.k3moe_forward(h, 0, xi, y, T, stream)

    for i in range(args.warmup):
        flush.zero_()
        fwd(i)
    torch.cuda.synchronize()
    assert km.k3moe_sync_status(h) == 0

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(dev)

    def timed_pass(profiled):
        if profiled:
            km.k3moe_set_profiling(h, True)
        for i in range(args.steps):
            flush.zero_()                      # L2 flush, outside the timed events
            starts[i].record(stream)
            fwd(args.warmup + i)
            ends[i].record(stream)
            km.k3moe_get_routing(h, counts=counts_log[i], stream=stream)
        torch.cuda.synchronize()
        stats = None
        if profiled:
            stats = km.k3moe_profile_read(h)
            km.k3moe_set_profiling(h, False)
        times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        return sum(times), stats, times

    # pass 1 (the measurement): no per-kernel events between the launches
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    tier0 = km.k3moe_get_tier_stats(h) if wl.get("tier") else None
    clocks.start()
    total_ms, _, step_times = timed_pass(False)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    tier1 = km.k3moe_get_tier_stats(h) if wl.get("tier") else None
    # pass 2: the same steps with every kernel bracketed by CUDA events on its
    # launching stream (per-kernel durations for the roofline)
    prof_ms, stats, _ = timed_pass(True)
    st = km.k3moe_sync_status(h)
    assert st == 0, km.strerror(st)
    if world > 1:
        total_ms = max_over_ranks(total_ms, "cuda")
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(world, T, args.steps, total_ms / 1e3)

    if args.dump_trace and rank == 0:
        # one forward per step: its layer (a chain exposes its last layer's routing)
        step_layer = [(args.warmup + i) % n_layers if alternate else n_layers - 1 for i in range(args.steps)]
        tier_trace.save_counts(args.dump_trace, step_layer, counts_log.cpu().numpy())
    touched = (counts_log.cpu().numpy() > 0).sum(1)
    n_touched = float(touched.mean())
    hbm_peak, bf16_peak, bf16_sust, peak_src = measured_peaks()
    # whether the grouped expert GEMM ran in its block-scaled form (the
    # library's automatic choice: fewer than 64 pairs per expert on average)
    P_ = T * shape.topk
    mx_path = shape.n_experts > 0 and P_ >= 128 and (
        args.expert_path == "mx" or (args.expert_path == "auto" and T >= 16 and P_ < 64 * shape.n_experts))
    model = kernel_model(shape, T, n_touched)
    tier = None
    if wl.get("tier"):
        tier2 = km.k3moe_get_tier_stats(h)   # after the profiled pass: its own counts
        fill_per_step = (tier2["bytes_filled"] - tier1["bytes_filled"]) / args.steps
        model["tier_fill"] = (2 * fill_per_step, 0)   # read over the host link, written to HBM
        d = {k: tier1[k] - tier0[k] for k in ("hits", "misses", "bytes_filled")}
        link = host_link_gbs()
        tier = {"slots": tier1["slots"], "hits": d["hits"], "misses": d["misses"],
                "hit_rate": round(d["hits"] / max(1, d["hits"] + d["misses"]), 4),
                "bytes_filled_per_step": int(d["bytes_filled"] / args.steps),
                "host_link_copy_gbs": link}
    by_name = {n: (l, ms) for n, l, ms in stats}
    ranked = sorted(((ms, n) for n, (l, ms) in by_name.items()), reverse=True)
    dom = ranked[0][1]
    launches, dom_ms = by_name[dom]
    avg_ms = dom_ms / launches
    if dom == "tier_fill":
        # the copy of missed experts reads host memory over the host link
        gbs = (model["tier_fill"][0] / 2) / (avg_ms / 1e3) / 1e9
        roof = {"kernel": dom, "bound": "host_link", "achieved": round(gbs, 1),
                "peak": tier["host_link_copy_gbs"], "unit": "GB/s",
                "frac": round(gbs / tier["host_link_copy_gbs"], 4),
                "peak_source": "pinned host -> device copy measured in this run", "traffic": None,
                "alg_bytes_per_launch": int(model["tier_fill"][0] / 2), "flops_per_launch": 0,
                "avg_launch_ms": round(avg_ms, 5)}
    else:
        roof = roofline(dom, model.get(dom), avg_ms, hbm_peak, bf16_sust, peak_src, args.workload,
                        mx=mx_path)
    layers_per_step = 1 if alternate else n_layers
    step_bytes = layer_bytes(shape, T, n_touched) * layers_per_step
    layer_gbs = step_bytes / (ms_per_step / 1e3) / 1e9
    kernels = {}
    for n, (l, ms) in by_name.items():
        ent = {"launches": l, "avg_ms": round(ms / l, 5),
               "share": round(ms / sum(m for _, m in by_name.values()), 4)}
        byt, fl = model.get(n, (0, 0))
        if byt:
            ent["gbs"] = round(byt / (ms / l / 1e3) / 1e9, 1)
        if fl:
            ent["tflops"] = round(fl / (ms / l / 1e3) / 1e12, 2)
        kernels[n] = ent
    kernels["_profiled_pass_ms_per_step"] = round(prof_ms / args.steps, 5)
    gpu_launches = sum(l for l, _ in by_name.values())

    # ---- the cut's effect on y over the pool (the pages' check before using a p) -------
    topp = None
    if wl.get("topp"):
        outs = []
        for p_ in (wl["topp"], 0.0):
            km.k3moe_set_topp(h, p_)
            ys = []
            for i in range(npool):
                fwd(i)
                ys.append(y.clone())
            torch.cuda.synchronize()
            outs.append(torch.stack(ys).view(torch.bfloat16).float().cpu().numpy().reshape(npool, -1))
        km.k3moe_set_topp(h, wl["topp"])
        yc, yf = outs
        rel = float(np.max(np.abs(yc - yf)) / np.max(np.abs(yf)))
        cos = [float(np.dot(a, b) / (np.linalg.norm(a) * np.linalg.norm(b))) for a, b in zip(yc, yf)]
        topp = {"p": wl["topp"], "experts_per_token": n_touched / T,
                "y_maxrel_vs_all_picks": round(rel, 5), "y_cos_vs_all_picks_min": round(min(cos), 6),
                "y_cos_vs_all_picks_mean": round(float(np.mean(cos)), 6)}

    # ---- e2e through the public host-buffer entry point --------------------------------
    e2e = None
    if n_layers == 1 and not residual and not args.no_e2e:
        xh = torch.from_numpy(xpool.view(np.int16).copy()).pin_memory()
        yh = torch.empty((T, shape.hidden), dtype=torch.int16).pin_memory()
        # the step's input rows are views of one pinned buffer, made before the
        # loop (a serving loop holds its buffers); the copy in, the layer and
        # the write of y stay inside the timed call
        xrows = [xh[j * T:j * T + T] for j in range(npool)]
        for i in range(2):
            km.k3moe_forward_host(h, 0, xrows[i % npool], yh, T, stream)
        tot = 0.0
        for i in range(args.steps):
            flush.zero_()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            km.k3moe_forward_host(h, 0, xrows[i % npool], yh, T, stream)
            tot += time.perf_counter() - t0
        if world > 1:
            tot = max_over_ranks(tot, "cuda")
        e2e = {"value": round(whole_job_rate(world, T, args.steps, tot), 2), "unit": UNIT,
               "h2d_bytes_per_step": T * shape.hidden * 2,
               "d2h_bytes_per_step": T * shape.hidden * 2}

    # ---- CPU baseline: the oracle on a bounded sample ---------------------------------------
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        n_tok = 320                      # about 10-20 s of the oracle on the machine's cores
        xs_host = oracle_x(args.workload, shape, xpool if T == 1 else xpool[:T])
        nrow, dt = time_oracle(shape, oracle_layer, xs_host, n_tok)
        cpu = {"value": round(nrow / dt / layers_per_step, 4), "unit": UNIT,
               "cores": omp_threads(nrow), "kind": "oracle",
               "sample": f"{nrow} token rows of the workload ({min(nrow, xs_host.shape[0])} distinct) "
                         f"through one layer (fp64 C oracle, OpenMP over tokens), {dt:.1f} s"
                         + (f"; chain value = per-layer rate / {n_layers}" if layers_per_step > 1 else "")}
    km.k3moe_destroy(h)
    if rank != 0:
        return None
    return {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "mxfp4w-bf16a-f32acc",
        "data": "synthetic (seeded K3-shape layer, random-init weights)",
        "config": {"workload": args.workload, "description": wl["desc"], "tokens_per_step": T,
                   "layers": n_layers, "hidden": shape.hidden, "latent": shape.latent,
                   "n_experts": shape.n_experts, "topk": shape.topk,
                   "moe_inter": shape.moe_inter, "shared_inter": shape.shared_inter,
                   "parallelism": f"replicas x{world}",
                   "l2": "256 MB flush between timed steps; working set > L2",
                   "experts_touched_per_step": n_touched},
        "expert_gemm": None if shape.n_experts == 0 else
                       ("block-scaled (kind::mxf8f6f4, two-term MXFP8 activations)" if mx_path else
                        ("f16 (e2m1 widened on the SM)" if shape.n_experts and T * shape.topk >= 128 and
                         args.expert_path != "gemv" and (T >= 16 or args.expert_path == "gemm") else "per-pair GEMVs")),
        "hbm_gbs_layer": round(layer_gbs, 1), "hbm_frac_layer": round(layer_gbs / hbm_peak, 4),
        "step_ms": {"median": round(float(np.median(step_times)), 5),
                    "p10": round(float(np.percentile(step_times, 10)), 5),
                    "p90": round(float(np.percentile(step_times, 90)), 5)},
        "roofline": roof, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": gpu_launches, "clocks": clk,
        **({"tier": tier} if tier else {}),
        **({"topp": topp} if topp else {}),
    }


# The K3 configurations timed beside the decode T=1 headline, each with at
# most this many timed steps (a step of the chain is eight layers).
EXTRA_CONFIGS = (("decode_t64", 30), ("prefill_t4096", 15), ("chain8_t256", 6))
EXTRA_KEYS = ("value", "unit", "ms_per_step", "steps", "warmup", "expert_gemm", "hbm_gbs_layer", "hbm_frac_layer", "step_ms",
              "roofline", "kernels", "e2e", "gpu_launches", "clocks", "config")


def run_extra_configs(args, rank, world):
    """The other K3 configurations, each timed like the headline (warm-up,
    L2 flush between steps, CUDA events, clocks sampled, a profiled second
    pass for the per-kernel table), in the same process one after another;
    no CPU baseline (the headline carries it)."""
    import torch
    extra = {}
    for wl, cap in EXTRA_CONFIGS:
        sub = argparse.Namespace(**vars(args))
        sub.workload = wl
        sub.steps = max(5, min(args.steps, cap))
        sub.no_cpu_baseline = True
        sub.dump_trace = ""
        r = run_native(sub, rank, world)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        if r is not None:
            extra[wl] = {k: r[k] for k in EXTRA_KEYS if k in r}
    return extra


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is one token of the workload
    (a bounded sample; one K3 token is seconds of fp64 work). The K steps' tokens
    go to the oracle as one batch, spread over the host cores by its OpenMP
    loop over tokens (each token's arithmetic unchanged), so that K steps end
    within minutes; the value is tokens per second of that batch."""
    wl = WORKLOADS[args.workload]
    T, n_layers = wl["T"], wl["layers"]
    layers_per_step = 1 if wl.get("alternate") else n_layers
    shape, d, x = make_inputs(args.workload)
    x = oracle_x(args.workload, shape, x)
    import oracle
    oracle.build()
    per = 1
    oracle_rows(shape, d, x, (np.arange(args.warmup) % x.shape[0]).astype(np.int32))
    rows = ((np.arange(args.steps * per) + args.warmup) % x.shape[0]).astype(np.int32)
    t0 = time.perf_counter()
    oracle_rows(shape, d, x, rows)
    dt = time.perf_counter() - t0
    value = per * args.steps / dt / layers_per_step
    cores = omp_threads(per * args.steps)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded K3-shape layer, random-init weights)",
        "config": {"workload": args.workload, "description": wl["desc"],
                   "tokens_per_step": T, "layers": n_layers},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "kind": "oracle",
                         "cores": cores,
                         "sample": f"{per} token per step through one layer (fp64 C oracle), the "
                                   f"{args.steps} steps' tokens as one batch over {cores} cores"
                                   + (f"; chain value = per-layer rate / {n_layers}" if layers_per_step > 1 else "")},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=list(WORKLOADS), default="decode_t1")
    ap.add_argument("--expert-path", choices=["auto", "gemv", "gemm", "mx"], default="auto",
                    help="routed-expert kernels: auto (grouped GEMM from T >= 16), per-pair GEMVs, the "
                         "grouped GEMM, or its block-scaled form (mxf8f6f4, two-term MXFP8 activations)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--dump-trace", default="",
                    help="write each timed step's layer and expert counts to this .npz (a routing trace "
                         "for python -m mxfp4_routed_expert_gb300.tier_trace)")
    ap.add_argument("--no-extra", action="store_true",
                    help="with the default workload, skip the other K3 configurations (decode T=64, "
                         "prefill T=4096, 8-layer chain) that the line otherwise carries under 'configs'")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    out = run_native(args, rank, world)
    if args.workload == "decode_t1" and not args.no_extra:
        extra = run_extra_configs(args, rank, world)
        if out is not None:
            out["configs"] = extra
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
