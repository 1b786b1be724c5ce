"""Throughput of the routed MoE FFN layer forward on GB300.

One step = one pass of the whole layer over one batch of synthetic tokens:
router (gating GEMM, scores, top-k, gates), dispatch (counts, scan,
permutation), Linear1 + SwiGLU (rows gathered by the permutation), Linear2
(routed experts and, where the layer has one, the shared expert),
gate-weighted combine.  Default workload: the largest layer, T=16384 (B=2,
S=8192), H=8192, 64 experts top-2 with softmax gates, I=22016; then, on the
same GPU, the V4-Pro-shaped layer (T=4096, H=7168, 384 experts top-6, I=2048,
one shared expert, sigmoid affinity with selection bias, alpha 2.5, Zipf(1.1)
load), reported under "other_workloads".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c5] [--also c3]
    python bench.py --impl reference ...   # the CPU oracle on this host's cores

Under torchrun each rank runs its own batch (weak scaling, no collective in
the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
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

METRIC = "MoE-layer tokens/s @1 GB300; grouped-GEMM TFLOP/s and % of bf16 peak"
UNIT = "tokens/s"

WORKLOAD_TEXT = {
    "c1": "tiny layer T=128 H=256 E=8 top-2 I=128, sigmoid routing",
    "c2": "given-routing layer T=4096 H=4096 E=32 top-8 I=1536 (E, G inputs)",
    "c3": "V4-Pro-shaped layer T=4096 H=7168 E=384 top-6 I=2048 +1 shared, sigmoid+bias, alpha 2.5, Zipf(1.1) load",
    "c4": "hash-routed layer, V4-Pro shapes, tid2eid[128000, 6]",
    "c5": "large-FFN layer T=16384 H=8192 E=64 top-2 I=22016, softmax gates",
    "c3_sp": "V4-Pro-shaped layer with the pages' sqrt-softplus affinity",
    "c3p": "V4-Pro expert shapes, T=512 E=48 (profiling size)",
    "c5p": "large-FFN expert shapes, T=1024 E=4 top-2 (~512 rows per expert; profiling size)",
    "c5x": "large-FFN hidden size with token rows beyond L2, T=9216 H=8192 E=8 top-2 I=256 (parity case)",
    "c5x_sh": "c5x with a shared expert (parity case)",
    "c3_f3072": "V4-Pro-shaped layer at the pages' expert width f=3072 (T=4096 H=7168 E=384 top-6 I=3072 +1 shared)",
    "c3r": "V4-Pro router at full size with I=64 (profiling size for the routing kernels)",
    "c3_q": "V4-Pro-shaped layer, A8W8-INT form (int8 weights, per-token int8 activations), no shared expert",
    "c2_q": "given-routing layer, A8W8-INT form",
    "c3_mx": "V4-Pro-shaped layer, MXFP8 form (E4M3 codes, E8M0 scales per 32), no shared expert",
    "c2_mx": "given-routing layer, MXFP8 form (E4M3)",
    "c3p_mx": "V4-Pro expert shapes, T=512 E=48, MXFP8 form (profiling size)",
    "c3p_q": "V4-Pro expert shapes, T=512 E=48, A8W8-INT form (profiling size)",
    "c3p_mxa4": "V4-Pro expert shapes, T=512 E=48, A4W4-FP form (profiling size)",
    "c3_mx4": "V4-Pro-shaped layer, A8W4-FP form (E4M3 activations, E2M1 weights, E8M0 scales), no shared expert",
    "c3_mxa4": "V4-Pro-shaped layer, A4W4-FP form (E2M1 activations and weights), no shared expert",
    "c2_mx4": "given-routing layer, A8W4-FP form",
}


def synth_mx_format(cfg):
    """Activation element format of an MX workload ('e4m3', 'e5m2', 'e2m1'), else None."""
    import synth
    return synth.mx_format(cfg.get("quant"))


def synth_mx_weight_format(cfg):
    import synth
    return synth.mx_weight_format(cfg.get("quant"))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples every 20 ms while running; summary of the samples
    taken between mark_start() and mark_end()."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.rows, self.t0, self.t1 = [], None, None
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def summary(self):
        if self.proc is None:
            return {"unavailable": "nvidia-smi not found"}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        inside = [r for t, r in self.rows if self.t0 is not None and self.t0 <= t <= (self.t1 or t)]
        rows = inside if inside else [r for _, r in self.rows]
        if not rows:
            return {"unavailable": "no samples"}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows), "samples_in_timed_region": len(inside)}


# ------------------------------------------------------------------ ranks
def rank_seeds(rank: int, base: int = 1234):
    """(weight seed, token seed) of a rank: one model everywhere, one token
    batch per rank."""
    return base, base + rank


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of each rank's value (the job is as slow as its slowest rank)."""
    if world <= 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ our arm
def route_launches(c):
    """Kernels moe_route launches: the fused router (gating GEMM with the
    decision in its epilogue) and, for top-k, the float64 re-decision of close
    tokens; layers of more than 384 experts take the general path (Wg
    transpose, gating GEMM, selection, re-decision; hash: GEMM, selection).
    The forward adds count, scan, place, Linear1 (row gather fused, or the
    row copy before it: forward_row_copy), Linear2 and combine; A8W8 adds the
    token and the activation quantisation, MX the token one."""
    if c["routing"] == "given":
        return 0
    fused = c["E"] <= 384 and c["E"] % 8 == 0
    if c["routing"] == "hash":
        return 1 if fused else 2
    return 2 if fused else 4


def forward_row_copy(c):
    """1 where the bf16 forward copies the token rows into expert order before
    Linear1 (the experts average two 128-row tiles or more and X exceeds
    L2: Linear1 then loads them by TMA), else 0; the library's criterion."""
    import torch
    l2 = torch.cuda.get_device_properties(0).L2_cache_size if torch.cuda.is_available() else 0
    return int(c["T"] * c["k"] >= 256 * c["E"] and c["T"] * c["H"] * 2 > l2)


def build_step(moe, dd, p, ws, stage_events=None):
    c = dd["cfg"]
    routed = c["routing"] != "given"
    E_ids = dd["E_ids"] if not routed else dd["_E_ids"]
    G = dd["G"] if not routed else dd["_G"]

    def step(X=None, Y=None, route_events=None):
        X = dd["X"] if X is None else X
        Y = dd["_Y"] if Y is None else Y
        if routed:
            if route_events:
                route_events[0].record()
            if c["routing"] == "hash":
                moe.moe_route(p, X, dd["Wg"], None, dd["token_ids"], dd["tid2eid"], c["V"], E_ids, G, ws)
            else:
                moe.moe_route(p, X, dd["Wg"], dd["bias"], None, None, 0, E_ids, G, ws)
            if route_events:
                route_events[1].record()
        if c.get("quant") == "a8w8":
            moe.moe_forward_a8w8(p, X, E_ids, G, dd["W1"], dd["S1"], dd["W2"], dd["S2"], Y,
                                 dd["_ws_q"], stage_events)
        elif synth_mx_format(c):
            moe.moe_forward_mx(p, moe.MX_FORMATS[synth_mx_format(c)], X, E_ids, G, dd["W1"], dd["S1"],
                               dd["W2"], dd["S2"], Y, dd["_ws_q"], stage_events,
                               wfmt=moe.MX_FORMATS[synth_mx_weight_format(c)])
        elif stage_events is not None:
            moe.moe_forward_timed(p, X, E_ids, G, dd["W1"], dd["W2"], dd["Ws1"], dd["Ws2"], Y, ws,
                                  stage_events)
        else:
            moe.moe_forward(p, X, E_ids, G, dd["W1"], dd["W2"], dd["Ws1"], dd["Ws2"], Y, ws)
    return step


def run_ours(args, rank, world, local_rank, workload=None, with_cpu=True):
    import torch
    import mixture_experts_ffn_route_gb300 as moe
    from mixture_experts_ffn_route_gb300 import accounting
    import synth

    workload = workload or args.workload
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    moe.lib()
    wseed, tseed = rank_seeds(rank)
    dd = synth.make_inputs_torch(workload, seed=wseed, token_seed=tseed, device=dev)
    c = dd["cfg"]
    T, H, E, k, I = c["T"], c["H"], c["E"], c["k"], c["I"]
    has_shared = c["shared"]
    p = moe.params_from_config(c)
    ws = moe.alloc_workspace(p, dev)
    quant = c.get("quant") == "a8w8"
    mx = synth_mx_format(c)
    if quant:
        dd["_ws_q"] = moe.alloc_workspace_a8w8(p, dev)
    if mx:
        dd["_ws_q"] = moe.alloc_workspace_mx(p, dev)
    dd["_E_ids"] = torch.empty((T, k), dtype=torch.int32, device=dev)
    dd["_G"] = torch.empty((T, k), dtype=torch.float32, device=dev)
    dd["_Y"] = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    routed = c["routing"] != "given"

    # events must exist before their handles go to the library
    K = args.steps
    st_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    rt_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for evs in st_ev + rt_ev:
        for ev in evs:
            ev.record()
    plain_step = build_step(moe, dd, p, ws)
    sampler = ClockSampler(local_rank) if rank == 0 else None

    for _ in range(args.warmup):
        plain_step()
    moe.moe_sync_status(ws)

    E_now = dd["_E_ids"] if routed else dd["E_ids"]
    counts = torch.bincount(E_now.reshape(-1).long(), minlength=E).cpu().numpy()

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    for i in range(K):
        build_step(moe, dd, p, ws, stage_events=st_ev[i])(route_events=rt_ev[i] if routed else None)
    t_end.record()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_end()
    moe.moe_sync_status(ws)
    if quant or mx:
        moe.moe_sync_status(dd["_ws_q"])
    ms = max_over_ranks(t_start.elapsed_time(t_end) / K, world, dev)

    # optionally, the same step captured once in a CUDA graph and replayed K
    # times (what a launch-bound small batch gains from it)
    graph_ms = None
    if args.graph:
        gs = torch.cuda.Stream()
        gs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(gs):
            plain_step()
        torch.cuda.current_stream().wait_stream(gs)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            plain_step()
        for _ in range(args.warmup):
            graph.replay()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record()
        for _ in range(K):
            graph.replay()
        g1.record()
        torch.cuda.synchronize()
        moe.moe_sync_status(ws)
        graph_ms = max_over_ranks(g0.elapsed_time(g1) / K, world, dev)

    def avg(evs, a, b):
        return sum(e[a].elapsed_time(e[b]) for e in evs) / len(evs)
    stages = {"dispatch": avg(st_ev, 0, 1), "gemm1_swiglu": avg(st_ev, 1, 2),
              "gemm2": avg(st_ev, 2, 3), "combine": avg(st_ev, 3, 4)}
    if quant:
        stages = {"dispatch_quant": stages["dispatch"], "gemm1_swiglu": stages["gemm1_swiglu"],
                  "quant_gemm2": stages["gemm2"], "combine": stages["combine"]}
    if mx:
        stages = {"dispatch_quant": stages["dispatch"], "gemm1_swiglu_quant": stages["gemm1_swiglu"],
                  "gemm2": stages["gemm2"], "combine": stages["combine"]}
    if routed:
        stages = {"route": avg(rt_ev, 0, 1), **stages}

    # ---- end to end through the C ABI with host buffers (pinned) each step.
    # A serving loop: step i's token rows (and given ids / gates, or hash token
    # ids) are copied host->device, the layer runs, and Y is copied back to
    # pinned host memory.  Copies run on a second stream into two device
    # slots, so the next step's input copy and the previous step's output copy
    # overlap this step's compute; every copy of every step is inside the
    # timed region.
    X_host = torch.empty((T, H), dtype=torch.bfloat16, pin_memory=True)
    X_host.copy_(dd["X"])
    Y_host = torch.empty((T, H), dtype=torch.bfloat16, pin_memory=True)
    in_keys = ["X"] + {"given": ["E_ids", "G"], "hash": ["token_ids"]}.get(c["routing"], [])
    host_in = {key: (X_host if key == "X" else dd[key].cpu().pin_memory()) for key in in_keys}
    slots = []
    for _ in range(2):
        dslot = dict(dd)
        for key in in_keys:
            dslot[key] = torch.empty_like(dd[key])
        dslot["_Y"] = torch.empty_like(dd["_Y"])
        slots.append((dslot, build_step(moe, dslot, p, ws)))
    h2d = sum(host_in[key].numel() * host_in[key].element_size() for key in in_keys)
    d2h = Y_host.numel() * 2
    comp = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    ev = lambda: [torch.cuda.Event() for _ in range(2)]  # noqa: E731
    in_ready, in_free, y_ready, y_free = ev(), ev(), ev(), ev()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(comp)

    def h2d_copy(i):
        sl = i % 2
        copy.wait_stream(comp) if i == 0 else None
        with torch.cuda.stream(copy):
            if i >= 2:
                copy.wait_event(in_free[sl])  # step i - 2 has read this slot
            for key in in_keys:
                slots[sl][0][key].copy_(host_in[key], non_blocking=True)
            in_ready[sl].record(copy)

    h2d_copy(0)
    for i in range(K):
        sl = i % 2
        if i + 1 < K:
            h2d_copy(i + 1)
        comp.wait_event(in_ready[sl])
        if i >= 2:
            comp.wait_event(y_free[sl])  # Y of step i - 2 is on the host
        slots[sl][1]()
        in_free[sl].record(comp)
        y_ready[sl].record(comp)
        with torch.cuda.stream(copy):
            copy.wait_event(y_ready[sl])
            Y_host.copy_(slots[sl][0]["_Y"], non_blocking=True)
            y_free[sl].record(copy)
    comp.wait_stream(copy)
    e1.record(comp)
    torch.cuda.synchronize()
    moe.moe_sync_status(ws)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / K, world, dev)

    if rank != 0:
        return None
    pk = peaks()
    if quant:
        g1_bytes = accounting.gemm1_bytes(counts, H, I, has_shared, T, w_bytes=1, x_bytes=2, act_bytes=4)
        g2_bytes = accounting.gemm2_bytes(counts, H, I, has_shared, T, w_bytes=1, act_bytes=2,
                                          out_bytes=accounting.BF16)
    elif mx:
        ab = accounting.MX4 if mx == "e2m1" else accounting.MX8
        wb = accounting.MX4 if synth_mx_weight_format(c) == "e2m1" else accounting.MX8
        g1_bytes = accounting.gemm1_bytes(counts, H, I, has_shared, T, w_bytes=wb, x_bytes=ab, act_bytes=ab)
        g2_bytes = accounting.gemm2_bytes(counts, H, I, has_shared, T, w_bytes=wb, act_bytes=ab,
                                          out_bytes=accounting.BF16)
    else:
        g1_bytes = accounting.gemm1_bytes(counts, H, I, has_shared, T)
        # Linear2 writes fp32 rows (top-1 without a shared expert: bf16 rows of Y)
        g2_bytes = accounting.gemm2_bytes(counts, H, I, has_shared, T,
                                          out_bytes=accounting.BF16 if (k == 1 and not has_shared) else 4)
    g1_flops = accounting.gemm1_flops(counts, H, I, has_shared, T)
    g2_flops = accounting.gemm2_flops(counts, H, I, has_shared, T)
    g1_s = stages["gemm1_swiglu_quant" if mx else "gemm1_swiglu"] / 1e3
    g2_s = stages["quant_gemm2" if quant else "gemm2"] / 1e3
    gemm_tflops = (g1_flops + g2_flops) / (g1_s + g2_s) / 1e12
    # the dominant kernel: Linear1 + SwiGLU.  Weight streaming bounds it when the
    # arithmetic intensity is below the ridge point.
    ai = g1_flops / g1_bytes
    # the FP8 block-scaled tensor rate is twice the bf16 rate (nominal 4.5 vs
    # 2.25 PFLOP/s dense): its peak is the measured bf16 figure times 2
    tc_peak = pk["bf16_tflops_sustained"] * (2 if mx else 1)
    ridge = tc_peak * 1e12 / (pk["hbm_gbs"] * 1e9)
    if ai < ridge:
        achieved = g1_bytes / g1_s / 1e9
        roof = {"kernel": "grouped Linear1 + SwiGLU (gemm_tc_kernel<1>)", "bound": "hbm",
                "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": None,
                "algorithmic_bytes_per_launch": int(g1_bytes),
                "peak_source": pk["source"] + " hbm_gbs"}
    else:
        achieved = g1_flops / g1_s / 1e12
        peak = tc_peak
        roof = {"kernel": "grouped Linear1 + SwiGLU (gemm_tc_kernel<1>)", "bound": "tensor",
                "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": None,
                "algorithmic_flops_per_launch": int(g1_flops),
                "peak_source": pk["source"] + " bf16_tflops_sustained" + (" x 2 (fp8)" if mx else "")}
    if not quant and not mx:
        roof["traffic"] = load_traffic(workload, g1_bytes)
    if quant:
        roof["kernel"] = "grouped A8W8 Linear1 + SwiGLU (gemm_q8_kernel<true>)"
    if mx:
        roof["kernel"] = "grouped MX Linear1 + SwiGLU + Q_MX (gemm_mx_kernel<true, %d>)" % moe.MX_FORMATS[mx]
    launches_per_step = route_launches(c) + (8 if quant else (7 if mx else 6 + forward_row_copy(c)))
    out = {
        "metric": METRIC, "value": round(T * world / (ms / 1e3), 1), "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8" if quant else (f"{mx} x {synth_mx_weight_format(c)}" if mx else "bf16"),
        "data": "synthetic (seeded; random-init weights of the workload's shapes)",
        "config": {"workload": f"{workload}: {WORKLOAD_TEXT.get(workload, '')}",
                   "T": T, "H": H, "E": E, "k": k, "I": I, "shared_experts": has_shared,
                   "routing": c["routing"], "score": c["score"],
                   "l2": "inputs larger than L2: %.1f GB of expert weights per step"
                         % ((E + has_shared) * 3 * H * I * (1 if quant else (
                             (accounting.MX4 if synth_mx_weight_format(c) == "e2m1" else accounting.MX8)
                             if mx else 2)) / 1e9),
                   "weights": ("int8 + per-channel fp32 scales (A8W8-INT)" if quant else
                               (f"{synth_mx_weight_format(c)} codes + E8M0 scales per 32 (MX), "
                                f"{mx} activations" if mx else "bf16")),
                   "parallelism": f"replicas x{world} (token batches, no collective)"},
        "stages_ms": {k_: round(v, 4) for k_, v in stages.items()},
        "grouped_gemm": {"tflops": round(gemm_tflops, 1),
                         "pct_bf16_peak": round(100 * gemm_tflops / pk["bf16_tflops_sustained"], 2),
                         "pct_own_dtype_peak": round(100 * gemm_tflops / tc_peak, 2),
                         "peak_tflops": pk["bf16_tflops_sustained"],
                         "gemm1_GBps": round(g1_bytes / g1_s / 1e9, 1),
                         "gemm2_GBps": round(g2_bytes / g2_s / 1e9, 1)},
        "roofline": roof,
        "e2e": {"value": round(T * world / (e2e_ms / 1e3), 1), "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": launches_per_step * K,
        "clocks": sampler.summary() if sampler else None,
        "load": {"max_expert_rows": int(counts.max()), "min_expert_rows": int(counts.min()),
                 "active_experts": int((counts > 0).sum())},
    }
    if graph_ms is not None:
        out["graph_replay"] = {"ms_per_step": round(graph_ms, 4),
                               "value": round(T * world / (graph_ms / 1e3), 1), "unit": UNIT}
    if world == 1 and with_cpu and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(dd, args.cpu_tokens, args.cpu_tokens_1core)
    return out


def run_train(args, rank, world, local_rank):
    """One training step of the layer: route, moe_forward_train, moe_backward
    (all gradients) on one batch; the upstream gradient is a seeded bf16
    N(0, 1) tensor.  Reports tokens/s of the whole step."""
    import torch
    import mixture_experts_ffn_route_gb300 as moe
    from mixture_experts_ffn_route_gb300 import accounting
    import synth

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    moe.lib()
    wseed, tseed = rank_seeds(rank)
    dd = synth.make_inputs_torch(args.workload, seed=wseed, token_seed=tseed, device=dev)
    c = dd["cfg"]
    if c["routing"] == "given" or c.get("quant"):
        raise SystemExit("--train needs a routed bf16 workload")
    T, H, E, k, I = c["T"], c["H"], c["E"], c["k"], c["I"]
    sh = c["shared"]
    p = moe.params_from_config(c)
    ws = moe.alloc_workspace_train(p, dev)
    dY = torch.from_numpy(synth.upstream_grad(T, H, seed=tseed).view(np.int16)).to(dev).view(torch.bfloat16)
    E_ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    G = torch.empty((T, k), dtype=torch.float32, device=dev)
    Y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    f32 = lambda *s_: torch.empty(s_, dtype=torch.float32, device=dev)  # noqa: E731
    grads = {"dX": torch.empty((T, H), dtype=torch.bfloat16, device=dev), "dWg": f32(H, E),
             "dW1": f32(E, H, 2 * I), "dW2": f32(E, I, H), "dG": f32(T, k),
             "dWs1": f32(H, 2 * I) if sh else None, "dWs2": f32(I, H) if sh else None}
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(K)]
    for e in ev:
        for x in e:
            x.record()

    def step(X=None, dYs=None, evs=None):
        X = dd["X"] if X is None else X
        dYs = dY if dYs is None else dYs
        if evs:
            evs[0].record()
        if c["routing"] == "hash":
            moe.moe_route(p, X, dd["Wg"], None, dd["token_ids"], dd["tid2eid"], c["V"], E_ids, G, ws)
        else:
            moe.moe_route(p, X, dd["Wg"], dd["bias"], None, None, 0, E_ids, G, ws)
        if evs:
            evs[1].record()
        moe.moe_forward_train(p, X, E_ids, G, dd["W1"], dd["W2"], dd["Ws1"], dd["Ws2"], Y, ws)
        moe.moe_backward(p, X, dd["Wg"], E_ids, G, dd["W1"], dd["W2"], dd["Ws1"], dd["Ws2"], dYs,
                         grads["dX"], grads["dWg"], grads["dW1"], grads["dW2"], grads["dWs1"],
                         grads["dWs2"], grads["dG"], ws, stage_events=evs[2:] if evs else None)

    sampler = ClockSampler(local_rank) if rank == 0 else None
    for _ in range(args.warmup):
        step()
    moe.moe_sync_status(ws)
    counts = torch.bincount(E_ids.reshape(-1).long(), minlength=E).cpu().numpy()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_start()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(K):
        step(evs=ev[i])
    t1.record()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_end()
    moe.moe_sync_status(ws)
    ms = max_over_ranks(t0.elapsed_time(t1) / K, world, dev)

    def avg(a, b):
        return sum(e[a].elapsed_time(e[b]) for e in ev) / K
    stages = {"route": avg(0, 1), "forward": avg(1, 2), "unpermute_bwd": avg(2, 3),
              "dgrad": avg(3, 4), "wgrad": avg(4, 5), "router_bwd_dx": avg(5, 6)}

    # end to end: X and dY from pinned host memory, Y and dX back, every step
    Xh = dd["X"].cpu().pin_memory()
    dYh = dY.cpu().pin_memory()
    Yh = torch.empty_like(Xh).pin_memory()
    dXh = torch.empty_like(Xh).pin_memory()
    Xd, dYd = torch.empty_like(dd["X"]), torch.empty_like(dY)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(K):
        Xd.copy_(Xh, non_blocking=True)
        dYd.copy_(dYh, non_blocking=True)
        step(Xd, dYd)
        Yh.copy_(Y, non_blocking=True)
        dXh.copy_(grads["dX"], non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / K, world, dev)
    if rank != 0:
        return None
    pk = peaks()
    # dominant kernel: the weight gradients, bound by writing fp32 dW1 and dW2
    rows, n_act = accounting._counts(counts, sh, T)
    wg_bytes = (n_act * 3 * H * I * 4                 # dW1, dW2 (and the shared) fp32 written
                + 2 * rows * (I + H) * 2 + 2 * rows * (H + 2 * I) * 2)  # bf16 operands read
    achieved = wg_bytes / (stages["wgrad"] / 1e3) / 1e9
    out = {
        "metric": "MoE-layer training-step tokens/s (route + forward + backward) @1 GB300",
        "value": round(T * world / (ms / 1e3), 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; random-init weights of the workload's shapes, N(0,1) upstream gradient)",
        "config": {"workload": f"{args.workload}: {WORKLOAD_TEXT.get(args.workload, '')}, training step",
                   "T": T, "H": H, "E": E, "k": k, "I": I, "shared_experts": sh,
                   "gradients": "dX bf16; dWg, dW1, dW2, dWs fp32",
                   "l2": "inputs larger than L2",
                   "parallelism": f"replicas x{world} (token batches, no collective)"},
        "stages_ms": {k_: round(v, 4) for k_, v in stages.items()},
        "roofline": {"kernel": "weight gradients (gemm_bwd_kernel<1,1,0,1>, split K)", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": None,
                     "algorithmic_bytes_per_launch": int(wg_bytes / 2),
                     "peak_source": pk["source"] + " hbm_gbs"},
        "e2e": {"value": round(T * world / (e2e_ms / 1e3), 1), "unit": UNIT,
                "h2d_bytes_per_step": int(2 * T * H * 2), "d2h_bytes_per_step": int(2 * T * H * 2)},
        # route + forward 6 + backward: unpermute, gather, 2 dgrad, 2 wgrad,
        # router GEMM, router backward, dWg, dXr, dX sum = 11
        "gpu_launches": (route_launches(c) + 6 + forward_row_copy(c) + 11) * K,
        "clocks": sampler.summary() if sampler else None,
    }
    return out


def load_traffic(workload, algorithmic_bytes):
    """DRAM bytes of one Linear1 launch, from the committed ncu summary of a
    capture at a profiling size of the same expert shapes (c3p for the V4-Pro
    layers, c5p for the large-FFN layer): that launch's DRAM bytes over its
    algorithmic bytes, times this launch's algorithmic bytes.  The profiling
    sizes hold 4.3 GB of weights, so their DRAM figures are not L2 hits; the
    full-size launches are not captured (they hold 35-69 GB)."""
    import re
    key = {"c3": "c3p", "c4": "c3p", "c3_sp": "c3p", "c3_f3072": "c3p", "c3p": "c3p",
           "c5": "c5p", "c5p": "c5p"}.get(workload)
    path = os.path.join(ROOT, "profiles", "traffic_gemm_bf16_c3p_c5p.md")
    if key is None or not os.path.exists(path):
        return None
    with open(path) as f:
        m = re.search(r"traffic_ratio_%s_gemm1:\s*([0-9.]+)" % key, f.read())
    return int(float(m.group(1)) * algorithmic_bytes) if m else None


# ------------------------------------------------------------------ oracle (CPU)
class OracleRunner:
    """The CPU oracle, as it stands, on the bench's workload.  Inputs come from
    the same seeded device drawing, copied to the host; expert weights are
    fetched to the host (bf16 bits) one expert at a time when the oracle asks
    for them, and the oracle decodes them itself."""

    def __init__(self, dd):
        import torch
        self.torch = torch
        self.dd = dd
        c = dd["cfg"]
        self.c = c
        bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)  # noqa: E731
        self.bits = bits
        self.X = bits(dd["X"])
        self.Wg = bits(dd["Wg"])
        self.bias = dd["bias"].cpu().numpy() if dd["bias"] is not None else None
        self.Ws1 = bits(dd["Ws1"]) if dd["Ws1"] is not None else None
        self.Ws2 = bits(dd["Ws2"]) if dd["Ws2"] is not None else None
        if c["routing"] == "given":
            self.E_ids = dd["E_ids"].cpu().numpy()
            self.G = dd["G"].cpu().numpy().astype(np.float64)
        if c["routing"] == "hash":
            self.tok = dd["token_ids"].cpu().numpy()
            self.tab = dd["tid2eid"].cpu().numpy()

    def route(self, rows=None):
        """The oracle's routing and dispatch of the given tokens (all by
        default): returns (ids, G) of those tokens."""
        import oracle
        c = self.c
        rows = np.arange(c["T"]) if rows is None else rows
        X = self.X[rows]
        if c["routing"] == "given":
            ids, G = self.E_ids[rows], self.G[rows]
        elif c["routing"] == "hash":
            ids, G, _ = oracle.route_hash(X, self.Wg, self.tok[rows], self.tab, c["score_fn"],
                                          c["alpha"], c["renorm"])
        else:
            ids, G, _ = oracle.route(X, self.Wg, self.bias, c["score_fn"], c["k"], c["alpha"], c["renorm"])
        oracle.dispatch(ids, c["E"])
        return ids, G

    def ffn(self, rows, ids, G):
        """The oracle's expert FFNs and combine of the given tokens (their ids
        and gates given), rounded to bf16."""
        import oracle
        c = self.c
        X = self.X[rows]
        dd = self.dd
        raw = lambda key: (lambda e: dd[key][e].cpu().numpy())  # noqa: E731
        if c.get("quant") == "a8w8":
            Y = oracle.forward_a8w8_tokens(rows, X, ids, G, raw("W1"), raw("S1"), raw("W2"), raw("S2"),
                                           E=c["E"])
        elif synth_mx_format(c):
            Y = oracle.forward_mx_tokens(rows, X, ids, G, raw("W1"), raw("S1"), raw("W2"), raw("S2"),
                                         E=c["E"], fmt=synth_mx_format(c))
        else:
            W1 = lambda e: self.bits(dd["W1"][e])  # noqa: E731
            W2 = lambda e: self.bits(dd["W2"][e])  # noqa: E731
            Y = oracle.forward_tokens(rows, X, ids, G, W1, W2, self.Ws1, self.Ws2, E=c["E"])
        return oracle.f64_to_bf16_bits(Y)


def _blas_threads(n=None):
    """Read (and, with n, set) the thread count of the BLAS library numpy
    loaded: threadpoolctl where installed, else the library's own
    set/get calls found through /proc/self/maps."""
    try:
        import threadpoolctl
        info = [i for i in threadpoolctl.threadpool_info() if i.get("user_api") == "blas"]
        if info:
            old = int(max(i["num_threads"] for i in info))
            if n is not None:
                threadpoolctl.threadpool_limits(n, user_api="blas")
            return old
    except Exception:
        pass
    import ctypes
    import re
    libs = set()
    try:
        with open("/proc/self/maps") as f:
            for line in f:
                m = re.search(r"(/\S*openblas\S*\.so\S*)", line)
                if m:
                    libs.add(m.group(1))
    except OSError:
        return None
    old = None
    for path in sorted(libs):
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for suffix in ("", "64_", "_64_"):
            for pre in ("openblas", "scipy_openblas"):
                get = getattr(lib, f"{pre}_get_num_threads{suffix}", None)
                put = getattr(lib, f"{pre}_set_num_threads{suffix}", None)
                if get is None or put is None:
                    continue
                old = int(get())
                if n is not None:
                    put(ctypes.c_int(n))
                return old
    return old


def oracle_leg(r, n_tokens, seed=0):
    """One timing of the oracle on the workload: routing and dispatch of all T
    tokens, then the expert FFNs and combine of a seeded set of n_tokens tokens
    that reaches every routed expert (each expert's weights fetched and decoded
    once), scaled to T tokens (rows are independent).  Returns (tokens/s of the
    whole layer, route seconds, FFN seconds, tokens in the FFN sample)."""
    import synth
    c = r.c
    T = c["T"]
    t0 = time.time()
    ids, G = r.route()
    t_route = time.time() - t0
    rows = synth.covering_tokens(ids, c["E"], n_tokens, 0, seed=seed)
    t0 = time.time()
    r.ffn(rows, ids[rows], G[rows])
    t_ffn = time.time() - t0
    return T / (t_route + t_ffn * T / len(rows)), t_route, t_ffn, len(rows)


def oracle_expert_leg(r, step, n_cap=256):
    """One bounded step of the reference arm: the oracle's routing and dispatch
    of all T tokens, then its expert FFN (swiglu_expert, which decodes the
    expert's bf16 weights itself) for one active expert, on up to n_cap of the
    rows routed to it and on one of them alone.  The experts are taken in
    order of their row counts, largest first, one per step.  The layer's FFN
    time is modelled from the two calls: each active expert decoded once (the
    one-row call) plus a cost per routed row (the difference over the other
    rows), the shared expert counted as one more expert of T rows.  Returns
    (tokens/s of the layer, route s, decode s, per-row s, rows used)."""
    import oracle
    c = r.c
    T = c["T"]
    t0 = time.time()
    ids, _ = r.route()
    t_route = time.time() - t0
    counts = np.bincount(ids[(ids >= 0) & (ids < c["E"])].ravel(), minlength=c["E"])
    order = np.argsort(-counts, kind="stable")
    active = order[counts[order] > 1]
    e = int(active[step % len(active)])
    rows = np.nonzero((ids == e).any(axis=1))[0]
    rows = np.random.default_rng(step).permutation(rows)[:n_cap]
    W1 = r.bits(r.dd["W1"][e])
    W2 = r.bits(r.dd["W2"][e])
    X64 = oracle.bf16_to_f64(r.X[rows])
    t0 = time.time()
    oracle.swiglu_expert(X64[:1], W1, W2)
    t_one = time.time() - t0
    t0 = time.time()
    oracle.swiglu_expert(X64, W1, W2)
    t_all = time.time() - t0
    per_row = max(t_all - t_one, 0.0) / max(len(rows) - 1, 1)
    n_active = int((counts > 0).sum()) + (1 if c["shared"] else 0)
    n_rows = int(counts.sum()) + (T if c["shared"] else 0)
    t_layer = t_route + n_active * t_one + n_rows * per_row
    return T / t_layer, t_route, t_one, per_row, len(rows)


def cpu_baseline(dd, n_all=512, n_one=128):
    """The oracle on this host's cores (all, then one) at the bench's workload."""
    r = OracleRunner(dd)
    r.route(np.arange(2))  # first-call costs (BLAS start-up) outside the timing
    cores = os.cpu_count()
    v_all, tr_all, tf_all, n_a = oracle_leg(r, n_all)
    old = _blas_threads(1)
    try:
        v_one, tr_one, tf_one, n_o = oracle_leg(r, n_one, seed=1)
    finally:
        if old:
            _blas_threads(old)
    T = r.c["T"]
    return {"value": round(v_all, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "cores_all": cores, "value_all": round(v_all, 4), "value_1core": round(v_one, 4),
            "blas_threads_all": old, "extrapolated": True,
            "sample": (f"routing and dispatch of all {T} tokens ({tr_all:.1f} s on all cores, "
                       f"{tr_one:.1f} s on one), then the fp64 expert FFNs and combine of {n_a} "
                       f"tokens chosen to reach every routed expert ({tf_all:.1f} s, all cores; "
                       f"{n_o} tokens, {tf_one:.1f} s, one core), each expert's weights decoded "
                       f"once per call, extrapolated x T/{n_a} (x T/{n_o}): token rows are "
                       f"independent")}


def run_reference(args, rank, world):
    """The oracle as it stands on this host's cores (rank 0 only), in steps
    bounded so that --steps K --warmup W end within a few minutes: each step
    routes all T tokens and runs one expert's FFN (oracle_expert_leg).  The
    in-line cpu_baseline of the GPU arm runs the full covering sample."""
    if rank != 0:
        return None
    import torch
    import synth
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    dd = synth.make_inputs_torch(args.workload, seed=1234, device=dev)
    r = OracleRunner(dd)
    r.route(np.arange(2))  # first-call costs (BLAS start-up) outside the timing
    quantised = bool(r.c.get("quant") or synth_mx_format(r.c))
    # the quantised forms keep the covering leg on a small token sample
    leg = ((lambda i: oracle_leg(r, args.ref_tokens, seed=i)) if quantised
           else (lambda i: oracle_expert_leg(r, i)))
    for i in range(args.warmup):
        leg(1000 + i)
    vals, secs, parts = [], [], []
    for i in range(args.steps):
        t0 = time.time()
        out = leg(i)
        secs.append(time.time() - t0)
        vals.append(out[0])
        parts.append(out[1:])
    v = len(vals) / sum(1.0 / x for x in vals)  # tokens/s over the K steps (harmonic mean)
    med = lambda j: float(np.median([p[j] for p in parts]))  # noqa: E731
    if quantised:
        sample = (f"each step: routing and dispatch of all {dd['cfg']['T']} tokens, then the fp64 "
                  f"expert FFNs and combine of {args.ref_tokens} tokens and as many more as reach "
                  f"every routed expert (each expert's weights decoded once per step), "
                  f"extrapolated x T/(tokens used)")
    else:
        sample = (f"each step: the oracle's routing and dispatch of all {dd['cfg']['T']} tokens "
                  f"({med(0):.2f} s), then its expert FFN for one expert (the most loaded first, "
                  f"one per step) on up to 256 of its rows and on one row alone; the layer's FFN "
                  f"time is modelled as (active experts x the one-row call, {med(1):.2f} s: the "
                  f"expert's weights decoded) + (routed rows x the per-row cost, "
                  f"{1e3 * med(2):.2f} ms)")
    return {"metric": METRIC, "value": round(v, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * sum(secs) / len(secs), 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "impl": "reference",
            "config": {"workload": f"{args.workload}: {WORKLOAD_TEXT.get(args.workload, '')}"},
            "cpu_baseline": {"value": round(v, 4), "unit": UNIT, "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample, "extrapolated": True},
            "e2e": {"value": round(v, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c5")
    ap.add_argument("--also", default="c3",
                    help="comma-separated workloads measured after the main one (1 GPU), "
                         "reported under other_workloads; empty for none")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=512,
                    help="tokens of the oracle's FFN sample on all cores")
    ap.add_argument("--cpu-tokens-1core", type=int, default=128,
                    help="tokens of the oracle's FFN sample on one core")
    ap.add_argument("--ref-tokens", type=int, default=8,
                    help="tokens of the reference arm's FFN sample per step (quantised forms)")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step captured once in a CUDA graph and replayed")
    ap.add_argument("--train", action="store_true",
                    help="time a training step (route + forward + backward) instead of the forward")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    elif args.train:
        out = run_train(args, rank, world, local_rank)
    else:
        out = run_ours(args, rank, world, local_rank)
        extra = [w for w in args.also.split(",") if w and w != args.workload] if world == 1 else []
        if extra:
            import gc
            import torch
            gc.collect()
            torch.cuda.empty_cache()
            other = {}
            for w in extra:
                o = run_ours(args, rank, world, local_rank, workload=w, with_cpu=False)
                gc.collect()
                torch.cuda.empty_cache()
                other[w] = {key: o[key] for key in ("value", "unit", "ms_per_step", "config", "stages_ms",
                                                     "grouped_gemm", "roofline", "e2e", "gpu_launches",
                                                     "clocks", "load") if key in o}
            out["other_workloads"] = other
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1 and args.impl == "ours":
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
