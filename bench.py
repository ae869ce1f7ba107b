#!/usr/bin/env python
"""Benchmark of one block-diffusion denoising step on GB300.

A step is one full pass of the hot path over one 32-token block per request:
for each of the 40 MoE layers x = RMSNorm(h), router top-8 of 256, block
coreset (top_p 0.9), routed + shared SwiGLU experts, h += out; then RMSNorm,
LM head (V = 152064) and the LowConfidence commit (threshold 0.95).  That is
one call of block_decode_step.  Inputs (64.4 GB of bf16 expert weights, the
LM head, the block's residual stream) are resident in HBM before the timed
region; every step streams the selected experts' weights from HBM (the
weights are far larger than L2).

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "block-steps/s (40-layer MoE, B=32) & expert-weight HBM GB/s vs peak; tokens/step"
UNIT = "block-steps/s"
THRESHOLD = 0.95
TOP_P = 0.9


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--config", choices=["clover_stack40", "clover_layer", "clover_stack40_fp8", "clover_layer_fp8"],
                    default="clover_stack40")
    ap.add_argument("--requests", type=int, default=1, help="concurrent requests (blocks) per GPU")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (profiling runs)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-loop", action="store_true", help="skip the whole-block round-loop measurement")
    ap.add_argument("--no-sweep", action="store_true", help="skip the batched-requests sweep (R = 1, 4, 16)")
    ap.add_argument("--sweep", type=str, default="1,4,16", help="requests per step of the batched sweep")
    ap.add_argument("--correlation", type=float, default=0.0,
                    help="workload variant: tokens of a block share a hidden component (0 = independent)")
    ap.add_argument("--block", type=int, default=None, help="workload variant: block size P (default 32)")
    ap.add_argument("--threshold", type=float, default=THRESHOLD, help="LowConfidence threshold")
    ap.add_argument("--loop-scale", type=float, default=16.0,
                    help="logit scale of the round-loop measurement (1 = every round is a fallback)")
    ap.add_argument("--prof-all", action="store_true", help="time every kernel in the roofline pass")
    ap.add_argument("--no-graph", action="store_true", help="time direct launches instead of CUDA-graph replays")
    ap.add_argument("--layer-head", type=int, choices=(0, 2), default=None,
                    help="between expert launches: 0 separate combine/router/coreset/gather launches, "
                         "2 combine inside the router launch (library default)")
    return ap.parse_args()


# ------------------------------------------------------------------------------------------ distributed
class Dist:
    def __init__(self, backend: str):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------------------------------ clocks
class Clocks:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", gpu_id], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        self.t0 = self.t1 = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def result(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(f[2]), float(f[3]), f[5], f[6], f[7], f[8], f[9]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t0 is not None and self.t0 - 1 <= r[0] <= self.t1 + 1]
        use = inside or rows
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in use:
            for name, v in zip(names, r[4:]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in use) if use else None,
                "sm_max_mhz": max(r[2] for r in use) if use else None,
                "reasons": sorted(reasons), "samples": len(use),
                "window": "timed region" if inside else "whole run"}


# ------------------------------------------------------------------------------------------ workload
def workload(name: str):
    from synth import workloads as W
    return W.CONFIGS[name]


def workload_desc(cfg, R: int, args=None) -> dict:
    thr = args.threshold if args is not None else THRESHOLD
    corr = args.correlation if args is not None else 0.0
    return {"workload": f"{cfg.name}: {cfg.n_layers}-layer MoE FFN stack (H={cfg.H}, {cfg.E} routed experts top-{cfg.k}, "
                        f"expert/shared SwiGLU I={cfg.I}, 1 shared expert, "
                        f"{'FP8 E4M3 expert weights with per-row fp32 scales, bf16 router and LM head' if cfg.dtype == 'fp8' else 'bf16 weights'}"
                        f", fp32 accumulate), "
                        f"block of {cfg.P} tokens x {R} request(s), coreset top_p {TOP_P}, RMSNorm eps 1e-6 "
                        f"between layers, LM head V={cfg.V}, LowConfidence commit threshold {thr}"
                        + (f", block tokens correlated (a={corr})" if corr > 0 else ""),
            "layers": cfg.n_layers, "block_tokens": cfg.P, "requests": R, "top_p": TOP_P,
            "threshold": thr, "vocab": cfg.V, "token_correlation": corr,
            "l2": "inputs larger than L2: every step streams the selected experts' weights (tens of GB) from HBM",
            "parallelism": "replicas (one independent block step per GPU)",
            "launch": "one block_decode_step call per step, replayed as a CUDA graph (programmatic dependent launch "
                      "between kernels)"}


def expert_bytes(cfg, unions) -> dict:
    """Algorithmic HBM bytes of one step: each selected expert's weights once, shared experts,
    routers and the LM head."""
    if cfg.dtype == "fp8":   # one byte per weight plus one fp32 scale per weight row
        per_expert = 3 * cfg.I * cfg.H + (2 * cfg.I + cfg.H) * 4
        shared = 3 * cfg.Is * cfg.H + (2 * cfg.Is + cfg.H) * 4
    else:
        per_expert = 3 * cfg.I * cfg.H * 2
        shared = 3 * cfg.Is * cfg.H * 2
    experts = sum(unions) * per_expert + cfg.n_layers * shared
    return {"expert_weights": experts, "router": cfg.n_layers * cfg.E * cfg.H * 2, "lm_head": cfg.V * cfg.H * 2,
            "per_expert": per_expert, "shared_per_layer": shared}


# ------------------------------------------------------------------------------------------ GPU arm
def run_gpu(args, dist: Dist):
    import numpy as np
    import torch

    import moe_expert_step_gb300 as ms
    from synth import workloads as W

    torch.cuda.set_device(dist.local)
    cfg = workload(args.config)
    if args.block:
        from dataclasses import replace
        cfg = replace(cfg, P=args.block)
    R = args.requests
    THR = args.threshold
    T = R * cfg.P
    d = ms.ModelDims(H=cfg.H, E=cfg.E, k=cfg.k, I=cfg.I, Is=cfg.Is, V=cfg.V, P=cfg.P,
                     dtype=ms.FP8 if cfg.dtype == "fp8" else ms.BF16)
    t_setup = time.time()
    layers_t = [W.device_layer(cfg, l) for l in range(cfg.n_layers)]
    layers = [ms.layer(l["Wr"], l["Wgu"], l["Wd"], l["Wsgu"], l["Wsd"], l.get("Sgu"), l.get("Sd"), l.get("Ssgu"),
                       l.get("Ssd")) for l in layers_t]
    Wlm = W.device_lm_head(cfg)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    h0_host = W.host_h0(cfg, R, correlation=args.correlation)
    masked_host = W.masked_subset(cfg, R).astype(np.uint8)
    h0 = dev(h0_host)
    tokens0 = torch.zeros(T, dtype=torch.int32, device="cuda")
    masked0 = dev(masked_host)
    top_p = torch.full((R,), TOP_P, dtype=torch.float32, device="cuda")
    tokens, masked = tokens0.clone(), masked0.clone()
    choice = torch.zeros(T, dtype=torch.int32, device="cuda")
    conf = torch.zeros(T, dtype=torch.float32, device="cuda")
    accept = torch.zeros(T, dtype=torch.uint8, device="cuda")
    n_comm = torch.zeros(R, dtype=torch.int32, device="cuda")
    ws = ms.workspace(d, R)
    if args.layer_head is not None:
        ms.set_route_fusion(args.layer_head)
    torch.cuda.synchronize()
    t_setup = time.time() - t_setup

    def step(h_in=h0, trace=None):
        tokens.copy_(tokens0)
        masked.copy_(masked0)
        kw = trace or {}
        ms.block_decode_step(d, R, layers, Wlm, top_p, THR, h_in, tokens, masked, choice, conf, accept, n_comm,
                             ws, **kw)

    # one traced step: per-layer coreset sizes and the union of kept experts
    n_sel = torch.zeros((cfg.n_layers, R), dtype=torch.int32, device="cuda")
    sel = torch.zeros((cfg.n_layers, R, cfg.E), dtype=torch.int32, device="cuda")
    step(trace=dict(trace_n_sel=n_sel, trace_sel=sel))
    torch.cuda.synchronize()
    if ms.read_device_error(ws) != ms.OK:
        raise RuntimeError("device error word set after the traced step")
    n_sel_h, sel_h = n_sel.cpu().numpy(), sel.cpu().numpy()
    unions = [len(set().union(*[set(sel_h[l, r, :n_sel_h[l, r]].tolist()) for r in range(R)]))
              for l in range(cfg.n_layers)]
    committed_per_step = int(n_comm.sum().item())

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    ref_out = (tokens.clone(), masked.clone(), conf.clone())

    # the step is capturable: every launch is asynchronous on the caller's stream
    run = step
    per_replay = None
    if not args.no_graph:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        c0 = ms.launch_count()
        with torch.cuda.graph(graph):
            step()
        per_replay = ms.launch_count() - c0      # library kernels captured into the graph
        run = graph.replay
        for _ in range(max(3, args.warmup)):
            run()
        torch.cuda.synchronize()
        for a, b in zip((tokens, masked, conf), ref_out):
            if not torch.equal(a, b):
                raise RuntimeError("graph replay differs from a direct call")

    stream = torch.cuda.current_stream()
    clocks = Clocks("GPU-" + str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid))
    time.sleep(0.3)
    # ---------------- timed region (device clock)
    dist.barrier()
    torch.cuda.synchronize()
    launches0 = ms.launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark_start()
    e0.record(stream)
    for _ in range(args.steps):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    dist.barrier()
    launches = ms.launch_count() - launches0 if per_replay is None else per_replay * args.steps
    ms_total = dist.max(e0.elapsed_time(e1))
    clk = clocks.result()

    # ---------------- roofline pass: events around the expert and LM-head kernels on their stream
    ms.prof_enable(None if args.prof_all else ["expert_ffn", "lm_head"])
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    prof = ms.prof_read()
    ms.prof_enable([])

    # ---------------- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        h_pin = torch.from_numpy(h0_host).pin_memory()
        m_pin = torch.from_numpy(masked_host).pin_memory()
        t_pin = torch.zeros(T, dtype=torch.int32).pin_memory()
        tp_pin = torch.full((R,), TOP_P, dtype=torch.float32).pin_memory()
        out_tok = torch.zeros(T, dtype=torch.int32).pin_memory()
        out_msk = torch.zeros(T, dtype=torch.uint8).pin_memory()
        out_n = torch.zeros(R, dtype=torch.int32).pin_memory()
        h_dev = torch.empty_like(h0)

        def e2e_step():
            h_dev.copy_(h_pin, non_blocking=True)
            tokens.copy_(t_pin, non_blocking=True)
            masked.copy_(m_pin, non_blocking=True)
            top_p.copy_(tp_pin, non_blocking=True)
            ms.block_decode_step(d, R, layers, Wlm, top_p, THR, h_dev, tokens, masked, choice, conf, accept,
                                 n_comm, ws)
            out_tok.copy_(tokens, non_blocking=True)
            out_msk.copy_(masked, non_blocking=True)
            out_n.copy_(n_comm, non_blocking=True)
            stream.synchronize()

        for _ in range(3):
            e2e_step()
        dist.barrier()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        t_e2e = dist.max(time.perf_counter() - t0)
        dist.barrier()
        h2d = h_pin.numel() * 4 + m_pin.numel() + t_pin.numel() * 4 + tp_pin.numel() * 4
        d2h = out_tok.numel() * 4 + out_msk.numel() + out_n.numel() * 4
        e2e = {"value": dist.world * args.steps * R / t_e2e, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h,
               "how": "wall clock over K public-API calls (Python binding -> C ABI), each with pinned H2D inputs, "
                      "the step, D2H of tokens/masked/n_committed and a stream synchronize"}
    # ---------------- the whole block: device-resident round loop vs rounds driven from the host
    round_loop = None
    if not args.no_loop:
        round_loop = measure_round_loop(ms, W, cfg, d, R, layers, Wlm, top_p, ws, args.loop_scale, dist, THR)
    if ms.read_device_error(ws) != ms.OK:
        raise RuntimeError("device error word set during the benchmark")
    sweep = None
    if not args.no_sweep and R == 1:
        sweep = measure_sweep(ms, W, cfg, d, layers, Wlm, [int(v) for v in args.sweep.split(",")], args, dist, THR)

    ms_step = ms_total / args.steps
    value = dist.world * args.steps * R / (ms_total / 1e3)   # one step advances R blocks
    eb = expert_bytes(cfg, unions)
    step_bytes = eb["expert_weights"] + eb["router"] + eb["lm_head"]
    peaks = load_peaks()
    hbm_peak = peaks.get("hbm_gbs")
    # dominant kernel: the fused expert FFN launch (gate/up + SwiGLU + down, all expert weight bytes)
    ff_n, ff_ms = prof["expert_ffn"]
    steps_prof = args.steps
    # per launch: every kept expert's and the shared expert's weights once, plus the gathered
    # activations read, the SwiGLU rows written and read back, and the per-slot outputs written
    # (at most T*(k+1) token slots)
    slots = T * (cfg.k + 1)
    ff_act = slots * (cfg.H * 2 + 2 * max(cfg.I, cfg.Is) * 2 + cfg.H * 4)
    ff_bytes_launch = eb["expert_weights"] / cfg.n_layers + ff_act
    ff_avg_ms = ff_ms / max(1, ff_n)
    achieved = ff_bytes_launch / (ff_avg_ms / 1e3) / 1e9
    roofline = {"kernel": "tc_gemm_kernel<experts> (routed + shared expert gate/up, SwiGLU and down in one launch)",
                "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4) if hbm_peak else None,
                "traffic": load_traffic(statistics.mean(unions) + 1, cfg.dtype),
                "peak_source": peaks.get("source"),
                "bytes_per_launch": int(ff_bytes_launch), "avg_launch_ms": round(ff_avg_ms, 5),
                "launches_timed": ff_n}
    expert_stream_ms = ff_ms / steps_prof
    step_gbs = step_bytes / (ms_step / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 experts, bf16 rest" if cfg.dtype == "fp8" else "bf16",
        "data": "synthetic",
        "config": workload_desc(cfg, R, args),
        "layer_head": layer_head_desc(cfg, R),
        "expert_weight_hbm": {
            "bytes_per_step": step_bytes, "expert_bytes_per_step": eb["expert_weights"],
            "experts_kept_per_layer": {"mean": round(statistics.mean(unions), 2), "min": min(unions),
                                       "max": max(unions)},
            "gbs_whole_step": round(step_gbs, 1),
            "frac_of_peak_whole_step": round(step_gbs / hbm_peak, 4) if hbm_peak else None,
            "gbs_expert_kernels": round(eb["expert_weights"] / (expert_stream_ms / 1e3) / 1e9, 1),
            "frac_of_peak_expert_kernels": round(eb["expert_weights"] / (expert_stream_ms / 1e3) / 1e9 / hbm_peak, 4)
            if hbm_peak else None,
            "peak_gbs": hbm_peak},
        "tokens_per_step": {"measured_synthetic": committed_per_step / R,
                            "committed_tokens_per_s": {"tau=1": round(value, 2), "tau=10": round(10 * value, 2),
                                                       "measured": round(value * committed_per_step / R, 2)},
                            "note": "tau = tokens committed per step; synthetic hidden states have low "
                                    "confidence, so the measured tau is the fallback's 1"},
        "roofline": roofline,
        "kernel_ms_per_step": {k: round(v[1] / steps_prof, 4) for k, v in prof.items() if v[0]},
        "clocks": clk, "gpu_launches": launches, "e2e": e2e,
        "round_loop": round_loop,
        "sweep": sweep,
        "graph": not args.no_graph,
        "setup_s": round(t_setup, 1),
    }
    return line, cfg


def measure_sweep(ms, W, cfg, d, layers, Wlm, Rs, args, dist, thr) -> dict:
    """The same 40-layer step for R concurrent requests (R blocks of P tokens, one coreset per
    request, experts grouped over the union of the requests' kept experts), each timed like the
    headline: K CUDA-graph replays between CUDA events, then a pass with events around every
    expert launch for that kernel's fraction of the HBM peak."""
    import numpy as np
    import torch

    peak = load_peaks().get("hbm_gbs")
    stream = torch.cuda.current_stream()
    out = {"what": "block_decode_step over R requests x 32-token blocks, 40 layers, per-request coreset top_p "
                   f"{TOP_P}; K = {args.steps} graph replays per R, inputs resident in HBM",
           "points": []}
    for R in Rs:
        T = R * cfg.P
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        h0 = dev(W.host_h0(cfg, R))
        tokens0 = torch.zeros(T, dtype=torch.int32, device="cuda")
        masked0 = dev(W.masked_subset(cfg, R).astype(np.uint8))
        top_p = torch.full((R,), TOP_P, dtype=torch.float32, device="cuda")
        tokens, masked = tokens0.clone(), masked0.clone()
        choice = torch.zeros(T, dtype=torch.int32, device="cuda")
        conf = torch.zeros(T, dtype=torch.float32, device="cuda")
        accept = torch.zeros(T, dtype=torch.uint8, device="cuda")
        ncomm = torch.zeros(R, dtype=torch.int32, device="cuda")
        ws = ms.workspace(d, R)

        def step(**kw):
            tokens.copy_(tokens0)
            masked.copy_(masked0)
            ms.block_decode_step(d, R, layers, Wlm, top_p, thr, h0, tokens, masked, choice, conf, accept, ncomm, ws,
                                 **kw)

        n_sel = torch.zeros((cfg.n_layers, R), dtype=torch.int32, device="cuda")
        sel = torch.zeros((cfg.n_layers, R, cfg.E), dtype=torch.int32, device="cuda")
        step(trace_n_sel=n_sel, trace_sel=sel)
        torch.cuda.synchronize()
        ns, sl = n_sel.cpu().numpy(), sel.cpu().numpy()
        unions = [len(set().union(*[set(sl[l, r, :ns[l, r]].tolist()) for r in range(R)]))
                  for l in range(cfg.n_layers)]
        for _ in range(max(3, args.warmup)):
            step()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(3):
            graph.replay()
        dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ms_step = dist.max(e0.elapsed_time(e1)) / args.steps
        ms.prof_enable(["expert_ffn"])
        for _ in range(args.steps):
            step()
        torch.cuda.synchronize()
        ff_n, ff_ms = ms.prof_read()["expert_ffn"]
        ms.prof_enable([])
        if ms.read_device_error(ws) != ms.OK:
            raise RuntimeError(f"device error word set in the sweep (R = {R})")
        eb = expert_bytes(cfg, unions)
        step_bytes = eb["expert_weights"] + eb["router"] + eb["lm_head"]
        ff_bytes = eb["expert_weights"] / cfg.n_layers + T * (cfg.k + 1) * (cfg.H * 2 + 4 * max(cfg.I, cfg.Is) + cfg.H * 4)
        ff_gbs = ff_bytes / (ff_ms / max(1, ff_n) / 1e3) / 1e9
        step_gbs = step_bytes / (ms_step / 1e3) / 1e9
        out["points"].append({
            "requests": R, "block_tokens": T, "block_steps_per_s": round(dist.world * R * 1e3 / ms_step, 2),
            "ms_per_step": round(ms_step, 4), "experts_kept_per_layer_mean": round(float(np.mean(unions)), 2),
            # routed tokens per kept expert (at most T k / |S|): the grouped GEMM's N, i.e. the flops per
            # weight byte on the tensor pipe
            "token_slots_per_kept_expert_at_most": round(T * cfg.k / float(np.mean(unions)), 2),
            "gbs_whole_step": round(step_gbs, 1),
            "frac_of_peak_whole_step": round(step_gbs / peak, 4) if peak else None,
            "expert_kernel_avg_ms": round(ff_ms / max(1, ff_n), 5),
            "frac_of_peak_expert_kernel": round(ff_gbs / peak, 4) if peak else None})
        del graph, ws
        torch.cuda.synchronize()
    return out


def measure_round_loop(ms, W, cfg, d, R, layers, Wlm, top_p, ws, scale, dist, thr, blocks=3):
    """Decode whole blocks (every position masked at the start) with block_decode_loop, the
    rounds as one CUDA-graph while loop, and with the same rounds driven from the host
    (block_embed + block_decode_step, reading `masked` back after each round)."""
    import numpy as np
    import torch

    T = R * cfg.P
    emb = W.to_device(W.host_activations(cfg, "emb", cfg.V), "bf16")
    pos = W.to_device(W.host_activations(cfg, "pos", cfg.P), "bf16")
    tokens = torch.zeros(T, dtype=torch.int32, device="cuda")
    masked = torch.ones(T, dtype=torch.uint8, device="cuda")
    rounds = torch.zeros(1, dtype=torch.int32, device="cuda")
    h = torch.empty((T, cfg.H), dtype=torch.float32, device="cuda")
    choice = torch.empty(T, dtype=torch.int32, device="cuda")
    conf = torch.empty(T, dtype=torch.float32, device="cuda")
    accept = torch.empty(T, dtype=torch.uint8, device="cuda")
    ncomm = torch.empty(R, dtype=torch.int32, device="cuda")

    def device_block():
        tokens.zero_()
        masked.fill_(1)
        ms.block_decode_loop(d, R, layers, Wlm, emb, pos, cfg.V - 1, top_p, thr, tokens, masked, rounds, ws,
                             logit_scale=scale)

    def host_block():
        tokens.zero_()
        masked.fill_(1)
        n = 0
        while bool(masked.any().item()) and n < cfg.P:
            ms.block_embed(d, R, tokens, masked, emb, pos, cfg.V - 1, h)
            ms.block_decode_step(d, R, layers, Wlm, top_p, thr, h, tokens, masked, choice, conf, accept,
                                 ncomm, ws, logit_scale=scale)
            n += 1
        return n

    device_block()
    torch.cuda.synchronize()
    dev_tokens, n_rounds = tokens.clone(), int(rounds.item())
    n_host = host_block()
    torch.cuda.synchronize()
    if n_host != n_rounds or not torch.equal(tokens, dev_tokens):
        raise RuntimeError("device round loop differs from the host-driven rounds")
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    e0.record(stream)
    for _ in range(blocks):
        device_block()
    e1.record(stream)
    torch.cuda.synchronize()
    ms_dev = dist.max(e0.elapsed_time(e1)) / blocks
    t0 = time.perf_counter()
    for _ in range(blocks):
        host_block()
    torch.cuda.synchronize()
    ms_host = dist.max(time.perf_counter() - t0) * 1e3 / blocks
    del emb, pos
    return {"what": "whole blocks: all positions masked, rounds until none is (LowConfidence, threshold "
                    f"{thr}), R={R}; synthetic N(0,1) bf16 embedding and positional tables",
            "logit_scale": scale, "rounds_per_block": n_rounds, "positions_per_round": round(T / n_rounds / R, 3),
            "ms_per_block_device_loop": round(ms_dev, 3), "ms_per_block_host_loop": round(ms_host, 3),
            "committed_tokens_per_s_device_loop": round(dist.world * T / (ms_dev / 1e3), 1),
            "blocks_timed": blocks, "identical_to_host_loop": True}


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def nch_for(T: int) -> int:
    """Token chunk of the expert GEMM (the library's rule): experts with more tokens are split."""
    return 32 if T <= 32 else 64


def kernel_sources_sha() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in ("expert_gemm.cu", "tc.cuh", "common.cuh"):
        h.update(open(os.path.join(ROOT, "moe_expert_step_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def layer_head_desc(cfg, R: int) -> str:
    """What ran between expert launches (the library's mode, where the shape qualifies for it)."""
    import moe_expert_step_gb300 as ms

    mode = ms.route_fusion()
    if mode == 2 and R * cfg.P <= 256 and cfg.E % 32 == 0 and cfg.E <= 256 and cfg.H % 512 == 0:
        return "combine + RMSNorm inside the router's cluster launch; coreset; gather"
    return "separate launches: combine + RMSNorm, router, coreset, gather"


def load_traffic(experts_per_launch: float, dtype: str = "bf16"):
    """DRAM bytes per expert-FFN launch: the ncu capture's bytes per expert (profiles/traffic.json,
    one Clover layer, the launch of this weight type) scaled to the experts of one launch here;
    None if the kernel sources changed since that capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get("tc_gemm_experts_fp8" if dtype == "fp8" else "tc_gemm_experts_bf16", {})
    if rec.get("kernel_sources_sha") != kernel_sources_sha() or "dram_bytes_per_expert" not in rec:
        return None
    return int(float(rec["dram_bytes_per_expert"]) * experts_per_launch)


# ------------------------------------------------------------------------------------------ oracle (CPU)
class OracleStep:
    """The fp64 oracle's whole block step, timed for real: oracle.block_decode_step over all
    40 layers (router, coreset, routed + shared experts, residual, RMSNorm per layer), the LM
    head and the LowConfidence commit, on the benchmark's block.  Every layer uses layer 0's
    weights: generating the stack's 64 GB of distinct weights on the host is far outside a
    sample budget, while the per-layer arithmetic and shapes are those of the stack.  All of
    layer 0's experts and the LM head are generated (float64) before timing starts."""

    def __init__(self, cfg, R: int):
        import numpy as np

        import oracle
        from synth import workloads as W
        self.cfg, self.R = cfg, R
        self.h0 = W.host_h0(cfg, R).astype(np.float64)
        self.masked = W.masked_subset(cfg, R)
        hl = W.HostLayer(cfg, 0)
        experts = [hl.expert(e) for e in range(cfg.E)]
        sh = hl.shared()
        self.layer = oracle.MoELayer(Wr=hl.Wr, expert=lambda e: experts[e], shared=lambda: sh)
        self.Wlm = W.host_lm_head(cfg)

    def run(self) -> float:
        """Seconds of one full step."""
        import numpy as np

        import oracle
        c = self.cfg
        t0 = time.perf_counter()
        oracle.block_decode_step(self.h0, [self.layer] * c.n_layers, self.Wlm, TOP_P, c.k, c.P, THRESHOLD,
                                 np.zeros(len(self.masked), np.int32), self.masked, bf16=True)
        return time.perf_counter() - t0

    def sample_desc(self) -> str:
        c = self.cfg
        return (f"the oracle's full block step (oracle.block_decode_step: {c.n_layers} layers of router, coreset, "
                f"routed + shared SwiGLU experts, residual and RMSNorm over {self.R} x {c.P} tokens, then the "
                f"V={c.V} LM head and the commit), every layer with layer 0's weights (the 64 GB of distinct "
                f"weights are not generated on the host); weights generated before timing; numpy float64")


def cpu_baseline(cfg, R: int, reps: int = 3) -> dict:
    s = OracleStep(cfg, R)
    secs = [s.run() for _ in range(reps)]
    return {"value": round(R / statistics.median(secs), 5), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": s.sample_desc() + f"; median of {reps} timed steps",
            "step_s": round(statistics.median(secs), 3)}


def run_reference(args, dist: Dist):
    cfg = workload(args.config)
    R = args.requests
    s = OracleStep(cfg, R)
    for _ in range(args.warmup):
        s.run()
    total = sum(s.run() for _ in range(args.steps))
    value = args.steps * R / total   # one step advances R blocks
    base = {"value": round(value, 5), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": s.sample_desc() + "; every step timed in full"}
    return {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": UNIT, "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_desc(cfg, R, args), "cpu_baseline": base,
            "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    if args.impl == "reference":
        dist = Dist("gloo")
        if dist.rank != 0:
            dist.close()
            return
        print(json.dumps(run_reference(args, dist)), flush=True)
        dist.close()
        return
    dist = Dist("nccl")
    line, cfg = run_gpu(args, dist)
    if dist.rank == 0:
        if dist.world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(cfg, args.requests)
        else:
            line["cpu_baseline"] = None
        print(json.dumps(line), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
