#!/usr/bin/env python3
"""Benchmark of the GB300 routed-MoE FFN block (one JSON line on stdout).

Default workload: single-token decode through a 30-layer stack of MoE blocks
(attention omitted; RMSNorm -> block -> residual per layer), d_model 2816, 128
experts top-8, expert width 704, shared width 2112, 4-bit group-64 experts,
8-bit router, BF16 activations, seed 1.  One step = one token through all 30
layers; ``value`` = tokens/s over all ranks.  ``--config 2|3|4`` times one
block on the other workloads (prefill T=512, skewed decode T=64, prefill
T=4096) instead.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config C]

``--impl reference`` times the CPU oracle (the plain C reference) on the host
cores, a bounded sample per step.  Under torchrun (N > 1) each rank runs its own
replica (no data-path collective) and the timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s; decode HBM GB/s and prefill TFLOP/s as % of GB300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = ("expert_ffn_gb300/csrc/mx_decode.cu", "expert_ffn_gb300/csrc/mx_ffn_decode.cu",
                  "expert_ffn_gb300/csrc/mx_common.cuh", "expert_ffn_gb300/csrc/mx_route.cu",
                  "expert_ffn_gb300/csrc/mx_prefill.cu")
PD_MAX_T, PD_MAX_LAYERS = 4, 30  # single-launch decode path: tokens per call, layers per launch


# ------------------------------------------------------------------ helpers

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_src_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str):
    """dram read+write bytes per launch from a committed ncu capture, or None
    when there is none or the kernel sources changed since it was taken."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    e = d.get(f"{kernel}@{workload}")
    if not e or e.get("src_sha") != kernel_src_hash():
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampler run during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t_start: float, t_stop: float):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, f in enumerate(flags) if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend="nccl")
        pg = dist
    return world, rank, local, pg


def max_over_ranks(ms: float, pg, device: str) -> float:
    """The slowest rank's time: every rank's replica ran the same work, so the
    job took as long as its slowest rank (identity without a process group)."""
    if pg is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, steps: int, tokens_per_step: float, ms: float) -> float:
    """Whole-job throughput: every rank processed steps x tokens_per_step
    tokens (independent replicas, weak scaling) in at most ms milliseconds."""
    return world * steps * tokens_per_step / (ms / 1e3)


# ----------------------------------------------------------- workload bytes

def qbytes(rows, cols, bits):
    return rows * cols * bits // 8 + 2 * rows * (cols // 64) * 2


def stage_bytes(cfg, unique_experts: int, T: int):
    """Algorithmic HBM bytes of one block call, per stage: the selected experts'
    packed weights + BF16 scales + biases (each distinct expert read once), the
    shared expert, the router, and the activations read and written."""
    D, I, S, E, K = cfg.D, cfg.I, cfg.S, cfg.E, cfg.K
    es = 4 if cfg.act == "f32" else 2
    route = qbytes(E, D, 8) + T * D * es + T * K * 8
    gate_up = unique_experts * 2 * qbytes(I, D, 4) + 2 * qbytes(S, D, 4) + T * D * es
    down = unique_experts * qbytes(D, I, 4) + qbytes(D, S, 4) + T * D * es * 2
    return {"route": route, "gate_up": gate_up, "down": down, "total": route + gate_up + down}


def flops(cfg, T):
    return 2 * T * cfg.E * cfg.D + T * cfg.K * 6 * cfg.I * cfg.D + T * 6 * cfg.S * cfg.D


# ------------------------------------------------------------------ ours

def bench_ours(args, cfg, world, rank, local, pg):
    import torch

    import __graft_entry__
    import expert_ffn_gb300 as mx
    __graft_entry__.build()
    torch.cuda.set_device(local)
    dev_name = torch.cuda.get_device_name(local)
    stream = torch.cuda.Stream()
    n_layers = cfg.layers
    T, K, D = cfg.T, cfg.K, cfg.D
    act = mx.MX_BF16 if cfg.act == "bf16" else mx.MX_F32

    t0 = time.time()
    hosts = [synth.make_layer(cfg, l) for l in range(n_layers)]
    devs = [mx.DeviceLayer(h, act) for h in hosts]
    x0 = synth.make_x(cfg)
    gen_s = time.time() - t0
    xv = x0.view(np.int16) if x0.dtype == np.uint16 else x0
    x_init = torch.from_numpy(xv).cuda()
    x_io = torch.empty_like(x_init)
    idx = torch.zeros((n_layers, T, K), dtype=torch.int32, device="cuda")
    wts = torch.zeros((n_layers, T, K), dtype=torch.float32, device="cuda")
    stack = mx.Stack(devs)
    if n_layers > 1:
        nbytes = mx.stack_workspace_bytes(devs[0].layout, T)
    else:
        nbytes = mx.workspace_bytes(devs[0].layout, T)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    mx.workspace_init(ws, nbytes, stream)
    out1 = torch.empty_like(x_init)

    def step(s):
        """One step: the workload's input through the block(s), on stream s."""
        if n_layers > 1:
            x_io.copy_(x_init)
            mx.stack_forward(x_io, T, stack, idx, wts, ws, nbytes, rms_eps=1e-6, stream=s)
        else:
            mx.layer_forward_ex(x_init, T, devs[0], out1, idx[0], wts[0], ws, nbytes, stream=s)

    # CUDA graph of one step (the library allocates nothing and syncs nothing)
    with torch.cuda.stream(stream):
        step(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step(stream)
    torch.cuda.synchronize()

    # routing statistics for the byte counts
    idx_h = idx.cpu().numpy()
    per_layer = [stage_bytes(cfg, len(np.unique(idx_h[l])), T) for l in range(n_layers)]
    step_bytes = sum(b["total"] for b in per_layer)
    gu_bytes_per_launch = statistics.mean(b["gate_up"] for b in per_layer)
    step_flops = n_layers * flops(cfg, T)

    def barrier():
        if pg is not None:
            pg.barrier()

    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        tw0 = time.time()
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            ev1.record(stream)
        torch.cuda.synchronize()
        tw1 = time.time()
    barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1), pg, "cuda")
    clocks = clk.summary(tw0, tw1)
    ms_per_step = ms / args.steps
    value = job_tokens_per_s(world, args.steps, T, ms)

    # stage timing (events on the launching stream, direct API calls)
    mx.profile_enable(True)
    nprof = max(3, min(args.steps, 50))
    with torch.cuda.stream(stream):
        for _ in range(nprof):
            step(stream)
    torch.cuda.synchronize()
    prof = mx.profile_read(reset=True)
    mx.profile_enable(False)
    gu_ms, gu_n = prof["gate_up"]
    gu_s = gu_ms / 1e3 / max(gu_n, 1)
    peaks, peak_src = load_peaks()

    # end to end: pinned host input -> device, API calls, result -> host, every step
    x_pin = torch.from_numpy(xv.copy()).pin_memory()
    out_pin = torch.empty(x_init.shape, dtype=x_init.dtype).pin_memory()
    idx_pin = torch.empty(idx.shape, dtype=torch.int32).pin_memory()
    w_pin = torch.empty(wts.shape, dtype=torch.float32).pin_memory()
    x_dev = torch.empty_like(x_init)

    def e2e_step(s):
        x_dev.copy_(x_pin, non_blocking=True)
        if n_layers > 1:
            mx.stack_forward(x_dev, T, stack, idx, wts, ws, nbytes, rms_eps=1e-6, stream=s)
            out_pin.copy_(x_dev, non_blocking=True)
        else:
            mx.layer_forward_ex(x_dev, T, devs[0], out1, idx[0], wts[0], ws, nbytes, stream=s)
            out_pin.copy_(out1, non_blocking=True)
        idx_pin.copy_(idx, non_blocking=True)
        w_pin.copy_(wts, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            e2e_step(stream)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step(stream)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), pg, "cuda")
    es = x_init.element_size()
    h2d = T * D * es
    d2h = T * D * es + n_layers * T * K * 8

    workload = cfg.name if n_layers == synth.CONFIGS[args.config].layers else f"{cfg.name}[{n_layers} layers]"
    single = T <= PD_MAX_T and os.environ.get("MX_MOE_SINGLE_LAUNCH", "1") != "0"
    prefill = T > 64 and cfg.act == "bf16" and os.environ.get("MX_MOE_PREFILL_GEMM", "1") != "0"
    if prefill:
        # the gate/up grouped GEMM (tcgen05, FP16 operands, fp32 accumulation)
        # is the dominant kernel: its algorithmic FLOPs per launch
        # norm, router floats, logits GEMM, top-k, grouping, tile index, scatter,
        # gate/up GEMM, down GEMM, combine
        launches = n_layers * 10
        kname = "pf_gemm<0>"
        gu_flops = 2 * 2 * T * (K * cfg.I + cfg.S) * D
        achieved = gu_flops / gu_s / 1e12
        # FP16 and BF16 run at the same tensor rate: the BF16 cuBLAS peak applies
        roof = {"bound": "tensor", "kernel": kname, "achieved": round(achieved, 1),
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                "peak_source": peak_src + " (bf16 burst; fp16 is the same tensor rate)",
                "traffic": committed_traffic(kname, workload),
                "flops_per_launch": int(gu_flops), "launch_us": round(gu_s * 1e6, 2), "launches_timed": gu_n}
        dn_ms, dn_n = prof["down"]
        if dn_n:
            dn_flops = 2 * T * (K * cfg.I + cfg.S) * D
            roof["down_gemm_tflops"] = round(dn_flops / (dn_ms / 1e3 / dn_n) / 1e12, 1)
    else:
        if single:
            # one persistent launch runs every layer of the step (up to 30 per
            # launch): its algorithmic bytes are the whole step's
            launches = -(-n_layers // PD_MAX_LAYERS)
            kname, bytes_launch = "pd_kernel", step_bytes / launches
        else:
            launches = n_layers * 3 * ((T + 63) // 64)
            kname, bytes_launch = "gateup_kernel", gu_bytes_per_launch
        achieved = bytes_launch / gu_s / 1e9
        roof = {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "peak_source": peak_src,
                "traffic": committed_traffic(kname, workload),
                "bytes_per_launch": int(bytes_launch), "launch_us": round(gu_s * 1e6, 2),
                "launches_timed": gu_n}
    step_gbs = step_bytes / (ms_per_step / 1e3) / 1e9
    stages_us = {k: round(v[0] * 1e3 / max(v[1], 1), 2) for k, v in prof.items()}
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if cfg.act == "bf16" else "f32", "data": "synthetic (seeded; random-init "
        "4-bit experts, 8-bit router)",
        "config": {"workload": workload, "T": T, "layers": n_layers, "d_model": D, "experts": cfg.E, "top_k": K,
                   "d_expert": cfg.I, "d_shared": cfg.S, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2 ({sum(h.blob.nbytes for h in hosts) / 1e9:.1f} GB of expert "
                         "weights; each step reads its selected experts from HBM)",
                   "timing": "CUDA graph replay of the step, CUDA events on the launching stream"},
        "step_bytes": int(step_bytes), "step_hbm_gbs": round(step_gbs, 1),
        "step_hbm_frac": round(step_gbs / peaks["hbm_gbs"], 4),
        "step_tflops": round(step_flops / (ms_per_step / 1e3) / 1e12, 3),
        "stage_us": stages_us,
        "roofline": roof,
        "clocks": clocks,
        "e2e": {"value": round(job_tokens_per_s(world, args.steps, T, e2e_ms), 2), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "pinned host input copied in, the C-ABI call (no graph), outputs copied out, every step"},
        "gpu_launches": args.steps * launches,
        "device": dev_name, "gen_s": round(gen_s, 1),
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(cfg, hosts, x0, budget_s=args.cpu_budget)
    return res


# --------------------------------------------------------------- CPU oracle

def oracle_step(cfg, hosts, x0, n_layers_sample: int, n_tokens: int):
    import oracle
    x = x0[:n_tokens]
    if cfg.layers > 1:
        oracle.stack_forward(hosts[:n_layers_sample], x, 1e-6)
    else:
        oracle.block_forward(hosts[0], x)


def cpu_baseline(cfg, hosts, x0, budget_s: float = 20.0, kind: str = "oracle"):
    """Time the oracle as it stands on a bounded sample; scale to tokens/s."""
    import oracle
    oracle.build()
    if cfg.layers > 1:
        # one token through the layers; time one layer first to size the sample
        t0 = time.perf_counter()
        oracle_step(cfg, hosts, x0, 1, 1)
        per_layer = time.perf_counter() - t0
        nl = int(max(1, min(cfg.layers, budget_s // max(per_layer, 1e-6))))
        t0 = time.perf_counter()
        oracle_step(cfg, hosts, x0, nl, 1)
        dt = time.perf_counter() - t0
        value = (nl / cfg.layers) / dt
        sample = f"1 token through {nl} of {cfg.layers} layers (tokens/s scaled by {nl}/{cfg.layers})"
    else:
        t0 = time.perf_counter()
        oracle_step(cfg, hosts, x0, 1, 1)
        per_tok = time.perf_counter() - t0
        n = int(max(1, min(cfg.T, budget_s // max(per_tok, 1e-6))))
        t0 = time.perf_counter()
        oracle_step(cfg, hosts, x0, 1, n)
        dt = time.perf_counter() - t0
        value = n / dt
        sample = f"{n} of {cfg.T} tokens through the block"
    return {"value": round(value, 4), "unit": "tokens/s", "cores": 1, "kind": kind, "sample": sample,
            "cpu": platform_cpu()}


def platform_cpu():
    import platform
    return f"{platform.machine()} x{os.cpu_count()}"


def bench_reference(args, cfg, world, rank, pg):
    """The oracle on the host cores, timed per step on a bounded sample."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    hosts = [synth.make_layer(cfg, l) for l in range(cfg.layers)]
    x0 = synth.make_x(cfg)
    # size the per-step sample so that all steps fit in about two minutes
    t0 = time.perf_counter()
    oracle_step(cfg, hosts, x0, 1, 1)
    unit = time.perf_counter() - t0
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    if cfg.layers > 1:
        nl = int(max(1, min(cfg.layers, per_step_budget // max(unit, 1e-6))))
        n_tok, tokens_per_step = 1, nl / cfg.layers
        sample = f"1 token through {nl} of {cfg.layers} layers per step"
    else:
        nl = 1
        n_tok = int(max(1, min(cfg.T, per_step_budget // max(unit, 1e-6))))
        tokens_per_step = n_tok
        sample = f"{n_tok} of {cfg.T} tokens per step"
    for _ in range(args.warmup):
        oracle_step(cfg, hosts, x0, nl, n_tok)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(cfg, hosts, x0, nl, n_tok)
    dt = time.perf_counter() - t0
    value = args.steps * tokens_per_step / dt
    return {"metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded)",
            "impl": "reference",
            "config": {"workload": cfg.name, "T": cfg.T, "layers": cfg.layers},
            "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": sample, "cpu": platform_cpu()},
            "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=1, choices=[1, 2, 3, 4])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--layers", type=int, default=0,
                    help="run only the first N layers of the workload (profiling captures; 0 = all)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    cfg = synth.CONFIGS[args.config]
    if args.layers > 0:
        import dataclasses
        cfg = dataclasses.replace(cfg, layers=min(args.layers, cfg.layers))
    world, rank, local, pg = dist_setup(args)
    if args.impl == "reference":
        res = bench_reference(args, cfg, world, rank, pg)
    else:
        res = bench_ours(args, cfg, world, rank, local, pg)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
