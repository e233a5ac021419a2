#!/usr/bin/env python3
"""Benchmark of the GB300 routed-MoE FFN block (one JSON line on stdout).

Default workload: single-token decode through a 30-layer stack of MoE blocks
(attention omitted; RMSNorm -> block -> residual per layer), d_model 2816, 128
experts top-8, expert width 704, shared width 2112, 4-bit group-64 experts,
8-bit router, BF16 activations, seed 1.  One step = one token through all 30
layers; ``value`` = tokens/s over all ranks, timed over exactly --steps graph
replays.  The same line then carries, under ``configs``, every other workload
(tiny T=4, prefill T=512, skewed decode T=64, prefill T=4096): for each, the
median, p10 and p90 of --calls timed calls, e2e, the dominant kernel's
roofline, whole-step HBM and tensor fractions and the oracle's CPU baselines.
``--config C`` makes workload C the headline instead.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config C]
                    [--calls N] [--no-all-configs] [--no-cpu-baseline]

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

PD_LAUNCH_NOTE = "single-launch decode kernel (all layers of the step in one persistent launch)"


def l2_flush_bytes():
    return 256 << 20  # twice the 129 MB L2


def time_calls(run, n, stream, flush=None):
    """Per-call device times (ms) of n calls, each between two events on the
    launching stream; ``flush`` (outside the event pair) evicts L2 first."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for a, b in evs:
            if flush is not None:
                flush()
            a.record(stream)
            run()
            b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def pct(v, q):
    return float(np.percentile(np.asarray(v, dtype=np.float64), q))


class Workload:
    """One workload on the device: its layers, a captured CUDA graph of one
    step, and the routing the step produced (for the byte counts)."""

    def __init__(self, mx, cfg, stream):
        import torch
        self.cfg = cfg
        self.stream = stream
        n_layers, T, K = cfg.layers, cfg.T, cfg.K
        act = mx.MX_BF16 if cfg.act == "bf16" else mx.MX_F32
        t0 = time.time()
        self.hosts = [synth.make_layer(cfg, l) for l in range(n_layers)]
        self.devs = [mx.DeviceLayer(h, act) for h in self.hosts]
        self.x0 = synth.make_x(cfg)
        self.gen_s = time.time() - t0
        xv = self.x0.view(np.int16) if self.x0.dtype == np.uint16 else self.x0
        self.xv = xv
        self.x_init = torch.from_numpy(xv).cuda()
        self.x_io = torch.empty_like(self.x_init)
        self.idx = torch.zeros((n_layers, T, K), dtype=torch.int32, device="cuda")
        self.wts = torch.zeros((n_layers, T, K), dtype=torch.float32, device="cuda")
        self.stack = mx.Stack(self.devs)
        self.nbytes = (mx.stack_workspace_bytes(self.devs[0].layout, T) if n_layers > 1
                       else mx.workspace_bytes(self.devs[0].layout, T))
        self.ws = torch.empty(self.nbytes, dtype=torch.uint8, device="cuda")
        mx.workspace_init(self.ws, self.nbytes, stream)
        self.out1 = torch.empty_like(self.x_init)
        self.mx = mx
        with torch.cuda.stream(stream):
            self.step(stream)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=stream):
            self.step(stream)
        torch.cuda.synchronize()
        mx.workspace_check(self.ws, stream)
        idx_h = self.idx.cpu().numpy()
        self.per_layer = [stage_bytes(cfg, len(np.unique(idx_h[l])), T) for l in range(n_layers)]
        self.step_bytes = sum(b["total"] for b in self.per_layer)
        self.step_flops = n_layers * flops(cfg, T)

    def step(self, s):
        """One step: the workload's input through the block(s), on stream s."""
        cfg, mx = self.cfg, self.mx
        if cfg.layers > 1:
            self.x_io.copy_(self.x_init)
            mx.stack_forward(self.x_io, cfg.T, self.stack, self.idx, self.wts, self.ws, self.nbytes, rms_eps=1e-6,
                             stream=s)
        else:
            mx.layer_forward_ex(self.x_init, cfg.T, self.devs[0], self.out1, self.idx[0], self.wts[0], self.ws,
                                self.nbytes, stream=s)

    def stage_profile(self, n):
        """Per-stage event timing of n direct API calls (not graph replays)."""
        import torch
        mx = self.mx
        mx.profile_enable(True)
        mx.profile_read(reset=True)
        with torch.cuda.stream(self.stream):
            for _ in range(n):
                self.step(self.stream)
        torch.cuda.synchronize()
        prof = mx.profile_read(reset=True)
        mx.profile_enable(False)
        return prof

    def e2e(self, steps, warmup):
        """Pinned host input -> device, the C-ABI call (no graph), outputs ->
        pinned host, every step; returns (ms for all steps, h2d, d2h bytes)."""
        import torch
        cfg, mx, s = self.cfg, self.mx, self.stream
        T, K, n_layers = cfg.T, cfg.K, cfg.layers
        x_pin = torch.from_numpy(self.xv.copy()).pin_memory()
        out_pin = torch.empty(self.x_init.shape, dtype=self.x_init.dtype).pin_memory()
        idx_pin = torch.empty(self.idx.shape, dtype=torch.int32).pin_memory()
        w_pin = torch.empty(self.wts.shape, dtype=torch.float32).pin_memory()
        x_dev = torch.empty_like(self.x_init)

        def e2e_step():
            x_dev.copy_(x_pin, non_blocking=True)
            if n_layers > 1:
                mx.stack_forward(x_dev, T, self.stack, self.idx, self.wts, self.ws, self.nbytes, rms_eps=1e-6,
                                 stream=s)
                out_pin.copy_(x_dev, non_blocking=True)
            else:
                mx.layer_forward_ex(x_dev, T, self.devs[0], self.out1, self.idx[0], self.wts[0], self.ws,
                                    self.nbytes, stream=s)
                out_pin.copy_(self.out1, non_blocking=True)
            idx_pin.copy_(self.idx, non_blocking=True)
            w_pin.copy_(self.wts, non_blocking=True)

        with torch.cuda.stream(s):
            for _ in range(warmup):
                e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            for _ in range(steps):
                e2e_step()
            e1.record(s)
        torch.cuda.synchronize()
        es = self.x_init.element_size()
        return e0.elapsed_time(e1), T * cfg.D * es, T * cfg.D * es + n_layers * T * K * 8


def path_of(cfg):
    single = cfg.T <= PD_MAX_T and os.environ.get("MX_MOE_SINGLE_LAUNCH", "1") != "0"
    prefill = cfg.T > PD_MAX_T and cfg.act == "bf16" and os.environ.get("MX_MOE_PREFILL_GEMM", "1") != "0"
    return "prefill" if prefill else ("single" if single else "multi")


def launches_per_step(cfg):
    path = path_of(cfg)
    if path == "prefill":
        # norm, router floats, logits GEMM, top-k, grouping, tile index,
        # scatter, gate/up GEMM, down GEMM, combine
        return cfg.layers * 10
    if path == "single":
        return -(-cfg.layers // PD_MAX_LAYERS)
    return cfg.layers * 3 * ((cfg.T + 63) // 64)


def roofline_of(wl, prof, peaks, peak_src):
    """The dominant kernel's achieved rate against its roof: the algorithmic
    bytes (or FLOPs) of one launch over its mean CUDA-event duration."""
    cfg, path = wl.cfg, path_of(wl.cfg)
    T, K, D = cfg.T, cfg.K, cfg.D
    gu_ms, gu_n = prof["gate_up"]
    gu_s = gu_ms / 1e3 / max(gu_n, 1)
    workload = cfg.name
    if path == "prefill":
        kname = "pf_gemm<0>"
        gu_flops = 2 * 2 * T * (K * cfg.I + cfg.S) * D
        achieved = gu_flops / gu_s / 1e12
        roof = {"bound": "tensor", "kernel": kname, "achieved": round(achieved, 1),
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                "peak_source": peak_src + " (bf16 burst; fp16 is the same tensor rate)",
                "traffic": committed_traffic(kname, workload),
                "flops_per_launch": int(gu_flops), "launch_us": round(gu_s * 1e6, 2), "launches_timed": gu_n}
        dn_ms, dn_n = prof["down"]
        if dn_n:
            dn_flops = 2 * T * (K * cfg.I + cfg.S) * D
            roof["down_gemm_tflops"] = round(dn_flops / (dn_ms / 1e3 / dn_n) / 1e12, 1)
        return roof
    if path == "single":
        launches = -(-cfg.layers // PD_MAX_LAYERS)
        kname, bytes_launch = "pd_kernel", wl.step_bytes / launches
    else:
        kname, bytes_launch = "gateup_kernel", statistics.mean(b["gate_up"] for b in wl.per_layer)
    achieved = bytes_launch / gu_s / 1e9
    roof = {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peak_src,
            "traffic": committed_traffic(kname, workload), "bytes_per_launch": int(bytes_launch),
            "launch_us": round(gu_s * 1e6, 2), "launches_timed": gu_n}
    if cfg.T * cfg.D * 2 * 64 < 128e6 and wl.step_bytes < 100e6:
        roof["note"] = "working set inside L2 (L2 flushed between timed calls): latency-bound, not HBM-bound"
    return roof


def step_fractions(wl, ms_per_step, peaks):
    gbs = wl.step_bytes / (ms_per_step / 1e3) / 1e9
    tfs = wl.step_flops / (ms_per_step / 1e3) / 1e12
    return {"step_bytes": int(wl.step_bytes), "step_hbm_gbs": round(gbs, 1),
            "step_hbm_frac": round(gbs / peaks["hbm_gbs"], 4), "step_flops": int(wl.step_flops),
            "step_tflops": round(tfs, 3), "step_tensor_frac": round(tfs / peaks["bf16_tflops"], 4)}


def config_entry(args, ci, mx, stream, peaks, peak_src, want_cpu):
    """A non-headline workload: per-call distribution over >= 100 timed calls,
    stage profile, e2e, roofline and the CPU baselines."""
    import torch
    cfg = synth.CONFIGS[ci]
    wl = Workload(mx, cfg, stream)
    flush = None
    if wl.step_bytes < 2 * 129e6:
        buf = torch.empty(l2_flush_bytes(), dtype=torch.uint8, device="cuda")
        flush = lambda: buf.fill_(1)  # noqa: E731
    for _ in range(max(args.warmup, 5)):
        wl.graph.replay()
    torch.cuda.synchronize()
    calls = time_calls(wl.graph.replay, args.calls, stream, flush)
    med = pct(calls, 50)
    prof = wl.stage_profile(max(3, min(args.calls, 30)))
    e2e_ms, h2d, d2h = wl.e2e(max(10, min(args.steps, 50)), 3)
    n_e2e = max(10, min(args.steps, 50))
    entry = {"index": ci, "workload": cfg.name, "T": cfg.T, "layers": cfg.layers, "path": path_of(cfg),
             "value": round(cfg.T / (med / 1e3), 2), "unit": "tokens/s", "ms_per_step": round(med, 5),
             "ms_p10": round(pct(calls, 10), 5), "ms_p90": round(pct(calls, 90), 5), "timed_calls": len(calls),
             "l2": "flushed between timed calls" if flush else "inputs larger than L2",
             "e2e": {"value": round(n_e2e * cfg.T / (e2e_ms / 1e3), 2), "unit": "tokens/s",
                     "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
             "roofline": roofline_of(wl, prof, peaks, peak_src),
             "stage_us": {k: round(v[0] * 1e3 / max(v[1], 1), 2) for k, v in prof.items()},
             "gpu_launches_per_step": launches_per_step(cfg)}
    entry.update(step_fractions(wl, med, peaks))
    if want_cpu:
        entry["cpu_baseline"] = cpu_baseline(cfg, wl.hosts, wl.x0, budget_s=args.cpu_budget)
    del wl
    torch.cuda.empty_cache()
    return entry


def bench_ours(args, cfg, world, rank, local, pg):
    import torch

    import __graft_entry__
    import expert_ffn_gb300 as mx
    __graft_entry__.build()
    torch.cuda.set_device(local)
    dev_name = torch.cuda.get_device_name(local)
    stream = torch.cuda.Stream()
    T = cfg.T
    peaks, peak_src = load_peaks()

    wl = Workload(mx, cfg, stream)
    flush = None
    if wl.step_bytes < 2 * 129e6:
        buf = torch.empty(l2_flush_bytes(), dtype=torch.uint8, device="cuda")
        flush = lambda: buf.fill_(1)  # noqa: E731

    def barrier():
        if pg is not None:
            pg.barrier()

    for _ in range(args.warmup):
        wl.graph.replay()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        tw0 = time.time()
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(args.steps):
                if flush is not None:
                    flush()
                wl.graph.replay()
            ev1.record(stream)
        torch.cuda.synchronize()
        tw1 = time.time()
    barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1), pg, "cuda")
    clocks = clk.summary(tw0, tw1)
    ms_per_step = ms / args.steps
    value = job_tokens_per_s(world, args.steps, T, ms)

    # the per-call distribution (>= 100 calls, outside the headline region)
    calls = time_calls(wl.graph.replay, args.calls, stream, flush)
    prof = wl.stage_profile(max(3, min(args.steps, 50)))
    roof = roofline_of(wl, prof, peaks, peak_src)
    e2e_ms, h2d, d2h = wl.e2e(args.steps, args.warmup)
    e2e_ms = max_over_ranks(e2e_ms, pg, "cuda")

    n_layers = cfg.layers
    workload = cfg.name if n_layers == synth.CONFIGS[args.config].layers else f"{cfg.name}[{n_layers} layers]"
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if cfg.act == "bf16" else "f32", "data": "synthetic (seeded; random-init "
        "4-bit experts, 8-bit router)",
        "config": {"workload": workload, "T": T, "layers": n_layers, "d_model": cfg.D, "experts": cfg.E,
                   "top_k": cfg.K, "d_expert": cfg.I, "d_shared": cfg.S, "parallelism": f"replicas x{world}",
                   "l2": ("flushed between timed steps" if flush else
                          f"inputs larger than L2 ({sum(h.blob.nbytes for h in wl.hosts) / 1e9:.1f} GB of expert "
                          "weights; each step reads its selected experts from HBM)"),
                   "timing": "CUDA graph replay of the step, CUDA events on the launching stream"},
        "ms_p10": round(pct(calls, 10), 5), "ms_p50": round(pct(calls, 50), 5), "ms_p90": round(pct(calls, 90), 5),
        "timed_calls": len(calls),
        "stage_us": {k: round(v[0] * 1e3 / max(v[1], 1), 2) for k, v in prof.items()},
        "roofline": roof,
        "clocks": clocks,
        "e2e": {"value": round(job_tokens_per_s(world, args.steps, T, e2e_ms), 2), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "pinned host input copied in, the C-ABI call (no graph), outputs copied out, every step"},
        "gpu_launches": args.steps * launches_per_step(cfg),
        "device": dev_name, "gen_s": round(wl.gen_s, 1),
    }
    res.update(step_fractions(wl, ms_per_step, peaks))
    want_cpu = rank == 0 and not args.no_cpu_baseline
    if want_cpu:
        res["cpu_baseline"] = cpu_baseline(cfg, wl.hosts, wl.x0, budget_s=args.cpu_budget)
    del wl
    torch.cuda.empty_cache()
    if args.all_configs:
        others = {}
        for ci in sorted(synth.CONFIGS):
            if ci == args.config:
                continue
            e = config_entry(args, ci, mx, stream, peaks, peak_src, want_cpu)
            others[e["workload"]] = e
        res["configs"] = others
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
    """Time the oracle as it stands on a bounded sample; scale to tokens/s.
    One host core, then every core (one thread per core, each running the
    single-threaded oracle on its own tokens -- or, for the one-token stack, its
    own independent token stream; ctypes releases the GIL during the call)."""
    import concurrent.futures as cf

    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
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
        with cf.ThreadPoolExecutor(max_workers=cores) as ex:
            t0 = time.perf_counter()
            list(ex.map(lambda _: oracle_step(cfg, hosts, x0, nl, 1), range(cores)))
            dt_all = time.perf_counter() - t0
        value_all = cores * (nl / cfg.layers) / dt_all
        sample_all = f"{cores} independent one-token streams through {nl} of {cfg.layers} layers, one per core"
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
        n_all = int(max(1, min(cfg.T, cores * budget_s // max(per_tok, 1e-6))))
        t0 = time.perf_counter()
        oracle.block_forward_tokens(hosts[0], x0, np.arange(n_all), threads=cores)
        dt_all = time.perf_counter() - t0
        value_all = n_all / dt_all
        sample_all = f"{n_all} of {cfg.T} tokens split over {cores} threads"
    return {"value": round(value, 4), "unit": "tokens/s", "cores": 1, "kind": kind, "sample": sample,
            "cpu": platform_cpu(),
            "all_cores": {"value": round(value_all, 4), "unit": "tokens/s", "cores": cores, "sample": sample_all}}


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
    ap.add_argument("--config", type=int, default=1, choices=[0, 1, 2, 3, 4])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=8.0, help="seconds of oracle work per CPU sample")
    ap.add_argument("--calls", type=int, default=100, help="timed calls of the per-call distribution")
    ap.add_argument("--no-all-configs", dest="all_configs", action="store_false",
                    help="time only --config (the other workloads are added under 'configs' by default)")
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
