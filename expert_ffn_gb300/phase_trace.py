"""Phase trace of the single-launch decode kernel.

Builds a second copy of ``libmx_moe.so`` with ``-DMX_PD_TRACE`` (into
``expert_ffn_gb300/_build_trace``; the product library is untouched), runs the
30-layer single-token decode stack of the decode workload, and prints, for
layer 10 of the launch, when each phase of the layer ended on each CTA
(%globaltimer, microseconds from the earliest CTA's start of the layer):
median, fastest and slowest CTA, each the median over several launches.

    python -m expert_ffn_gb300.phase_trace [--runs N]

Phases, in kernel order: start of the layer, prologue (RMSNorm, planes of x;
indented: its sum of squares, elementwise pass, plane scale, group sums and
planes), router rows, the shared-expert units, the logit exchange (indented:
the CTA's own barrier, the grid counter reached), top-k / softmax / grouping
(indented: logit loads issued, top-k and softmax done), the routed units, the
y exchange, the rebuild of x_{l+1}.  CTAs without shared units pass the
shared-unit phase at once, and CTAs without routed units the routed one.
Other indented rows time the inside of each CTA's
first routed unit (over the CTAs that hold one): when the producer warp saw
the routing, when item 0 and item 7 of its gate/up work had landed (as warp 0
and warp 7 saw them) and when warp 7 was done with item 7, the end of its
gate/up work, of the planes of h, and when each of its four down items had
landed in shared memory and was done.
"""
from __future__ import annotations

import argparse
import ctypes
import os
import sys

PHASES = ["layer start", "prologue", "router rows", "shared units", "logit exchange", "top-k + grouping",
          "  unit gate/up", "  unit h planes", None, "routed units", "y exchange", "x rebuild",
          "  down 0 landed", "  down 1 landed", "  down 2 landed", "  down 3 landed",
          "  down 0 done", "  down 1 done", "  down 2 done", "  down 3 done",
          "  item 0 landed", "  item 7 landed", "  item 7 done", "  routing seen",
          "  sum of squares", "  elementwise", "  plane scale", "  group sums, planes",
          "  logits loads issued", "  top-k, softmax", "  own barrier", "  counter reached"]
UNIT_PHASES = range(6, 24)  # inside the first routed unit of a CTA (CTAs that hold one)
TRACE_LAYER, TRACE_CTAS, TRACE_PTS = 10, 160, 32


def build_trace_lib() -> str:
    from . import build
    saved = (build.NVCC_FLAGS, build.BUILD, build.LIB)
    try:
        build.NVCC_FLAGS = list(build.NVCC_FLAGS) + ["-DMX_PD_TRACE"]
        build.BUILD = os.path.join(build.PKG, "_build_trace")
        build.LIB = os.path.join(build.BUILD, "libmx_moe.so")
        return build.build()
    finally:
        build.NVCC_FLAGS, build.BUILD, build.LIB = saved


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--runs", type=int, default=8)
    args = ap.parse_args(argv)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    import numpy as np
    import torch

    import expert_ffn_gb300 as mx
    import synth

    lib_path = build_trace_lib()
    mx.LIB_PATH = lib_path  # the binding loads this copy in this process
    L = mx.lib()
    L.mx_pd_trace_read.argtypes = [ctypes.c_void_p]
    L.mx_pd_trace_read.restype = ctypes.c_int

    cfg = synth.CONFIGS[1]
    T, K = cfg.T, cfg.K
    devs = [mx.DeviceLayer(synth.make_layer(cfg, l), mx.MX_BF16) for l in range(cfg.layers)]
    x0 = synth.make_x(cfg)
    x_init = torch.from_numpy(x0.view(np.int16)).cuda()
    x_io = torch.empty_like(x_init)
    idx = torch.zeros((cfg.layers, T, K), dtype=torch.int32, device="cuda")
    wts = torch.zeros((cfg.layers, T, K), dtype=torch.float32, device="cuda")
    stack = mx.Stack(devs)
    nbytes = mx.stack_workspace_bytes(devs[0].layout, T)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    mx.workspace_init(ws, nbytes, stream)
    ncta = torch.cuda.get_device_properties(0).multi_processor_count
    rows = {i: [] for i, n in enumerate(PHASES) if n}
    for it in range(args.runs + 3):
        x_io.copy_(x_init)
        with torch.cuda.stream(stream):
            mx.stack_forward(x_io, T, stack, idx, wts, ws, nbytes, rms_eps=1e-6, stream=stream)
        torch.cuda.synchronize()
        if it < 3:
            continue
        buf = np.zeros((TRACE_CTAS, TRACE_PTS), dtype=np.uint64)
        if L.mx_pd_trace_read(buf.ctypes.data) != 0:
            raise RuntimeError("mx_pd_trace_read failed")
        stamps = buf[:ncta].astype(np.int64)
        t0 = stamps[:, 0].min()
        for i in rows:
            col = stamps[:, i]
            if i in UNIT_PHASES:
                col = col[col != 0]  # CTAs that ran a routed unit
            v = (col - t0) / 1e3
            rows[i].append((np.median(v), v.min(), v.max()))
    print(f"single-launch decode, d_model {cfg.D}, {cfg.E} experts top-{cfg.K}, T={T}, {cfg.layers} layers: "
          f"layer {TRACE_LAYER}, {ncta} CTAs, median of {args.runs} launches (us)")
    print(f"{'phase ends':18s} {'median CTA':>10s} {'fastest':>9s} {'slowest':>9s}")
    order = [0, 24, 25, 26, 27, 1, 2, 3, 30, 31, 4, 28, 29, 5, 23, 20, 21, 22, 6, 7, 12, 16, 13, 17, 14, 18, 15,
             19, 9, 10, 11]  # kernel order
    for i in order:
        a = np.median(np.array(rows[i]), axis=0)
        print(f"{PHASES[i]:18s} {a[0]:10.2f} {a[1]:9.2f} {a[2]:9.2f}")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
