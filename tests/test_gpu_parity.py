"""GPU parity: the CUDA path (through the C-ABI) against the CPU oracle on the
same seeded inputs.

Bars: top-k indices, counts, offsets and the expert permutation bit-exact;
fp32 outputs rel-L2 <= 1e-4 and max|diff| <= 2e-2; BF16 outputs compared with
the oracle's output rounded once to BF16, rel-L2 <= 1e-3 and max|diff| /
max|oracle| <= 2e-2; routing weights rel-L2 <= 1e-4."""
from __future__ import annotations

import numpy as np
import pytest

import synth
from tests.helpers import max_abs_rel, rel_l2

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from expert_ffn_gb300 import build
    build.build()


@pytest.fixture(scope="module")
def gu():
    from tests import gpu_util
    return gpu_util


def check_out(got, ref, act):
    from tests.gpu_util import as_f32
    g, r = as_f32(got).astype(np.float64), as_f32(ref).astype(np.float64)
    assert np.all(np.isfinite(g))
    if act == "f32":
        assert rel_l2(g, r) <= 1e-4, rel_l2(g, r)
        assert np.max(np.abs(g - r)) <= 2e-2
    else:
        assert rel_l2(g, r) <= 1e-3, rel_l2(g, r)
        assert max_abs_rel(g, r) <= 2e-2, max_abs_rel(g, r)


def check_block(orc, gu, cfg, layer, x, **kw):
    dev = __import__("expert_ffn_gb300").DeviceLayer(layer, gu.act_code(cfg))
    out, idx, w = gu.run_block(dev, x, **kw)
    ref, ridx, rw = orc.block_forward(layer, x)
    assert np.array_equal(idx, ridx)
    assert rel_l2(w, rw) <= 1e-4
    check_out(out, ref, cfg.act)
    return dev, out, idx, w


# ------------------------------------------------------------- small shapes

SHAPES = [
    # T, D, E, K, I, S, act
    (4, 256, 16, 2, 128, 128, "f32"),      # the tiny workload
    (1, 256, 16, 2, 128, 128, "bf16"),
    (13, 320, 24, 3, 192, 128, "bf16"),    # ragged token tiles, odd group counts
    (64, 512, 32, 8, 128, 256, "bf16"),    # a full decode chunk
    (65, 256, 16, 4, 128, 64, "f32"),      # one past the chunk: two passes
    (40, 192, 8, 8, 64, 64, "bf16"),       # K = E: every expert gets every token
    (3, 64, 4, 1, 64, 64, "f32"),          # one group per row, K = 1
    (150, 384, 64, 6, 320, 192, "bf16"),   # several chunks, ragged tail
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"T{s[0]}_D{s[1]}_E{s[2]}_K{s[3]}_{s[6]}" for s in SHAPES])
def test_block_small_shapes(orc, gu, shape):
    T, D, E, K, I, S, act = shape
    cfg = synth.small_config(T=T, D=D, E=E, K=K, I=I, S=S, act=act, seed=T + D)
    layer = synth.make_layer(cfg)
    x = synth.make_x(cfg)
    check_block(orc, gu, cfg, layer, x)


def test_tiny_workload_route_exact(orc, gu):
    cfg = synth.CONFIGS[0]
    layer = synth.make_layer(cfg)
    x = synth.make_x(cfg)
    dev = __import__("expert_ffn_gb300").DeviceLayer(layer, gu.act_code(cfg))
    idx, w, counts, offsets, perm, logits = gu.run_route(dev, x)
    rl = orc.router_logits(layer.router, gu.as_f32(x))
    assert np.array_equal(logits, rl)          # canonical order: bit-exact
    ridx, rw = orc.topk_softmax(rl, cfg.K)
    rc, ro, rp = orc.permute(ridx, cfg.E)
    assert np.array_equal(idx, ridx) and np.array_equal(counts, rc)
    assert np.array_equal(offsets, ro) and np.array_equal(perm, rp)
    assert rel_l2(w, rw) <= 1e-4


def test_determinism_and_entry_points_agree(orc, gu):
    cfg = synth.small_config(T=24, D=512, E=32, K=4, I=128, S=128, act="bf16", seed=9)
    layer = synth.make_layer(cfg)
    x = synth.make_x(cfg)
    dev = __import__("expert_ffn_gb300").DeviceLayer(layer, gu.act_code(cfg))
    a = gu.run_block(dev, x)
    b = gu.run_block(dev, x)
    c = gu.run_block(dev, x, ex=False)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)
    for u, v in zip(a, c):
        assert np.array_equal(u, v)


def test_residual_and_prenorm_options(orc, gu):
    cfg = synth.small_config(T=5, D=256, E=16, K=2, I=128, S=128, act="bf16", seed=21)
    layer = synth.make_layer(cfg)
    x = synth.make_x(cfg)
    dev = __import__("expert_ffn_gb300").DeviceLayer(layer, gu.act_code(cfg))
    out, idx, w = gu.run_block(dev, x, residual=x, pre_norm=True, eps=1e-6)
    xn = orc.rmsnorm_bf16(x, 1e-6)
    ref, ridx, rw = orc.block_forward(layer, xn, residual=x)
    assert np.array_equal(idx, ridx)
    check_out(out, ref, "bf16")


def test_zero_tokens_writes_nothing(gu):
    import expert_ffn_gb300 as mx
    cfg = synth.small_config(T=2, act="bf16")
    dev = mx.DeviceLayer(synth.make_layer(cfg), mx.MX_BF16)
    out = torch.full((2, cfg.D), 7, dtype=torch.int16, device="cuda")
    x = torch.zeros((2, cfg.D), dtype=torch.int16, device="cuda")
    idx = torch.full((2, cfg.K), -5, dtype=torch.int32, device="cuda")
    w = torch.zeros((2, cfg.K), dtype=torch.float32, device="cuda")
    mx.layer_forward(x, 0, dev, out, idx, w)
    torch.cuda.synchronize()
    assert bool((out == 7).all()) and bool((idx == -5).all())


# ------------------------------------------------------------ full workloads

def test_skewed_decode_T64_full(orc, gu):
    cfg = synth.CONFIGS[3]
    layer = synth.make_layer(cfg)
    x = synth.make_x(cfg)
    check_block(orc, gu, cfg, layer, x)


def covering_tokens(counts, offsets, perm, K, T, tile=128):
    """Tokens that put at least one output row through every work unit of the
    grouped GEMMs: for each expert, the first slot of each 128-slot tile of its
    slot range and its last slot; the first token of every 128-token tile (the
    shared expert's units); and every token of the last, ragged, token tile."""
    tok = set(range(((T - 1) // tile) * tile, T))
    tok.update(range(0, T, tile))
    for e in range(len(counts)):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        for a in range(lo, hi, tile):
            tok.add(int(perm[a]) // K)
        if hi > lo:
            tok.add(int(perm[hi - 1]) // K)
    return np.array(sorted(tok), dtype=np.int64)


@pytest.mark.parametrize("ci", [2, 4])
def test_prefill_route_exact_and_full_outputs(orc, gu, ci):
    """Full-size prefill: every token's top-k, the counts and the permutation
    exact (the oracle routes all T tokens).  Outputs: every token of the
    T=512 workload; at T=4096 the tokens that cover every (expert, 128-slot
    tile) unit, every shared-expert token tile and the whole last token tile
    (the oracle runs on all host cores)."""
    import expert_ffn_gb300 as mx
    cfg = synth.CONFIGS[ci]
    layer = synth.make_layer(cfg)
    x = synth.make_x(cfg)
    dev = mx.DeviceLayer(layer, gu.act_code(cfg))
    out, idx, w = gu.run_block(dev, x)
    ridx_all, rw_all = orc.topk_softmax(orc.router_logits(layer.router, gu.as_f32(x)), cfg.K)
    assert np.array_equal(idx, ridx_all)
    assert rel_l2(w, rw_all) <= 1e-4
    ridx, _, counts, offsets, perm, _ = gu.run_route(dev, x)
    rc, ro, rp = orc.permute(ridx_all, cfg.E)
    assert np.array_equal(ridx, ridx_all) and np.array_equal(perm, rp)
    assert np.array_equal(counts, rc) and np.array_equal(offsets, ro)
    tok = np.arange(cfg.T) if ci == 2 else covering_tokens(rc, ro, rp, cfg.K, cfg.T)
    ref, ridx_t, _ = orc.block_forward_tokens(layer, x, tok)
    assert np.array_equal(ridx_t, ridx_all[tok])
    check_out(out[tok], ref, cfg.act)


# ------------------------------------------- routing edge cases and options

def skewed_router_layer(cfg, hot=5, n_empty=16):
    """The layer of ``cfg`` with its router rewritten so that, for activations
    >= 0, expert ``hot`` (all router bytes 255, scale 2^-11, bias 0) has the
    largest logit of every token and the ``n_empty`` experts after it (all
    bytes 0, bias -0.03) have logits below every other expert's: they receive
    no token.  The oracle's routing is checked to confirm it."""
    layer = synth.make_layer(cfg)
    r = layer.router
    empty = [(hot + 1 + j) % cfg.E for j in range(n_empty)]
    r.w[hot] = 0xFFFFFFFF
    r.s[hot] = synth.f32_to_bf16_bits(np.full(r.s.shape[1], 2.0 ** -11, np.float32))
    r.b[hot] = 0
    for e in empty:
        r.w[e] = 0
        r.b[e] = synth.f32_to_bf16_bits(np.full(r.b.shape[1], -0.03, np.float32))
    return layer, hot, empty


def nonneg_x(cfg):
    x = synth.make_x(cfg)
    return (x & np.uint16(0x7FFF)) if x.dtype == np.uint16 else np.abs(x)


EMPTY_CASES = [(3, "1"), (40, "0"), (40, "1"), (200, "1")]


@pytest.mark.parametrize("case", EMPTY_CASES, ids=["single_launch_T3", "decode_kernels_T40", "grouped_gemm_T40",
                                                   "grouped_gemm_T200"])
def test_empty_experts_and_one_expert_with_every_token(orc, gu, case, monkeypatch):
    """Sixteen of 64 experts receive no token and one expert receives every
    token (more than one 128-slot tile at T = 200): the single-launch decode
    kernel at T = 3, the multi-launch decode kernels at T = 40
    (MX_MOE_PREFILL_GEMM=0), the grouped tensor-core GEMMs at T = 40 and 200."""
    import expert_ffn_gb300 as mx
    T, gemm = case
    monkeypatch.setenv("MX_MOE_PREFILL_GEMM", gemm)
    cfg = synth.small_config(T=T, D=512, E=64, K=2, I=256, S=128, act="bf16", seed=400 + T)
    layer, hot, empty = skewed_router_layer(cfg)
    x = nonneg_x(cfg)
    ridx, _ = orc.topk_softmax(orc.router_logits(layer.router, gu.as_f32(x)), cfg.K)
    rc, _, _ = orc.permute(ridx, cfg.E)
    assert rc[hot] == T and np.all(rc[empty] == 0)
    mx.profile_enable(True)
    try:
        mx.profile_read(reset=True)
        check_block(orc, gu, cfg, layer, x)
        prof = mx.profile_read(reset=True)
    finally:
        mx.profile_enable(False)
    if T <= 4:
        assert prof["route"][1] == 0 and prof["gate_up"][1] == 1, prof   # the single launch
    else:
        assert prof["route"][1] == 1 and prof["gate_up"][1] == 1 and prof["down"][1] == 1, prof
    dev = mx.DeviceLayer(layer, mx.MX_BF16)
    _, _, counts, _, _, _ = gu.run_route(dev, x)
    assert np.array_equal(counts, rc)


PES_CASES = [(2, 1), (2, 0), (24, 0), (130, 1)]


@pytest.mark.parametrize("case", PES_CASES, ids=["single_launch_T2", "multi_launch_T2", "multi_launch_T24",
                                                 "prefill_T130"])
def test_per_expert_scale(orc, gu, case, monkeypatch):
    """A per-expert scale multiplies each selected expert's softmax weight on
    every path (router formula of the "Decode" section)."""
    T, single = case
    monkeypatch.setenv("MX_MOE_SINGLE_LAUNCH", str(single))
    cfg = synth.small_config(T=T, D=384, E=32, K=4, I=192, S=128, act="bf16", seed=500 + T)
    layer = synth.make_layer(cfg)
    layer.per_expert_scale = np.random.default_rng(T).uniform(0.5, 2.0, cfg.E).astype(np.float32)
    x = synth.make_x(cfg)
    _, _, w, = check_block(orc, gu, cfg, layer, x)[1:]
    _, rw_plain = orc.topk_softmax(orc.router_logits(layer.router, gu.as_f32(x)), cfg.K)
    assert rel_l2(w, rw_plain) > 1e-2            # the scale did change the weights


# --------------------------------- the decode path's fixed-point sums: range

def check_scaled(got, ref):
    g, r = got.astype(np.float64), ref.astype(np.float64)
    assert np.all(np.isfinite(g))
    assert rel_l2(g, r) <= 1e-4, rel_l2(g, r)
    assert max_abs_rel(g, r) <= 2e-2


@pytest.mark.parametrize("e", [-20, 20], ids=["x_times_2^-20", "x_times_2^20"])
def test_fixed_point_range_follows_input(orc, gu, e):
    """fp32 inputs scaled by 2^-20 (block outputs near 1e-10: far below the
    fixed-point unit of unscaled inputs) and by 2^20 (outputs above 2^31)
    through the single-launch decode kernel: the fp32 bars of the oracle."""
    import expert_ffn_gb300 as mx
    cfg = synth.small_config(T=4, D=256, E=16, K=2, I=128, S=128, act="f32", seed=600)
    layer = synth.make_layer(cfg)
    x = (synth.make_x(cfg) * np.float32(2.0 ** e)).astype(np.float32)
    dev = mx.DeviceLayer(layer, mx.MX_F32)
    out, idx, w = gu.run_block(dev, x)
    ref, ridx, rw = orc.block_forward(layer, x)
    assert np.array_equal(idx, ridx) and rel_l2(w, rw) <= 1e-4
    check_scaled(out, ref)
    if e > 0:
        assert np.max(np.abs(ref)) > 2.0 ** 31


def test_fixed_point_out_of_range_is_reported(orc, gu):
    """A shared down projection with scales of 2^20 drives the partial sums
    past the fixed-point range: the call reports MX_ERR_RANGE through the
    workspace check; after re-initialising the workspace an ordinary call
    matches the oracle again."""
    import expert_ffn_gb300 as mx
    cfg = synth.small_config(T=1, D=256, E=16, K=2, I=128, S=128, act="bf16", seed=601)
    layer = synth.make_layer(cfg)
    big = synth.make_layer(cfg)
    big.shared_down.s[:] = synth.f32_to_bf16_bits(np.full(big.shared_down.s.shape, 2.0 ** 20, np.float32))
    x = synth.make_x(cfg)
    ws = gu.Workspace(mx.workspace_bytes(mx.DeviceLayer(layer, mx.MX_BF16).layout, 1))
    with pytest.raises(mx.MxError) as ei:
        gu.run_block(mx.DeviceLayer(big, mx.MX_BF16), x, ws=ws)
    assert ei.value.status == -7                 # MX_ERR_RANGE
    mx.workspace_init(ws.t, ws.nbytes)
    out, idx, w = gu.run_block(mx.DeviceLayer(layer, mx.MX_BF16), x, ws=ws)
    ref, ridx, rw = orc.block_forward(layer, x)
    assert np.array_equal(idx, ridx)
    check_out(out, ref, "bf16")


def test_decode_stack_30_layers(orc, gu):
    """Single-token decode through the 30-layer stack (RMSNorm -> block ->
    residual).

    Per layer on identical inputs: layer l of the GPU path is fed the oracle's
    own output of layer l-1 (inputs flow from the oracle to the GPU, never
    back); top-k exact, routing weights rel-L2 <= 1e-4, output within the BF16
    bars.  Free-running through the stack entry point from the same input:
    top-k exact in every layer, and the stack entry point equal bit for bit to
    the chain of single-layer calls.  Free-running, the two sides' residual
    streams may round differently to BF16 in a few elements per layer, and the
    difference grows with depth; the final output is held to the BF16 bars and
    the routing weights to 5e-3."""
    import expert_ffn_gb300 as mx
    cfg = synth.CONFIGS[1]
    layers = [synth.make_layer(cfg, l) for l in range(cfg.layers)]
    x = synth.make_x(cfg)
    devs = [mx.DeviceLayer(l, mx.MX_BF16) for l in layers]
    stack = mx.Stack(devs)
    T, K, n = cfg.T, cfg.K, cfg.layers
    xs_ref, idx_ref, w_ref = orc.stack_forward(layers, x, 1e-6)

    ws1 = gu.Workspace(mx.workspace_bytes(devs[0].layout, T))
    for l in range(n):
        xin = x if l == 0 else xs_ref[l - 1]
        out, li, lw = gu.run_block(devs[l], xin, residual=xin, pre_norm=True, eps=1e-6, ws=ws1)
        assert np.array_equal(li, idx_ref[l]), l
        assert rel_l2(lw, w_ref[l]) <= 1e-4, (l, rel_l2(lw, w_ref[l]))
        check_out(out, xs_ref[l], "bf16")

    xd = gu.to_dev(x)
    idx = torch.full((n, T, K), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((n, T, K), dtype=torch.float32, device="cuda")
    ws = gu.Workspace(mx.stack_workspace_bytes(devs[0].layout, T))
    mx.stack_forward(xd, T, stack, idx, w, ws.t, ws.nbytes, rms_eps=1e-6, stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    idx, w = idx.cpu().numpy(), w.cpu().numpy()
    x_final = gu.to_host(xd, np.uint16)
    cur = x
    for l in range(n):
        out, li, lw = gu.run_block(devs[l], cur, residual=cur, pre_norm=True, eps=1e-6, ws=ws1)
        assert np.array_equal(li, idx[l]) and np.array_equal(lw, w[l])
        cur = out
    assert np.array_equal(x_final, cur)
    assert np.array_equal(idx, idx_ref)
    assert rel_l2(w, w_ref) <= 5e-3
    check_out(x_final, xs_ref[-1], "bf16")


# ------------------------------------------- the two decode paths, T <= 4

PATH_SHAPES = [
    # T, D, E, K, I, S, act
    (1, 512, 32, 4, 128, 192, "bf16"),
    (2, 320, 24, 3, 192, 128, "bf16"),
    (4, 256, 16, 2, 128, 128, "f32"),
    (3, 64, 4, 1, 64, 64, "f32"),
    (4, 768, 64, 8, 256, 128, "bf16"),     # 32 slots: many active experts per layer
]


@pytest.mark.parametrize("single", [1, 0], ids=["single_launch", "multi_launch"])
@pytest.mark.parametrize("shape", PATH_SHAPES, ids=[f"T{s[0]}_D{s[1]}_E{s[2]}_K{s[3]}_{s[6]}" for s in PATH_SHAPES])
def test_decode_paths(orc, gu, shape, single, monkeypatch):
    """T <= 4 runs as one persistent launch by default; MX_MOE_SINGLE_LAUNCH=0
    selects the router / gate-up / down launches.  Both against the oracle;
    the stage profiler tells which path ran (the single launch records one
    launch under the gate/up stage and none under routing)."""
    import expert_ffn_gb300 as mx
    monkeypatch.setenv("MX_MOE_SINGLE_LAUNCH", str(single))
    T, D, E, K, I, S, act = shape
    cfg = synth.small_config(T=T, D=D, E=E, K=K, I=I, S=S, act=act, seed=3 * T + D)
    layer = synth.make_layer(cfg)
    x = synth.make_x(cfg)
    mx.profile_enable(True)
    try:
        mx.profile_read(reset=True)
        dev, _, _, _ = check_block(orc, gu, cfg, layer, x)
        prof = mx.profile_read(reset=True)
    finally:
        mx.profile_enable(False)
    if single:
        assert prof["route"][1] == 0 and prof["gate_up"][1] == 1, prof
    else:
        assert prof["route"][1] == 1, prof
    # a second call on the same workspace (counters must have been reset)
    ws = gu.Workspace(mx.workspace_bytes(dev.layout, T))
    a = gu.run_block(dev, x, ws=ws)
    b = gu.run_block(dev, x, ws=ws)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_decode_stack_paths_agree(orc, gu, monkeypatch):
    """A short stack at T = 2 through both paths: same top-k in every layer,
    outputs within the BF16 bars of the oracle's stack."""
    import expert_ffn_gb300 as mx
    cfg = synth.small_config(T=2, D=512, E=32, K=4, I=128, S=192, act="bf16", seed=77)
    n = 5
    layers = [synth.make_layer(cfg, l) for l in range(n)]
    x = synth.make_x(cfg)
    devs = [mx.DeviceLayer(l, mx.MX_BF16) for l in layers]
    stack = mx.Stack(devs)
    xs_ref, idx_ref, w_ref = orc.stack_forward(layers, x, 1e-6)
    for single in (1, 0):
        monkeypatch.setenv("MX_MOE_SINGLE_LAUNCH", str(single))
        xd = gu.to_dev(x)
        idx = torch.full((n, cfg.T, cfg.K), -1, dtype=torch.int32, device="cuda")
        w = torch.zeros((n, cfg.T, cfg.K), dtype=torch.float32, device="cuda")
        ws = gu.Workspace(mx.stack_workspace_bytes(devs[0].layout, cfg.T))
        mx.stack_forward(xd, cfg.T, stack, idx, w, ws.t, ws.nbytes, rms_eps=1e-6,
                         stream=torch.cuda.current_stream())
        mx.workspace_check(ws.t, torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), idx_ref), single
        assert rel_l2(w.cpu().numpy(), w_ref) <= 5e-3
        check_out(gu.to_host(xd, np.uint16), xs_ref[-1], "bf16")


# --------------------------------------------- prefill: tensor-core GEMMs

PREFILL_SHAPES = [
    # T, D, E, K, I, S
    (5, 256, 16, 4, 128, 64),        # one past the single-launch range
    (16, 512, 32, 8, 192, 128),      # a batch of 16: many experts with one token
    (64, 768, 64, 8, 128, 256),      # a full decode batch
    (65, 256, 16, 4, 128, 64),
    (200, 320, 8, 3, 192, 320),      # D, I, S not multiples of 128; T ragged; experts with >128 slots
    (300, 512, 4, 2, 704, 128),      # few experts: several token tiles each
    (129, 1024, 64, 8, 256, 384),
    (700, 256, 4, 2, 128, 64),       # ~350 slots per expert: three token tiles; above the per-group router's 512
]


@pytest.mark.parametrize("shape", PREFILL_SHAPES, ids=[f"T{s[0]}_D{s[1]}_E{s[2]}_K{s[3]}_I{s[4]}_S{s[5]}"
                                                       for s in PREFILL_SHAPES])
def test_prefill_gemm_shapes(orc, gu, shape, monkeypatch):
    """BF16 inputs with T > 4 run the grouped tensor-core GEMMs (stage
    profiler: one routing launch, the GEMM sequence under gate/up); against
    the oracle, and against the decode kernels on the same inputs."""
    import expert_ffn_gb300 as mx
    T, D, E, K, I, S = shape
    cfg = synth.small_config(T=T, D=D, E=E, K=K, I=I, S=S, act="bf16", seed=T + 7 * D)
    layer = synth.make_layer(cfg)
    x = synth.make_x(cfg)
    mx.profile_enable(True)
    try:
        mx.profile_read(reset=True)
        dev, out, idx, w = check_block(orc, gu, cfg, layer, x)
        prof = mx.profile_read(reset=True)
    finally:
        mx.profile_enable(False)
    assert prof["route"][1] == 1 and prof["gate_up"][1] == 1 and prof["down"][1] == 1, prof
    monkeypatch.setenv("MX_MOE_PREFILL_GEMM", "0")
    out2, idx2, w2 = gu.run_block(dev, x)
    assert np.array_equal(idx, idx2)
    check_out(out, out2, "bf16")


def test_prefill_residual_and_prenorm(orc, gu):
    cfg = synth.small_config(T=96, D=512, E=16, K=4, I=256, S=128, act="bf16", seed=31)
    layer = synth.make_layer(cfg)
    x = synth.make_x(cfg)
    dev = __import__("expert_ffn_gb300").DeviceLayer(layer, gu.act_code(cfg))
    out, idx, w = gu.run_block(dev, x, residual=x, pre_norm=True, eps=1e-6)
    xn = orc.rmsnorm_bf16(x, 1e-6)
    ref, ridx, rw = orc.block_forward(layer, xn, residual=x)
    assert np.array_equal(idx, ridx)
    check_out(out, ref, "bf16")


# ------------------------------------------- failure detection (no GPU fault)

def test_device_wait_runs_out_and_is_reported(orc, gu, monkeypatch):
    """A CTA held back (on the host's say-so) from the first logit exchange of
    the single-launch decode kernel: every other CTA's bounded wait runs out
    after 1 ms, the kernel returns, and the workspace check reports
    MX_ERR_DEVICE_TIMEOUT (the failed eager-fill case of the "Decode" section:
    the step is abandoned rather than emitting a result).  After the workspace
    is re-initialised, an ordinary call matches the oracle again."""
    import expert_ffn_gb300 as mx
    cfg = synth.CONFIGS[0]
    layer = synth.make_layer(cfg)
    x = synth.make_x(cfg)
    dev = mx.DeviceLayer(layer, mx.MX_F32)
    ws = gu.Workspace(mx.workspace_bytes(dev.layout, cfg.T))
    monkeypatch.setenv("MX_MOE_WAIT_LIMIT_US", "1000")
    monkeypatch.setenv("MX_MOE_HOLD_CTA", "3")
    with pytest.raises(mx.MxError) as ei:
        gu.run_block(dev, x, ws=ws)
    assert ei.value.status == -6                 # MX_ERR_DEVICE_TIMEOUT
    monkeypatch.delenv("MX_MOE_WAIT_LIMIT_US")
    monkeypatch.delenv("MX_MOE_HOLD_CTA")
    mx.workspace_init(ws.t, ws.nbytes)
    out, idx, w = gu.run_block(dev, x, ws=ws)
    ref, ridx, rw = orc.block_forward(layer, x)
    assert np.array_equal(idx, ridx)
    check_out(out, ref, "f32")
