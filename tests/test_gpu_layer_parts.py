"""GPU parity of the layer's optional parts (layout version 2) against the CPU
oracle, on every path that implements them:

  - the resident-set expert table ("Mference System design", "Load and
    ownership"): a permuted or reduced blob with its table gives the same
    outputs, bit for bit, as the plain blob on the GPU, and the oracle's; an
    absent selected expert is reported (MX_ERR_NOT_RESIDENT);
  - the router's input scale x * router_scale / sqrt(D) (router formula of
    the "Decode" section): top-k exact, and the routing does change;
  - the post-FFN norm of the combined output (cb2 row of "Decode");
  - the gated shared expert sigmoid(g . x).

Paths: the single-launch decode kernel (T <= 4, both dtypes), the grouped
tensor-core GEMMs (BF16, T > 4); the table also on the multi-launch decode
kernels.  Bars as in test_gpu_parity."""
from __future__ import annotations

import numpy as np
import pytest

import synth
from synth import f32_to_bf16_bits
from tests.helpers import rel_l2
from tests.test_gpu_parity import check_out

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


def _layer(T, act, seed, D=384, E=32, K=4, I=192, S=128):
    cfg = synth.small_config(T=T, D=D, E=E, K=K, I=I, S=S, act=act, seed=seed)
    return cfg, synth.make_layer(cfg), synth.make_x(cfg)


def _with_blob(layer, order):
    """Copy of `layer` whose blob holds the records of experts `order`, in
    that order, with the matching expert -> record table (-1 elsewhere)."""
    import dataclasses
    st = layer.stride
    blob = np.concatenate([layer.blob[e * st:(e + 1) * st] for e in order])
    slot = np.full(layer.E, -1, dtype=np.int16)
    for r, e in enumerate(order):
        slot[e] = r
    return dataclasses.replace(layer, blob=blob, expert_slot=slot, n_slots=len(order))


def _run(gu, layer, x, act, **kw):
    import expert_ffn_gb300 as mx
    return gu.run_block(mx.DeviceLayer(layer, gu.act_code(act)), x, **kw)


def _check(orc, gu, cfg, layer, x, **kw):
    out, idx, w = _run(gu, layer, x, cfg.act, **kw)
    ref, ridx, rw = orc.block_forward(layer, x)
    assert np.array_equal(idx, ridx)
    assert rel_l2(w, rw) <= 1e-4, rel_l2(w, rw)
    check_out(out, ref, cfg.act)
    return out, idx, w, ref


# (T, act, MX_MOE_SINGLE_LAUNCH, MX_MOE_PREFILL_GEMM): which kernels run
TABLE_PATHS = [
    (3, "bf16", "1", "1"),    # single-launch decode kernel
    (2, "f32", "1", "1"),
    (3, "bf16", "0", "1"),    # multi-launch decode kernels
    (24, "f32", "1", "1"),
    (40, "bf16", "1", "0"),
    (40, "bf16", "1", "1"),   # grouped GEMMs
    (130, "bf16", "1", "1"),
]
TABLE_IDS = ["single_bf16_T3", "single_f32_T2", "multi_bf16_T3", "multi_f32_T24", "multi_bf16_T40",
             "gemm_T40", "gemm_T130"]


@pytest.mark.parametrize("case", TABLE_PATHS, ids=TABLE_IDS)
def test_expert_table_permuted_and_resident_subset(orc, gu, case, monkeypatch):
    T, act, single, gemm = case
    monkeypatch.setenv("MX_MOE_SINGLE_LAUNCH", single)
    monkeypatch.setenv("MX_MOE_PREFILL_GEMM", gemm)
    cfg, layer, x = _layer(T, act, seed=700 + T)
    plain, pidx, pw = _run(gu, layer, x, act)
    order = [int(e) for e in np.random.default_rng(T).permutation(layer.E)]
    perm = _with_blob(layer, order)
    out, idx, w, _ = _check(orc, gu, cfg, perm, x)
    # only the record addresses change: the GPU result is the plain one, bit for bit
    assert np.array_equal(out, plain) and np.array_equal(idx, pidx) and np.array_equal(w, pw)
    chosen = sorted(set(int(e) for e in pidx.ravel()))
    sub = _with_blob(layer, chosen[::-1])
    out2, idx2, w2, _ = _check(orc, gu, cfg, sub, x)
    assert np.array_equal(out2, plain) and np.array_equal(idx2, pidx) and np.array_equal(w2, pw)


@pytest.mark.parametrize("case", [TABLE_PATHS[0], TABLE_PATHS[2], TABLE_PATHS[6]],
                         ids=["single_T3", "multi_T3", "gemm_T130"])
def test_absent_expert_is_reported(orc, gu, case, monkeypatch):
    """A table without a record for one selected expert: the workspace check
    returns MX_ERR_NOT_RESIDENT (the oracle refuses the same layer); once the
    workspace is re-initialised an ordinary call matches the oracle."""
    import expert_ffn_gb300 as mx
    T, act, single, gemm = case
    monkeypatch.setenv("MX_MOE_SINGLE_LAUNCH", single)
    monkeypatch.setenv("MX_MOE_PREFILL_GEMM", gemm)
    cfg, layer, x = _layer(T, act, seed=720 + T)
    _, pidx, _ = _run(gu, layer, x, act)
    chosen = sorted(set(int(e) for e in pidx.ravel()))
    missing = _with_blob(layer, chosen[1:])
    with pytest.raises(orc.ExpertNotResident):
        orc.block_forward(missing, x)
    dev = mx.DeviceLayer(missing, gu.act_code(act))
    ws = gu.Workspace(mx.workspace_bytes(dev.layout, T))
    with pytest.raises(mx.MxError) as ei:
        gu.run_block(dev, x, ws=ws)
    assert ei.value.status == -8               # MX_ERR_NOT_RESIDENT
    mx.workspace_init(ws.t, ws.nbytes)
    _check(orc, gu, cfg, layer, x, ws=ws)


def _router_scale(D, seed):
    rng = np.random.default_rng(seed)
    return f32_to_bf16_bits((np.sqrt(D) * rng.uniform(0.25, 1.75, D)).astype(np.float32))


def _post_norm(D, seed):
    return f32_to_bf16_bits(np.random.default_rng(seed).uniform(0.5, 1.5, D).astype(np.float32))


def _gate(D, seed, spread=4.0):
    rng = np.random.default_rng(seed)
    return f32_to_bf16_bits((rng.uniform(-spread, spread, D) / np.sqrt(D)).astype(np.float32))


PART_PATHS = [(1, "bf16"), (4, "bf16"), (3, "f32"), (40, "bf16"), (130, "bf16")]
PART_IDS = ["single_bf16_T1", "single_bf16_T4", "single_f32_T3", "gemm_T40", "gemm_T130"]


@pytest.mark.parametrize("case", PART_PATHS, ids=PART_IDS)
def test_router_scale(orc, gu, case):
    T, act = case
    cfg, layer, x = _layer(T, act, seed=740 + T)
    _, idx0, _ = orc.block_forward(layer, x)
    layer.router_scale = _router_scale(cfg.D, T)
    _, idx, _, _ = _check(orc, gu, cfg, layer, x)
    if T >= 4:
        assert not np.array_equal(idx, idx0)   # the scale did change the routing


@pytest.mark.parametrize("case", PART_PATHS, ids=PART_IDS)
def test_post_norm(orc, gu, case):
    T, act = case
    cfg, layer, x = _layer(T, act, seed=760 + T)
    layer.post_norm, layer.post_eps = _post_norm(cfg.D, T), 1e-5
    _, _, _, ref = _check(orc, gu, cfg, layer, x)
    plain, _, _ = orc.block_forward(synth.make_layer(cfg), x)
    assert rel_l2(gu.as_f32(ref), gu.as_f32(plain)) > 1e-2   # the norm did change the output


@pytest.mark.parametrize("case", PART_PATHS, ids=PART_IDS)
def test_gated_shared_expert(orc, gu, case):
    T, act = case
    cfg, layer, x = _layer(T, act, seed=780 + T)
    layer.shared_expert_gate = _gate(cfg.D, T)
    _check(orc, gu, cfg, layer, x)


@pytest.mark.parametrize("case", PART_PATHS, ids=PART_IDS)
def test_all_parts_with_residual(orc, gu, case):
    """Table, router scale, post-norm and gate together, with a residual."""
    T, act = case
    cfg, layer, x = _layer(T, act, seed=800 + T)
    order = [int(e) for e in np.random.default_rng(T + 1).permutation(layer.E)]
    layer = _with_blob(layer, order)
    layer.router_scale = _router_scale(cfg.D, T + 1)
    layer.post_norm, layer.post_eps = _post_norm(cfg.D, T + 1), 1e-6
    layer.shared_expert_gate = _gate(cfg.D, T + 1)
    res = synth.make_x(synth.small_config(T=T, D=cfg.D, E=cfg.E, K=cfg.K, I=cfg.I, S=cfg.S, act=act, seed=9))
    out, idx, w = _run(gu, layer, x, act, residual=res)
    ref, ridx, rw = orc.block_forward(layer, x, residual=res)
    assert np.array_equal(idx, ridx) and rel_l2(w, rw) <= 1e-4
    check_out(out, ref, act)


def test_decode_stack_with_parts(orc, gu):
    """Four layers, each with its own table, router scale, post-norm and gate,
    through the stack entry point (one launch for all layers): equal bit for
    bit to the chain of single-layer calls, and layer by layer within the bars
    of the oracle fed the same inputs."""
    import expert_ffn_gb300 as mx
    n, T = 4, 1
    cfg = synth.small_config(T=T, D=512, E=32, K=4, I=256, S=256, act="bf16", seed=830)
    layers = []
    for l in range(n):
        lay = synth.make_layer(cfg, l)
        lay = _with_blob(lay, [int(e) for e in np.random.default_rng(l).permutation(lay.E)])
        lay.router_scale = _router_scale(cfg.D, 10 + l)
        lay.post_norm, lay.post_eps = _post_norm(cfg.D, 20 + l), 1e-6
        lay.shared_expert_gate = _gate(cfg.D, 30 + l)
        layers.append(lay)
    x = synth.make_x(cfg)
    devs = [mx.DeviceLayer(l, mx.MX_BF16) for l in layers]
    xs_ref, idx_ref, w_ref = orc.stack_forward(layers, x, 1e-6)
    ws1 = gu.Workspace(mx.workspace_bytes(devs[0].layout, T))
    for l in range(n):
        xin = x if l == 0 else xs_ref[l - 1]
        out, li, lw = gu.run_block(devs[l], xin, residual=xin, pre_norm=True, eps=1e-6, ws=ws1)
        assert np.array_equal(li, idx_ref[l]), l
        assert rel_l2(lw, w_ref[l]) <= 1e-4
        check_out(out, xs_ref[l], "bf16")
    xd = gu.to_dev(x)
    idx = torch.full((n, T, cfg.K), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((n, T, cfg.K), dtype=torch.float32, device="cuda")
    ws = gu.Workspace(mx.stack_workspace_bytes(devs[0].layout, T))
    mx.stack_forward(xd, T, mx.Stack(devs), idx, w, ws.t, ws.nbytes, rms_eps=1e-6,
                     stream=torch.cuda.current_stream())
    mx.workspace_check(ws.t, torch.cuda.current_stream())
    torch.cuda.synchronize()
    cur = x
    for l in range(n):
        out, li, lw = gu.run_block(devs[l], cur, residual=cur, pre_norm=True, eps=1e-6, ws=ws1)
        assert np.array_equal(li, idx.cpu().numpy()[l]) and np.array_equal(lw, w.cpu().numpy()[l])
        cur = out
    assert np.array_equal(gu.to_host(xd, np.uint16), cur)


def test_decode_stack_T3_with_parts(orc, gu):
    """Three tokens through a 3-layer stack whose layers carry every optional
    part: the stack entry point equals the chain of single-layer calls bit for
    bit, every layer's top-k equals the oracle's, and the final output is
    within the BF16 bars of the oracle's stack."""
    import expert_ffn_gb300 as mx
    n, T = 3, 3
    cfg = synth.small_config(T=T, D=384, E=32, K=4, I=192, S=128, act="bf16", seed=840)
    layers = []
    for l in range(n):
        lay = synth.make_layer(cfg, l)
        lay = _with_blob(lay, [int(e) for e in np.random.default_rng(40 + l).permutation(lay.E)])
        lay.router_scale = _router_scale(cfg.D, 50 + l)
        lay.post_norm, lay.post_eps = _post_norm(cfg.D, 60 + l), 1e-6
        lay.shared_expert_gate = _gate(cfg.D, 70 + l)
        layers.append(lay)
    x = synth.make_x(cfg)
    devs = [mx.DeviceLayer(l, mx.MX_BF16) for l in layers]
    xs_ref, idx_ref, w_ref = orc.stack_forward(layers, x, 1e-6)
    xd = gu.to_dev(x)
    idx = torch.full((n, T, cfg.K), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((n, T, cfg.K), dtype=torch.float32, device="cuda")
    ws = gu.Workspace(mx.stack_workspace_bytes(devs[0].layout, T))
    mx.stack_forward(xd, T, mx.Stack(devs), idx, w, ws.t, ws.nbytes, rms_eps=1e-6,
                     stream=torch.cuda.current_stream())
    mx.workspace_check(ws.t, torch.cuda.current_stream())
    torch.cuda.synchronize()
    ws1 = gu.Workspace(mx.workspace_bytes(devs[0].layout, T))
    cur = x
    for l in range(n):
        out, li, lw = gu.run_block(devs[l], cur, residual=cur, pre_norm=True, eps=1e-6, ws=ws1)
        assert np.array_equal(li, idx.cpu().numpy()[l]) and np.array_equal(lw, w.cpu().numpy()[l])
        cur = out
    assert np.array_equal(gu.to_host(xd, np.uint16), cur)
    assert np.array_equal(idx.cpu().numpy(), idx_ref)
    assert rel_l2(w.cpu().numpy(), w_ref) <= 5e-3
    check_out(cur, xs_ref[-1], "bf16")
