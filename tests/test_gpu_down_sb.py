"""The packed down-projection scale / bias table (layout version 3, down_sb):
the device table equals a host gather of the blob's BF16 values in the
documented column-major order (records, then the shared expert), with and
without a resident-set table; and the single-launch decode path gives the same
bits with the table as with its strided gathers, equal to the oracle."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest

import synth
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


def host_table(layer, n_rec: int) -> np.ndarray:
    """(scale | bias << 16) of down row d, group g: records r < n_rec at
    (r * GI + g) * D + d, then the shared expert's group g at n_rec * GI * D +
    g * D + d."""
    D, GI, GS = layer.D, layer.I // 64, layer.S // 64
    _, so, bo = layer.offsets["down"]
    parts = []
    for r in range(n_rec):
        rec = layer.blob[r * layer.stride:(r + 1) * layer.stride]
        s = rec[so:so + D * GI * 2].view(np.uint16).reshape(D, GI).astype(np.uint32)
        b = rec[bo:bo + D * GI * 2].view(np.uint16).reshape(D, GI).astype(np.uint32)
        parts.append((s | (b << 16)).T.reshape(-1))
    s = layer.shared_down.s.reshape(D, GS).astype(np.uint32)
    b = layer.shared_down.b.reshape(D, GS).astype(np.uint32)
    parts.append((s | (b << 16)).T.reshape(-1))
    return np.concatenate(parts)


def _resident(layer, order):
    st = layer.stride
    blob = np.concatenate([layer.blob[e * st:(e + 1) * st] for e in order])
    slot = np.full(layer.E, -1, dtype=np.int16)
    for r, e in enumerate(order):
        slot[e] = r
    return dataclasses.replace(layer, blob=blob, expert_slot=slot, n_slots=len(order))


@pytest.mark.parametrize("resident", [False, True], ids=["all_records", "resident_set"])
def test_packed_table_is_the_blob_gathered(resident):
    import expert_ffn_gb300 as mx
    cfg = synth.small_config(T=1, D=320, E=24, K=3, I=192, S=192, act="bf16", seed=41)
    layer = synth.make_layer(cfg)
    n_rec = cfg.E
    if resident:
        order = [5, 0, 17, 3, 22, 9, 11]
        layer, n_rec = _resident(layer, order), len(order)
    dev = mx.DeviceLayer(layer, mx.MX_BF16)
    assert dev.down_sb is not None and dev.layout.down_sb == dev.down_sb.data_ptr()
    assert dev.down_sb.numel() == mx.down_sb_bytes(dev.layout)
    got = dev.down_sb.cpu().numpy().view(np.uint32)
    assert np.array_equal(got, host_table(layer, n_rec))


CASES = [
    # D, E, K, I, S, pre-norm + residual
    (2816, 128, 8, 704, 2112, True),       # the decode workload's shapes, one layer
    (320, 24, 3, 192, 128, False),        # odd group counts
    (256, 16, 2, 128, 64, True),          # one shared group
]


@pytest.mark.parametrize("case", range(len(CASES)), ids=[f"D{c[0]}_E{c[1]}_K{c[2]}" for c in CASES])
def test_decode_same_bits_with_and_without_table(orc, gu, case):
    """One BF16 token: the kernel variant that copies the packed words and the
    one that gathers them agree bit for bit (the words are the same values),
    and both match the oracle."""
    import expert_ffn_gb300 as mx
    D, E, K, I, S, opts = CASES[case]
    cfg = synth.small_config(T=1, D=D, E=E, K=K, I=I, S=S, act="bf16", seed=50 + case)
    layer = synth.make_layer(cfg)
    x = synth.make_x(cfg)
    res = synth.make_x(cfg, 1) if opts else None
    runs = []
    for pack in (True, False):
        dev = mx.DeviceLayer(layer, mx.MX_BF16, pack_down_sb=pack)
        assert (dev.layout.down_sb is not None) == pack
        runs.append(gu.run_block(dev, x, residual=res, pre_norm=opts))
    for a, b in zip(*runs):
        assert np.array_equal(a, b)
    xin = orc.rmsnorm_bf16(x) if opts else x
    ref, ridx, rw = orc.block_forward(layer, xin, residual=res)
    out, idx, _ = runs[0]
    assert np.array_equal(idx, ridx)
    check_out(out, ref, "bf16")


def test_stack_with_and_without_tables(gu):
    """A 3-layer single-token stack: tables on every layer, on none, or on
    some (then the launch takes the gathering variant) give the same bits."""
    import expert_ffn_gb300 as mx
    cfg = synth.small_config(T=1, D=384, E=32, K=4, I=192, S=128, act="bf16", seed=61)
    layers = [synth.make_layer(cfg, l) for l in range(3)]
    x0 = synth.make_x(cfg)
    outs = []
    for packs in ((True, True, True), (False, False, False), (True, False, True)):
        devs = [mx.DeviceLayer(L, mx.MX_BF16, pack_down_sb=p) for L, p in zip(layers, packs)]
        stack = mx.Stack(devs)
        nbytes = mx.stack_workspace_bytes(devs[0].layout, 1)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        mx.workspace_init(ws, nbytes)
        x_io = gu.to_dev(x0)
        idx = torch.zeros((3, 1, cfg.K), dtype=torch.int32, device="cuda")
        w = torch.zeros((3, 1, cfg.K), dtype=torch.float32, device="cuda")
        mx.stack_forward(x_io, 1, stack, idx, w, ws, nbytes, rms_eps=1e-6)
        mx.workspace_check(ws)
        torch.cuda.synchronize()
        outs.append((x_io.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()))
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert np.array_equal(a, b)
