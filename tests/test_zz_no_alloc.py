"""The allocation-free entry point mx_moe_layer_forward_static: host-side
rejections (CPU), and on the GPU the same results as mx_moe_layer_forward_ex
-- the same kernel -- on two calls in a row, with and without the options.

Collected last (file name) so that it also runs after every other test of the
session has used the library."""
import ctypes as C
import gc

import numpy as np
import pytest

import expert_ffn_gb300 as mx
import synth

OK, INVALID, UNSUP = 0, -1, -3
FAKE = 0x7F0000000000  # aligned, never dereferenced: validation fails first or T == 0


def _call(L, T, D=256, E=16, x=FAKE + 0x1000000):
    off, stride = synth.default_layout(D, 128)
    lay = mx.make_layout(D, 128, E, 2, 128, stride, off, mx.MX_BF16, 0.5)
    q = lambda r, c, b: mx.make_qlinear(FAKE, FAKE + 0x100000, FAKE + 0x200000, r, c, b)
    router, shared = q(E, D, 8), mx.Ffn(q(128, D, 4), q(128, D, 4), q(D, 128, 4))
    return L.mx_moe_layer_forward_static(x, T, C.byref(router), C.byref(shared), FAKE + 0x3000000, C.byref(lay),
                                         FAKE + 0x2000000, FAKE + 0x4000000, FAKE + 0x5000000, None, None)


def test_static_call_host_checks():
    L = mx.lib()
    assert _call(L, 0) == OK                 # nothing to do
    assert _call(L, -1) == INVALID
    assert _call(L, 1, x=0) == INVALID        # null input
    assert _call(L, 5) == UNSUP              # more tokens than the single-launch path takes
    assert _call(L, 1, D=8192) == UNSUP      # d_model above the path's limit
    assert len(L.mx_last_error_string()) > 0


CASES = [
    # cfg, residual + pre-rmsnorm
    (synth.small_config(T=2, D=320, E=24, K=3, I=192, S=128, act="bf16", seed=11), False),
    (synth.small_config(T=4, D=256, E=16, K=2, I=128, S=128, act="f32", seed=12), True),
    (synth.CONFIGS[1], True),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", range(len(CASES)), ids=["T2_bf16", "T4_f32_opts", "decode_T1_D2816"])
def test_static_matches_workspace_call(case):
    """Two static calls in a row equal the workspace call bit for bit, and
    after a first (warm-up) static call they change neither the device's free
    memory nor torch's allocator statistics: the calls themselves allocate
    nothing on the device."""
    import torch
    from tests.gpu_util import Workspace, to_dev

    cfg, opts = CASES[case]
    layer = synth.make_layer(cfg)
    dev = mx.DeviceLayer(layer, mx.MX_BF16 if cfg.act == "bf16" else mx.MX_F32)
    T, K = cfg.T, cfg.K
    x = to_dev(synth.make_x(cfg))
    res = to_dev(synth.make_x(cfg, T)[::-1].copy()) if opts else None
    s = torch.cuda.current_stream()
    ws = Workspace(mx.workspace_bytes(dev.layout, T))
    out = torch.empty_like(x)
    idx = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, K), dtype=torch.float32, device="cuda")

    def run(static: bool):
        out.fill_(0)
        idx.fill_(-1)
        w.fill_(0)
        if static:
            mx.layer_forward_static(x, T, dev, out, idx, w, stream=s, residual=res, pre_rmsnorm=opts)
        else:
            mx.layer_forward_ex(x, T, dev, out, idx, w, ws.t, ws.nbytes, stream=s, residual=res, pre_rmsnorm=opts)
        torch.cuda.synchronize()
        return out.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()

    ref = run(False)
    mx.workspace_check(ws.t, s)
    run(True)  # warm-up: the first static call on the device resolves the scratch address
    # tensors of earlier tests that only the cycle collector frees would
    # otherwise be released in the middle of the measurement
    gc.collect()
    gc.disable()
    try:
        free0 = torch.cuda.mem_get_info()[0]
        stats0 = torch.cuda.memory_stats().get("num_alloc_retries", 0), torch.cuda.memory_allocated()
        for _ in range(2):  # two calls in a row: each leaves the scratch ready for the next
            got = run(True)
            for g, r in zip(got, ref):
                assert np.array_equal(g, r)
        assert torch.cuda.mem_get_info()[0] == free0
        assert (torch.cuda.memory_stats().get("num_alloc_retries", 0), torch.cuda.memory_allocated()) == stats0
    finally:
        gc.enable()
    assert np.all(ref[1] >= 0)
