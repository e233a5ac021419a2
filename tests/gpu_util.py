"""Helpers of the GPU tests: move synthetic inputs to the device, call the
C-ABI through the binding, bring results back.  Imports torch lazily."""
from __future__ import annotations

import numpy as np

import expert_ffn_gb300 as mx
from synth import bf16_bits_to_f32


def act_code(cfg_or_act) -> int:
    act = cfg_or_act if isinstance(cfg_or_act, str) else cfg_or_act.act
    return mx.MX_BF16 if act == "bf16" else mx.MX_F32


def to_dev(a: np.ndarray):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host(t, like_dtype) -> np.ndarray:
    a = t.cpu().numpy()
    return a.view(np.uint16) if like_dtype == np.uint16 else a


def as_f32(a: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(a) if a.dtype == np.uint16 else a.astype(np.float32)


class Workspace:
    def __init__(self, nbytes: int):
        import torch
        self.nbytes = int(nbytes)
        self.t = torch.empty(max(self.nbytes, 256), dtype=torch.uint8, device="cuda")
        mx.workspace_init(self.t, self.nbytes)


def run_block(dev: mx.DeviceLayer, x: np.ndarray, residual: np.ndarray | None = None, pre_norm: bool = False,
              eps: float = 1e-6, ex: bool = True, ws: Workspace | None = None):
    """Run the block on the GPU; returns (out, topk_idx, topk_w) as numpy."""
    import torch
    T = x.shape[0]
    K = dev.layout.top_k
    xd = to_dev(x)
    out = torch.empty_like(xd)
    idx = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, K), dtype=torch.float32, device="cuda")
    if ex:
        ws = ws or Workspace(mx.workspace_bytes(dev.layout, T))
        rd = to_dev(residual) if residual is not None else None
        mx.layer_forward_ex(xd, T, dev, out, idx, w, ws.t, ws.nbytes, stream=torch.cuda.current_stream(),
                            residual=rd, pre_rmsnorm=pre_norm, rms_eps=eps)
        mx.workspace_check(ws.t, torch.cuda.current_stream())
    else:
        assert residual is None and not pre_norm
        mx.layer_forward(xd, T, dev, out, idx, w)
    torch.cuda.synchronize()
    return to_host(out, x.dtype), idx.cpu().numpy(), w.cpu().numpy()


def run_route(dev: mx.DeviceLayer, x: np.ndarray, pre_norm: bool = False, eps: float = 1e-6):
    import torch
    T = x.shape[0]
    K, E = dev.layout.top_k, dev.layout.n_experts
    xd = to_dev(x)
    idx = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, K), dtype=torch.float32, device="cuda")
    counts = torch.zeros(E, dtype=torch.int32, device="cuda")
    offsets = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.zeros(T * K, dtype=torch.int32, device="cuda")
    logits = torch.zeros((T, E), dtype=torch.float32, device="cuda")
    ws = Workspace(mx.workspace_bytes(dev.layout, T))
    mx.route(xd, T, dev, idx, w, counts, offsets, perm, ws.t, ws.nbytes, logits=logits,
             stream=torch.cuda.current_stream(), pre_rmsnorm=pre_norm, rms_eps=eps)
    torch.cuda.synchronize()
    return (idx.cpu().numpy(), w.cpu().numpy(), counts.cpu().numpy(), offsets.cpu().numpy(), perm.cpu().numpy(),
            logits.cpu().numpy())
