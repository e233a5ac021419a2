"""Python binding of ``libmx_moe.so`` -- the GB300 routed-MoE FFN block.

Argument marshalling only: every step of the block runs in the library's CUDA
kernels.  The library must have been built (``expert_ffn_gb300.build.build()``
or ``__graft_entry__.build()``); if it is missing, loading raises -- there is
no fallback path.  PyTorch provides device memory and streams.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

from .build import LIB as LIB_PATH

__all__ = ["MxError", "lib", "QLinear", "Ffn", "Sub", "Layout", "Options", "LAYOUT_MAGIC", "LAYOUT_VERSION",
           "MX_F32", "MX_BF16", "DeviceLayer", "layer_forward", "layer_forward_ex", "route", "stack_forward",
           "workspace_bytes", "stack_workspace_bytes", "workspace_init", "layer_forward_static", "EXPORTED",
           "down_sb_bytes", "pack_down_sb"]

LAYOUT_MAGIC = 0x4D584D45
LAYOUT_VERSION = 3
MX_F32, MX_BF16 = 0, 1

# Every symbol include/mx_moe.h declares.
EXPORTED = ("mx_moe_layer_forward", "mx_moe_layer_forward_ex", "mx_moe_workspace_bytes", "mx_moe_workspace_init",
            "mx_moe_route", "mx_moe_stack_forward", "mx_moe_stack_workspace_bytes", "mx_status_string",
            "mx_last_error_string", "mx_version", "mx_moe_profile_enable", "mx_moe_profile_read",
            "mx_moe_workspace_check", "mx_moe_layer_forward_static", "mx_moe_down_sb_bytes", "mx_moe_pack_down_sb")


class MxError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{status}: {msg}")
        self.status = status


class QLinear(C.Structure):
    _fields_ = [("w", C.c_void_p), ("scales", C.c_void_p), ("biases", C.c_void_p),
                ("rows", C.c_int32), ("cols", C.c_int32), ("bits", C.c_int32)]


class Ffn(C.Structure):
    _fields_ = [("gate", QLinear), ("up", QLinear), ("down", QLinear)]


class Sub(C.Structure):
    _fields_ = [("w", C.c_uint64), ("s", C.c_uint64), ("b", C.c_uint64)]


class Layout(C.Structure):
    _fields_ = [("magic", C.c_uint32), ("version", C.c_uint32), ("d_model", C.c_int32), ("d_expert", C.c_int32),
                ("n_experts", C.c_int32), ("top_k", C.c_int32), ("d_shared", C.c_int32), ("group", C.c_int32),
                ("bits", C.c_int32), ("record_stride", C.c_uint64), ("gate", Sub), ("up", Sub), ("down", Sub),
                ("act_dtype", C.c_int32), ("layer_scalar", C.c_float), ("per_expert_scale", C.c_void_p),
                # version 2: optional parts of the layer (NULL = absent)
                ("expert_slot", C.c_void_p), ("n_slots", C.c_int32), ("router_scale", C.c_void_p),
                ("post_norm", C.c_void_p), ("post_eps", C.c_float), ("shared_expert_gate", C.c_void_p),
                # version 3: the packed down-projection scale / bias words (NULL = absent)
                ("down_sb", C.c_void_p)]


class Options(C.Structure):
    _fields_ = [("residual", C.c_void_p), ("pre_rmsnorm", C.c_int32), ("rms_eps", C.c_float)]


_lock = threading.Lock()
_lib = None


def lib():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: build it with expert_ffn_gb300.build.build()")
            L = C.CDLL(LIB_PATH)
            P, I32, SZ = C.c_void_p, C.c_int, C.c_size_t
            L.mx_moe_layer_forward.argtypes = [P, I32, C.POINTER(QLinear), C.POINTER(Ffn), P, C.POINTER(Layout),
                                               P, P, P]
            L.mx_moe_layer_forward_ex.argtypes = L.mx_moe_layer_forward.argtypes + [C.POINTER(Options), P, P, SZ]
            L.mx_moe_layer_forward_static.argtypes = L.mx_moe_layer_forward.argtypes + [C.POINTER(Options), P]
            L.mx_moe_workspace_bytes.argtypes = [C.POINTER(Layout), I32]
            L.mx_moe_workspace_bytes.restype = SZ
            L.mx_moe_stack_workspace_bytes.argtypes = [C.POINTER(Layout), I32]
            L.mx_moe_stack_workspace_bytes.restype = SZ
            L.mx_moe_workspace_init.argtypes = [P, SZ, P]
            L.mx_moe_down_sb_bytes.argtypes = [C.POINTER(Layout)]
            L.mx_moe_down_sb_bytes.restype = SZ
            L.mx_moe_pack_down_sb.argtypes = [C.POINTER(Layout), P, C.POINTER(QLinear), P, P]
            L.mx_moe_route.argtypes = [P, I32, C.POINTER(QLinear), C.POINTER(Layout), P, P, P, P, P, P,
                                       C.POINTER(Options), P, P, SZ]
            L.mx_moe_stack_forward.argtypes = [P, I32, I32, C.POINTER(QLinear), C.POINTER(Ffn), C.POINTER(P),
                                               C.POINTER(Layout), P, P, C.c_float, P, P, SZ]
            L.mx_status_string.argtypes = [I32]
            L.mx_status_string.restype = C.c_char_p
            L.mx_last_error_string.restype = C.c_char_p
            L.mx_version.restype = C.c_char_p
            L.mx_moe_profile_enable.argtypes = [I32]
            L.mx_moe_workspace_check.argtypes = [P, P]
            L.mx_moe_profile_read.argtypes = [C.POINTER(C.c_double), C.POINTER(C.c_int), I32]
            for name in ("mx_moe_layer_forward", "mx_moe_layer_forward_ex", "mx_moe_layer_forward_static",
                         "mx_moe_workspace_init", "mx_moe_pack_down_sb",
                         "mx_moe_route", "mx_moe_stack_forward", "mx_moe_profile_enable", "mx_moe_profile_read",
                         "mx_moe_workspace_check"):
                getattr(L, name).restype = C.c_int
            _lib = L
    return _lib


def _check(status: int):
    if status != 0:
        L = lib()
        raise MxError(status, f"{L.mx_status_string(status).decode()}: {L.mx_last_error_string().decode()}")


def _ptr(t):
    """Device (or host) address of a tensor, or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream_handle(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------------------- structs

def make_qlinear(w, s, b, rows: int, cols: int, bits: int) -> QLinear:
    return QLinear(_ptr(w), _ptr(s), _ptr(b), rows, cols, bits)


def make_layout(D, I, E, K, S, stride, offsets, act_dtype, lam, per_expert_scale=None, expert_slot=None,
                n_slots=0, router_scale=None, post_norm=None, post_eps=0.0, shared_expert_gate=None,
                down_sb=None) -> Layout:
    L = Layout()
    L.magic, L.version = LAYOUT_MAGIC, LAYOUT_VERSION
    L.d_model, L.d_expert, L.n_experts, L.top_k, L.d_shared = D, I, E, K, S
    L.group, L.bits = 64, 4
    L.record_stride = stride
    for name in ("gate", "up", "down"):
        w, s, b = offsets[name]
        setattr(L, name, Sub(w, s, b))
    L.act_dtype = act_dtype
    L.layer_scalar = lam
    L.per_expert_scale = _ptr(per_expert_scale)
    L.expert_slot = _ptr(expert_slot)
    L.n_slots = n_slots if expert_slot is not None else 0
    L.router_scale = _ptr(router_scale)
    L.post_norm = _ptr(post_norm)
    L.post_eps = post_eps
    L.shared_expert_gate = _ptr(shared_expert_gate)
    L.down_sb = _ptr(down_sb)
    return L


class DeviceLayer:
    """Device copy of one MoE layer given as host arrays.

    ``host`` is any object with attributes D, E, K, I, S, lam, router, shared_gate,
    shared_up, shared_down (each with .w .s .b .rows .cols .bits numpy arrays),
    blob, stride, offsets and optionally per_expert_scale and the layer's
    optional parts expert_slot (int16 [E]) with n_slots, router_scale,
    post_norm (with post_eps) and shared_expert_gate (BF16 bits [D]).

    ``pack_down_sb`` (default on) also builds the layout's packed
    down-projection scale / bias table (mx_moe_pack_down_sb) on the device."""

    def __init__(self, host, act_dtype: int, device="cuda", pack_down_sb: bool = True):
        import numpy as np
        import torch
        self.host = host
        self.act_dtype = act_dtype

        def dev(a):
            return torch.from_numpy(a.reshape(-1).view("uint8")).to(device, non_blocking=False)

        def q(m):
            ts = (dev(m.w), dev(m.s), dev(m.b))
            return ts, make_qlinear(*ts, m.rows, m.cols, m.bits)

        self._router_t, self.router = q(host.router)
        sg_t, sg = q(host.shared_gate)
        su_t, su = q(host.shared_up)
        sd_t, sd = q(host.shared_down)
        self._shared_t = (sg_t, su_t, sd_t)
        self.shared = Ffn(sg, su, sd)
        self.blob = torch.from_numpy(host.blob).to(device)
        assert self.blob.data_ptr() % 256 == 0
        pes = getattr(host, "per_expert_scale", None)
        self.pes = None if pes is None else torch.from_numpy(pes.astype("float32")).to(device)
        def opt(name, dtype):
            a = getattr(host, name, None)
            return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=dtype)).to(device)

        self.expert_slot = opt("expert_slot", np.int16)
        self.router_scale = opt("router_scale", np.uint16)
        self.post_norm = opt("post_norm", np.uint16)
        self.shared_expert_gate = opt("shared_expert_gate", np.uint16)
        self.layout = make_layout(host.D, host.I, host.E, host.K, host.S, host.stride, host.offsets, act_dtype,
                                  host.lam, self.pes, self.expert_slot, int(getattr(host, "n_slots", 0) or 0),
                                  self.router_scale, self.post_norm, float(getattr(host, "post_eps", 0.0)),
                                  self.shared_expert_gate)
        self.down_sb = None
        if pack_down_sb:
            self.down_sb = _pack_down_sb(self.layout, self.blob, self.shared.down, device=device)
            self.layout.down_sb = self.down_sb.data_ptr()

    def set_layer_scalar(self, lam: float):
        self.layout.layer_scalar = lam


# --------------------------------------------------------------- entry points

def down_sb_bytes(layout: Layout) -> int:
    return lib().mx_moe_down_sb_bytes(C.byref(layout))


def _pack_down_sb(layout: Layout, blob, shared_down: QLinear, device="cuda", stream=None):
    """The layout's packed down-projection (scale | bias << 16) words as a new
    device uint8 tensor (mx_moe_pack_down_sb); the copy is done when this
    returns."""
    import torch
    n = down_sb_bytes(layout)
    if n == 0:
        _check(-1)
    out = torch.empty(n, dtype=torch.uint8, device=device)
    _check(lib().mx_moe_pack_down_sb(C.byref(layout), _ptr(blob), C.byref(shared_down), _ptr(out),
                                     _stream_handle(stream)))
    torch.cuda.synchronize(out.device)
    return out


pack_down_sb = _pack_down_sb


def workspace_bytes(layout: Layout, T: int) -> int:
    return lib().mx_moe_workspace_bytes(C.byref(layout), T)


def stack_workspace_bytes(layout: Layout, T: int) -> int:
    return lib().mx_moe_stack_workspace_bytes(C.byref(layout), T)


def workspace_init(ws, nbytes: int, stream=None):
    _check(lib().mx_moe_workspace_init(_ptr(ws), nbytes, _stream_handle(stream)))


def workspace_check(ws, stream=None):
    """Raise MxError(MX_ERR_DEVICE_TIMEOUT) if a device-side wait gave up."""
    _check(lib().mx_moe_workspace_check(_ptr(ws), _stream_handle(stream)))


def layer_forward(x, T, layer: DeviceLayer, out, topk_idx, topk_w):
    _check(lib().mx_moe_layer_forward(_ptr(x), T, C.byref(layer.router), C.byref(layer.shared),
                                      _ptr(layer.blob), C.byref(layer.layout), _ptr(out), _ptr(topk_idx),
                                      _ptr(topk_w)))


def layer_forward_ex(x, T, layer: DeviceLayer, out, topk_idx, topk_w, ws, ws_bytes, stream=None, residual=None,
                     pre_rmsnorm=False, rms_eps=1e-6):
    opt = Options(_ptr(residual), 1 if pre_rmsnorm else 0, rms_eps)
    _check(lib().mx_moe_layer_forward_ex(_ptr(x), T, C.byref(layer.router), C.byref(layer.shared),
                                         _ptr(layer.blob), C.byref(layer.layout), _ptr(out), _ptr(topk_idx),
                                         _ptr(topk_w), C.byref(opt), _stream_handle(stream), _ptr(ws), ws_bytes))


def layer_forward_static(x, T, layer: DeviceLayer, out, topk_idx, topk_w, stream=None, residual=None,
                         pre_rmsnorm=False, rms_eps=1e-6):
    """The block for T <= 4 with the library's fixed device scratch (no workspace, no allocation)."""
    opt = Options(_ptr(residual), 1 if pre_rmsnorm else 0, rms_eps)
    _check(lib().mx_moe_layer_forward_static(_ptr(x), T, C.byref(layer.router), C.byref(layer.shared),
                                             _ptr(layer.blob), C.byref(layer.layout), _ptr(out), _ptr(topk_idx),
                                             _ptr(topk_w), C.byref(opt), _stream_handle(stream)))


def route(x, T, layer: DeviceLayer, topk_idx, topk_w, counts, offsets, perm, ws, ws_bytes, logits=None,
          stream=None, pre_rmsnorm=False, rms_eps=1e-6):
    opt = Options(None, 1 if pre_rmsnorm else 0, rms_eps)
    _check(lib().mx_moe_route(_ptr(x), T, C.byref(layer.router), C.byref(layer.layout), _ptr(topk_idx),
                              _ptr(topk_w), _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(logits), C.byref(opt),
                              _stream_handle(stream), _ptr(ws), ws_bytes))


class Stack:
    """Arrays of per-layer C structs for mx_moe_stack_forward."""

    def __init__(self, layers: list[DeviceLayer]):
        n = len(layers)
        self.layers = layers
        self.routers = (QLinear * n)(*[l.router for l in layers])
        self.shareds = (Ffn * n)(*[l.shared for l in layers])
        self.blobs = (C.c_void_p * n)(*[l.blob.data_ptr() for l in layers])
        self.layouts = (Layout * n)(*[l.layout for l in layers])


def stack_forward(x_io, T, stack: Stack, topk_idx, topk_w, ws, ws_bytes, rms_eps=1e-6, stream=None):
    _check(lib().mx_moe_stack_forward(_ptr(x_io), T, len(stack.layers), stack.routers, stack.shareds, stack.blobs,
                                      stack.layouts, _ptr(topk_idx), _ptr(topk_w), rms_eps, _stream_handle(stream),
                                      _ptr(ws), ws_bytes))


PROFILE_STAGES = ("route", "gate_up", "down")


def profile_enable(on: bool):
    _check(lib().mx_moe_profile_enable(1 if on else 0))


def profile_read(reset: bool = True) -> dict:
    """Per-stage summed milliseconds and launch counts since the last reset."""
    ms = (C.c_double * 3)()
    n = (C.c_int * 3)()
    _check(lib().mx_moe_profile_read(ms, n, 1 if reset else 0))
    return {name: (ms[i], n[i]) for i, name in enumerate(PROFILE_STAGES)}
