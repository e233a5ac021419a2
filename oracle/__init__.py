"""ctypes wrapper around the plain C oracle (``mx_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this module.  The
product path (``expert_ffn_gb300``) never imports it, and this module imports
nothing from the product.  Inputs come from the seeded generator in ``synth``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mx_oracle.c")
_HDR = os.path.join(_HERE, "mx_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
# -ffp-contract=off: the only fused multiply-adds are the explicit fmaf calls.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with gcc (portable flags, no arch tuning)."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class QMat(C.Structure):
    _fields_ = [("w", C.c_void_p), ("s", C.c_void_p), ("b", C.c_void_p),
                ("rows", C.c_int32), ("cols", C.c_int32), ("bits", C.c_int32)]


class Layer(C.Structure):
    _fields_ = [("d_model", C.c_int32), ("d_expert", C.c_int32), ("n_experts", C.c_int32),
                ("top_k", C.c_int32), ("layer_scalar", C.c_float),
                ("router", QMat), ("shared_gate", QMat), ("shared_up", QMat), ("shared_down", QMat),
                ("blob", C.c_void_p), ("record_stride", C.c_uint64),
                ("off_w", C.c_uint64 * 3), ("off_s", C.c_uint64 * 3), ("off_b", C.c_uint64 * 3),
                ("per_expert_scale", C.c_void_p),
                ("expert_slot", C.c_void_p), ("n_slots", C.c_int32),
                ("router_scale", C.c_void_p), ("post_norm", C.c_void_p), ("post_eps", C.c_float),
                ("shared_expert_gate", C.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            P = C.c_void_p
            L.oracle_bf16_to_f32.restype = C.c_float
            L.oracle_bf16_to_f32.argtypes = [C.c_uint16]
            L.oracle_f32_to_bf16.restype = C.c_uint16
            L.oracle_f32_to_bf16.argtypes = [C.c_float]
            L.oracle_gelu.restype = C.c_float
            L.oracle_gelu.argtypes = [C.c_float]
            L.oracle_qmatvec.argtypes = [C.POINTER(QMat), P, P]
            L.oracle_router_logits.argtypes = [C.POINTER(QMat), P, C.c_int, P]
            L.oracle_topk_softmax.argtypes = [P, C.c_int, C.c_int, C.c_int, P, P, P]
            L.oracle_topk_softmax.restype = C.c_int
            L.oracle_permute.argtypes = [P, C.c_int, C.c_int, C.c_int, P, P, P]
            L.oracle_permute.restype = C.c_int
            L.oracle_expert_ffn.argtypes = [C.POINTER(QMat)] * 3 + [P, P]
            L.oracle_block_forward.argtypes = [C.POINTER(Layer), P, C.c_int, C.c_int, P, P, P, P]
            L.oracle_block_forward.restype = C.c_int
            L.oracle_rmsnorm_bf16.argtypes = [P, C.c_int, C.c_int, C.c_float, P]
            L.oracle_stack_forward.argtypes = [C.POINTER(Layer), C.c_int, P, C.c_int, C.c_float, P, P, P]
            L.oracle_stack_forward.restype = C.c_int
            _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def qmat(m) -> QMat:
    """Build the C view of a ``synth.QMat`` (keeps references in the caller)."""
    return QMat(_ptr(m.w), _ptr(m.s), _ptr(m.b), m.rows, m.cols, m.bits)


def layer_struct(layer) -> Layer:
    """C view of a ``synth.MoeLayer``.  The numpy arrays must outlive the struct."""
    o = layer.offsets
    L = Layer()
    L.d_model, L.d_expert, L.n_experts, L.top_k = layer.D, layer.I, layer.E, layer.K
    L.layer_scalar = layer.lam
    L.router = qmat(layer.router)
    L.shared_gate, L.shared_up, L.shared_down = (qmat(layer.shared_gate), qmat(layer.shared_up),
                                                 qmat(layer.shared_down))
    L.blob = _ptr(layer.blob)
    L.record_stride = layer.stride
    for j, name in enumerate(("gate", "up", "down")):
        L.off_w[j], L.off_s[j], L.off_b[j] = o[name]
    L.per_expert_scale = _ptr(layer.per_expert_scale)
    opt = lambda name, dt: _ptr(None if getattr(layer, name, None) is None  # noqa: E731
                                else np.ascontiguousarray(getattr(layer, name), dtype=dt))
    # the arrays must be the layer's own (contiguous, of the right dtype) so they outlive the struct
    for name, dt in (("expert_slot", np.int16), ("router_scale", np.uint16), ("post_norm", np.uint16),
                     ("shared_expert_gate", np.uint16)):
        a = getattr(layer, name, None)
        if a is not None:
            assert a.dtype == dt and a.flags["C_CONTIGUOUS"], f"{name} must be contiguous {dt.__name__}"
    L.expert_slot = opt("expert_slot", np.int16)
    L.n_slots = int(getattr(layer, "n_slots", 0) or 0)
    L.router_scale = opt("router_scale", np.uint16)
    L.post_norm = opt("post_norm", np.uint16)
    L.post_eps = float(getattr(layer, "post_eps", 1e-6))
    L.shared_expert_gate = opt("shared_expert_gate", np.uint16)
    return L


# ------------------------------------------------------------------ scalars

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of BF16 bit patterns (plain bit shift)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def gelu(z: float) -> float:
    return lib().oracle_gelu(float(z))


def f32_to_bf16(v: float) -> int:
    return lib().oracle_f32_to_bf16(float(v))


def f32_to_bf16_array(a: np.ndarray) -> np.ndarray:
    f = lib().oracle_f32_to_bf16
    flat = np.ascontiguousarray(a, dtype=np.float32).ravel()
    return np.array([f(float(v)) for v in flat], dtype=np.uint16).reshape(np.shape(a))


# ------------------------------------------------------------------- pieces

def qmatvec(m, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.zeros(m.rows, dtype=np.float32)
    q = qmat(m)
    lib().oracle_qmatvec(C.byref(q), _ptr(x), _ptr(y))
    return y


def router_logits(router, x: np.ndarray) -> np.ndarray:
    """x: fp32 [T, D] values (BF16 inputs already widened)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    T = x.shape[0]
    out = np.zeros((T, router.rows), dtype=np.float32)
    q = qmat(router)
    lib().oracle_router_logits(C.byref(q), _ptr(x), T, _ptr(out))
    return out


def topk_softmax(logits: np.ndarray, K: int, per_expert_scale=None):
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    idx = np.zeros((T, K), dtype=np.int32)
    w = np.zeros((T, K), dtype=np.float32)
    pes = None if per_expert_scale is None else np.ascontiguousarray(per_expert_scale, np.float32)
    rc = lib().oracle_topk_softmax(_ptr(logits), T, E, K, _ptr(pes), _ptr(idx), _ptr(w))
    if rc:
        raise ValueError("oracle_topk_softmax: bad arguments")
    return idx, w


def permute(topk_idx: np.ndarray, E: int):
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, K = topk_idx.shape
    counts = np.zeros(E, dtype=np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    perm = np.zeros(T * K, dtype=np.int32)
    rc = lib().oracle_permute(_ptr(topk_idx), T, K, E, _ptr(counts), _ptr(offsets), _ptr(perm))
    if rc:
        raise ValueError("oracle_permute: expert index out of range")
    return counts, offsets, perm


def expert_ffn(gate, up, down, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.zeros(down.rows, dtype=np.float32)
    g, u, d = qmat(gate), qmat(up), qmat(down)
    lib().oracle_expert_ffn(C.byref(g), C.byref(u), C.byref(d), _ptr(x), _ptr(y))
    return y


class ExpertNotResident(ValueError):
    pass


def block_forward(layer, x: np.ndarray, residual: np.ndarray | None = None):
    """Run the block on the tokens in ``x`` (fp32 or BF16 bits, [T, D]).

    Returns ``(out, topk_idx, topk_w)``; ``out`` has x's dtype."""
    x = np.ascontiguousarray(x)
    dtype = 1 if x.dtype == np.uint16 else 0
    if dtype == 0:
        x = np.ascontiguousarray(x, dtype=np.float32)
    T = x.shape[0]
    out = np.zeros_like(x)
    idx = np.zeros((T, layer.K), dtype=np.int32)
    w = np.zeros((T, layer.K), dtype=np.float32)
    if residual is not None:
        residual = np.ascontiguousarray(residual, dtype=x.dtype)
    L = layer_struct(layer)
    rc = lib().oracle_block_forward(C.byref(L), _ptr(x), dtype, T, _ptr(residual), _ptr(out),
                                    _ptr(idx), _ptr(w))
    if rc == -2:
        raise ExpertNotResident("oracle_block_forward: a selected expert is not resident in the blob")
    if rc:
        raise ValueError("oracle_block_forward: bad arguments")
    return out, idx, w


def block_forward_tokens(layer, x: np.ndarray, tokens=None, threads: int | None = None):
    """``block_forward`` on the rows ``tokens`` of ``x`` (all rows if None),
    split over host threads: each thread runs the plain single-threaded oracle
    on its own share of the tokens (ctypes releases the GIL during the call,
    and every token is independent of the others).  Returns (out, idx, w) for
    the selected rows, in the order given."""
    import concurrent.futures as cf
    x = np.ascontiguousarray(x)
    tok = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens, dtype=np.int64)
    n = len(tok)
    threads = max(1, min(threads or (os.cpu_count() or 1), n))
    parts = np.array_split(np.arange(n), threads)
    out = np.zeros((n, x.shape[1]), dtype=x.dtype if x.dtype == np.uint16 else np.float32)
    idx = np.zeros((n, layer.K), dtype=np.int32)
    w = np.zeros((n, layer.K), dtype=np.float32)

    def run(part):
        if len(part):
            o, i, ww = block_forward(layer, np.ascontiguousarray(x[tok[part]]))
            out[part], idx[part], w[part] = o, i, ww

    lib()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(run, parts))
    return out, idx, w


def rmsnorm_bf16(x_bits: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, D = x_bits.shape
    y = np.zeros_like(x_bits)
    lib().oracle_rmsnorm_bf16(_ptr(x_bits), T, D, eps, _ptr(y))
    return y


def stack_forward(layers, x_bits: np.ndarray, eps: float = 1e-6):
    """Decode stack over ``layers``; returns (per-layer outputs, topk_idx, topk_w)."""
    x = np.array(x_bits, dtype=np.uint16, copy=True, order="C")
    T, D = x.shape
    n = len(layers)
    K = layers[0].K
    structs = (Layer * n)(*[layer_struct(l) for l in layers])
    xs = np.zeros((n, T, D), dtype=np.uint16)
    idx = np.zeros((n, T, K), dtype=np.int32)
    w = np.zeros((n, T, K), dtype=np.float32)
    rc = lib().oracle_stack_forward(structs, n, _ptr(x), T, eps, _ptr(xs), _ptr(idx), _ptr(w))
    if rc:
        raise ValueError("oracle_stack_forward: bad arguments")
    return xs, idx, w
