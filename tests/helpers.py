"""Test-side helpers: hand construction of quantized matrices and the
comparison metrics.  Independent of both the oracle and the CUDA library."""
from __future__ import annotations

import numpy as np

from synth import QMat, f32_to_bf16_bits, bf16_bits_to_f32, write_blob, MoeLayer


def pack(q: np.ndarray, bits: int) -> np.ndarray:
    """Pack integer values [rows, cols] into uint32 words, low nibble/byte first."""
    q = np.asarray(q, dtype=np.uint64)
    per = 32 // bits
    rows, cols = q.shape
    q = q.reshape(rows, cols // per, per)
    shifts = (np.arange(per, dtype=np.uint64) * bits)[None, None, :]
    return (q << shifts).sum(axis=2).astype(np.uint32)


def qmat_from(q, s, b, bits) -> QMat:
    """q: ints [rows, cols]; s, b: floats [rows, cols/64] (must be exact in BF16)."""
    q = np.asarray(q)
    rows, cols = q.shape
    s = np.broadcast_to(np.asarray(s, dtype=np.float32), (rows, cols // 64))
    b = np.broadcast_to(np.asarray(b, dtype=np.float32), (rows, cols // 64))
    sb, bb = f32_to_bf16_bits(s), f32_to_bf16_bits(b)
    assert np.array_equal(bf16_bits_to_f32(sb), s) and np.array_equal(bf16_bits_to_f32(bb), b), \
        "hand-built scales/biases must be exact in BF16"
    return QMat(pack(q, bits), np.ascontiguousarray(sb), np.ascontiguousarray(bb), rows, cols, bits)


def dequant64(m: QMat) -> np.ndarray:
    """fp64 dense copy of a quantized matrix (test-side, for closed forms)."""
    per = 32 // m.bits
    mask = (1 << m.bits) - 1
    w = m.w.astype(np.uint64)
    q = np.stack([(w >> np.uint64(m.bits * j)) & np.uint64(mask) for j in range(per)], axis=2)
    q = q.reshape(m.rows, m.cols).astype(np.float64)
    s = np.repeat(bf16_bits_to_f32(m.s).astype(np.float64), 64, axis=1)
    b = np.repeat(bf16_bits_to_f32(m.b).astype(np.float64), 64, axis=1)
    return s * q + b


def layer_from(router, shared, experts, D, I, S, K, lam=0.5) -> MoeLayer:
    blob, offsets, stride = write_blob(experts, D, I)
    return MoeLayer(D=D, E=len(experts), K=K, I=I, S=S, lam=lam, router=router,
                    shared_gate=shared[0], shared_up=shared[1], shared_down=shared[2],
                    blob=blob, stride=stride, offsets=offsets)


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a - b))


def max_abs_rel(a, b) -> float:
    """max |a - b| / max |b| (the max-abs bar read relative to the output scale)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    m = np.max(np.abs(b))
    return float(np.max(np.abs(a - b)) / m) if m > 0 else float(np.max(np.abs(a - b)))
