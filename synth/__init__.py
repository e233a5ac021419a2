"""Seeded synthetic inputs for the routed-MoE FFN block.

This module is shared by the tests, the smoke check and the benchmark.  It
holds none of the block's arithmetic: it draws random packed words, BF16 scale
and bias bit patterns and activations, and writes them into the fixed-stride
expert-record layout ("packed_experts" of the .gturbo directory on the
"Mference System design" page: fixed-stride, page-aligned records, one offset
per sub-tensor).  The oracle and the CUDA library each decode these bytes on
their own.

Distributions (the workload table of the block's benchmark):
  experts and shared expert: q ~ U{0..15} packed 8 per uint32, low nibble first;
      scale ~ U[0.005, 0.02], bias ~ U[-0.08, 0], both rounded RNE to BF16;
  router (8-bit): q ~ U{0..255} packed 4 per uint32, low byte first;
      scale ~ U[1e-4, 4e-4], bias ~ U[-0.03, 0];
  activations ~ N(0, 1), fp32 or rounded RNE to BF16; layer scalar 0.5.
Every tensor has its own generator keyed by (seed, layer, role, expert), so the
draw of one tensor does not depend on the order or the set of tensors drawn.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

GROUP = 64
PAGE = 4096
SUB_ALIGN = 256

# tensor roles (part of the generator key)
_ROLE_X, _ROLE_ROUTER, _ROLE_SHARED, _ROLE_EXPERT, _ROLE_ZIPF = 1, 2, 3, 4, 5


@dataclass(frozen=True)
class Config:
    name: str
    T: int
    D: int
    E: int
    K: int
    I: int
    S: int
    act: str            # "f32" or "bf16"
    seed: int
    layers: int = 1
    routing: str = "uniform"   # or "zipf"
    lam: float = 0.5


CONFIGS = {
    0: Config("tiny_T4_D256_E16_K2", T=4, D=256, E=16, K=2, I=128, S=128, act="f32", seed=0),
    1: Config("decode_T1_D2816_E128_K8_x30", T=1, D=2816, E=128, K=8, I=704, S=2112,
              act="bf16", seed=1, layers=30),
    2: Config("prefill_T512_D2816_E128_K8", T=512, D=2816, E=128, K=8, I=704, S=2112,
              act="bf16", seed=2),
    3: Config("skewed_decode_T64_D2816_E128_K8_zipf", T=64, D=2816, E=128, K=8, I=704, S=2112,
              act="bf16", seed=3, routing="zipf"),
    4: Config("prefill_T4096_D4096_E256_K8", T=4096, D=4096, E=256, K=8, I=1024, S=4096,
              act="bf16", seed=4),
}


@dataclass
class QMat:
    """Quantized matrix [rows, cols]: packed uint32 words and BF16 bit patterns."""
    w: np.ndarray          # uint32 [rows, cols*bits/32]
    s: np.ndarray          # uint16 [rows, cols/64]
    b: np.ndarray          # uint16 [rows, cols/64]
    rows: int
    cols: int
    bits: int


@dataclass
class MoeLayer:
    D: int
    E: int
    K: int
    I: int
    S: int
    lam: float
    router: QMat
    shared_gate: QMat
    shared_up: QMat
    shared_down: QMat
    blob: np.ndarray                     # uint8 [E * stride]
    stride: int
    offsets: dict                        # name -> (w_off, s_off, b_off)
    per_expert_scale: np.ndarray | None = None
    meta: dict = field(default_factory=dict)
    # optional parts of the layer (None = absent)
    expert_slot: np.ndarray | None = None       # int16 [E]: record of expert e (-1 = not resident)
    n_slots: int = 0                            # records in the blob when expert_slot is set
    router_scale: np.ndarray | None = None      # BF16 bits [D]
    post_norm: np.ndarray | None = None         # BF16 bits [D]
    post_eps: float = 1e-6
    shared_expert_gate: np.ndarray | None = None  # BF16 bits [D]

    def expert(self, e: int) -> tuple[QMat, QMat, QMat]:
        """Views of expert e's (gate, up, down) inside the blob."""
        rec = self.blob[e * self.stride:(e + 1) * self.stride]
        out = []
        for name, rows, cols in (("gate", self.I, self.D), ("up", self.I, self.D),
                                 ("down", self.D, self.I)):
            wo, so, bo = self.offsets[name]
            G = cols // GROUP
            w = rec[wo:wo + rows * cols // 2].view(np.uint32).reshape(rows, cols // 8)
            s = rec[so:so + rows * G * 2].view(np.uint16).reshape(rows, G)
            b = rec[bo:bo + rows * G * 2].view(np.uint16).reshape(rows, G)
            out.append(QMat(w, s, b, rows, cols, 4))
        return tuple(out)


# --------------------------------------------------------------- primitives

def rng_for(seed: int, layer: int, role: int, index: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, layer, role, index])))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to BF16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    u = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return u.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def uniform_bf16(rng: np.random.Generator, lo: float, hi: float, shape) -> np.ndarray:
    u = rng.random(shape, dtype=np.float32)
    return f32_to_bf16_bits(np.float32(lo) + np.float32(hi - lo) * u)


def random_words(rng: np.random.Generator, shape) -> np.ndarray:
    """Uniform uint32 words (raw generator output): every nibble and byte is
    uniform and independent."""
    n = int(np.prod(shape))
    raw = rng.bit_generator.random_raw((n + 1) // 2).view(np.uint32)[:n]
    return raw.reshape(shape)


def make_qmat(rng: np.random.Generator, rows: int, cols: int, bits: int,
              s_range: tuple[float, float], b_range: tuple[float, float]) -> QMat:
    assert cols % GROUP == 0
    G = cols // GROUP
    w = random_words(rng, (rows, cols * bits // 32))
    s = uniform_bf16(rng, *s_range, (rows, G))
    b = uniform_bf16(rng, *b_range, (rows, G))
    return QMat(w, s, b, rows, cols, bits)


EXPERT_S = (0.005, 0.02)
EXPERT_B = (-0.08, 0.0)
ROUTER_S = (1e-4, 4e-4)
ROUTER_B = (-0.03, 0.0)


# ------------------------------------------------------------------- layout

def _align(n: int, a: int) -> int:
    return (n + a - 1) // a * a


def default_layout(D: int, I: int) -> tuple[dict, int]:
    """Sub-tensor offsets inside one expert record and the record stride.

    Order: gate.w, up.w, down.w, gate.s, up.s, down.s, gate.b, up.b, down.b, each
    256-byte aligned; the stride is rounded up to a 4 KiB page."""
    sizes_w = {"gate": I * D // 2, "up": I * D // 2, "down": D * I // 2}
    sizes_sb = {"gate": I * (D // GROUP) * 2, "up": I * (D // GROUP) * 2,
                "down": D * (I // GROUP) * 2}
    off, pos = {n: [0, 0, 0] for n in ("gate", "up", "down")}, 0
    for n in ("gate", "up", "down"):
        off[n][0] = pos
        pos = _align(pos + sizes_w[n], SUB_ALIGN)
    for j in (1, 2):
        for n in ("gate", "up", "down"):
            off[n][j] = pos
            pos = _align(pos + sizes_sb[n], SUB_ALIGN)
    stride = _align(pos, PAGE)
    return {n: tuple(v) for n, v in off.items()}, stride


def payload_bytes(D: int, I: int) -> int:
    """Packed values + scales + biases of one expert (no padding)."""
    return 3 * (I * D // 2) + 6 * (I * (D // GROUP) * 2)


def write_blob(experts: list[tuple[QMat, QMat, QMat]], D: int, I: int,
               offsets: dict | None = None, stride: int | None = None) -> tuple[np.ndarray, dict, int]:
    if offsets is None:
        offsets, stride = default_layout(D, I)
    E = len(experts)
    blob = np.zeros(E * stride, dtype=np.uint8)
    for e, mats in enumerate(experts):
        rec = blob[e * stride:(e + 1) * stride]
        for name, m in zip(("gate", "up", "down"), mats):
            wo, so, bo = offsets[name]
            for off, arr in ((wo, m.w), (so, m.s), (bo, m.b)):
                raw = np.ascontiguousarray(arr).view(np.uint8).ravel()
                rec[off:off + raw.size] = raw
    return blob, offsets, stride


# ------------------------------------------------------------------ configs

def _fill_blob_random(blob: np.ndarray, offsets: dict, stride: int, D: int, I: int,
                      seed: int, layer: int) -> None:
    E = blob.size // stride
    for e in range(E):
        rng = rng_for(seed, layer, _ROLE_EXPERT, e)
        rec = blob[e * stride:(e + 1) * stride]
        for name, rows, cols in (("gate", I, D), ("up", I, D), ("down", D, I)):
            wo, so, bo = offsets[name]
            G = cols // GROUP
            rec[wo:wo + rows * cols // 2].view(np.uint32)[:] = random_words(rng, rows * cols // 8)
            rec[so:so + rows * G * 2].view(np.uint16)[:] = uniform_bf16(rng, *EXPERT_S, rows * G)
            rec[bo:bo + rows * G * 2].view(np.uint16)[:] = uniform_bf16(rng, *EXPERT_B, rows * G)


# Zipf-skewed routing (skewed batched decode): the router's group biases of the
# expert with popularity rank r (1-based, a seeded permutation of the experts)
# are multiplied by 1 + ZIPF_A * r**-ZIPF_S.  With zero-mean activations a larger
# bias raises the variance of that expert's logit and so how often it lands in
# the top-K.  ZIPF_A is calibrated on the skewed-decode workload (T = 64, seed
# 3) with the oracle's router: 30.3% of the 512 slots fall on the 8 most
# popular experts and 116 of the 128 experts are selected at all
# (tests/test_synth.py keeps that calibration).
ZIPF_S = 1.1
ZIPF_A = 20.0


def zipf_bias_multipliers(E: int, seed: int) -> tuple[np.ndarray, np.ndarray]:
    rng = rng_for(seed, 0, _ROLE_ZIPF)
    order = rng.permutation(E)                 # order[r-1] = expert of rank r
    rank = np.empty(E, dtype=np.int64)
    rank[order] = np.arange(1, E + 1)
    mult = 1.0 + ZIPF_A * rank.astype(np.float64) ** (-ZIPF_S)
    return mult.astype(np.float32), order


def make_layer(cfg: Config, layer: int = 0) -> MoeLayer:
    D, E, I, S = cfg.D, cfg.E, cfg.I, cfg.S
    router = make_qmat(rng_for(cfg.seed, layer, _ROLE_ROUTER), E, D, 8, ROUTER_S, ROUTER_B)
    meta = {}
    if cfg.routing == "zipf":
        mult, order = zipf_bias_multipliers(E, cfg.seed)
        b = bf16_bits_to_f32(router.b) * mult[:, None]
        router.b = f32_to_bf16_bits(b)
        meta["zipf_order"] = order
    rs = rng_for(cfg.seed, layer, _ROLE_SHARED)
    sg = make_qmat(rs, S, D, 4, EXPERT_S, EXPERT_B)
    su = make_qmat(rs, S, D, 4, EXPERT_S, EXPERT_B)
    sd = make_qmat(rs, D, S, 4, EXPERT_S, EXPERT_B)
    offsets, stride = default_layout(D, I)
    blob = np.zeros(E * stride, dtype=np.uint8)
    _fill_blob_random(blob, offsets, stride, D, I, cfg.seed, layer)
    return MoeLayer(D=D, E=E, K=cfg.K, I=I, S=S, lam=cfg.lam, router=router, shared_gate=sg,
                    shared_up=su, shared_down=sd, blob=blob, stride=stride, offsets=offsets,
                    meta=meta)


def make_x(cfg: Config, T: int | None = None) -> np.ndarray:
    """Activations [T, D]: fp32, or BF16 bit patterns (uint16) for bf16 configs."""
    T = cfg.T if T is None else T
    x = rng_for(cfg.seed, 0, _ROLE_X).standard_normal((T, cfg.D), dtype=np.float32)
    return x if cfg.act == "f32" else f32_to_bf16_bits(x)


def small_config(T=4, D=256, E=16, K=2, I=128, S=128, act="f32", seed=0, routing="uniform",
                 lam=0.5) -> Config:
    return Config(f"custom_T{T}_D{D}_E{E}_K{K}_I{I}_S{S}_{act}", T=T, D=D, E=E, K=K, I=I, S=S,
                  act=act, seed=seed, routing=routing, lam=lam)
