"""Pins for the CPU oracle: closed forms, brute force, invariants, and the
by-hand example.  Each test is chosen so that a plausible mistake in the oracle
(a wrong nibble order, group index, transposed operand, dropped bias term,
wrong GELU form, wrong tie rule, wrong sign) fails at least one of them.

Cited passages: "Mference System design" page -- "Why the runtime has this
shape" (128 experts / top-8, shared expert without routing weight, MLX affine
group-64 quantization with BF16 scale and bias, 8-bit router), "Decode"
(router formula), "Metal execution" (affine decode + GeGLU + weighted
reduction); "TinyTitan_Datacenter Architecture" page, "Invariants" (fp32
accumulation, fixed reduction order, discrete decisions checked exactly)."""
from __future__ import annotations

import math
import os

import numpy as np
import pytest

import synth
from synth import bf16_bits_to_f32, f32_to_bf16_bits
from tests.helpers import dequant64, layer_from, pack, qmat_from, rel_l2

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "two_expert_example.txt")


def read_golden(path):
    vals = {}
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, *v = line.split()
        vals[k] = [float(x) for x in v] if len(v) > 1 else float(v[0])
    return vals


# ----------------------------------------------------------------- dtypes

def test_bf16_rounding_textbook_cases(orc):
    # 1.0; exact ties go to even; above-half rounds up; sign; overflow to inf.
    cases = {0x3F800000: 0x3F80, 0x3F808000: 0x3F80, 0x3F818000: 0x3F82, 0x3F80C000: 0x3F81,
             0x3F807FFF: 0x3F80, 0xBF80C000: 0xBF81, 0x7F7FFFFF: 0x7F80, 0x00000001: 0x0000}
    for bits, want in cases.items():
        f = np.array([bits], dtype=np.uint32).view(np.float32)[0]
        assert orc.f32_to_bf16(float(f)) == want, hex(bits)
    for h in (0x0000, 0x3F80, 0xC2F7, 0x0001, 0x7F7F):
        assert orc.lib().oracle_bf16_to_f32(h) == bf16_bits_to_f32(np.array([h]))[0]


# ------------------------------------------------------------------- GELU

def test_gelu_tanh_form(orc):
    assert orc.gelu(0.0) == 0.0
    # odd-part identity of the tanh form: gelu(z) - gelu(-z) = z
    for z in (0.125, 0.25, 1.0, 3.0, 7.5):
        assert abs((orc.gelu(z) - orc.gelu(-z)) - z) <= 4e-7 * max(1.0, z)
    # limits
    assert orc.gelu(12.0) == pytest.approx(12.0, rel=1e-7)
    assert abs(orc.gelu(-12.0)) < 1e-6
    # the tanh form (not the erf form) at |z| = 1: 0.84119199 vs 0.84134475
    ref_tanh = 0.5 * (1 + math.tanh(math.sqrt(2 / math.pi) * (1 + 0.044715)))
    ref_erf = 0.5 * (1 + math.erf(1 / math.sqrt(2)))
    assert abs(orc.gelu(1.0) - ref_tanh) < 1e-6
    assert abs(orc.gelu(1.0) - ref_erf) > 1e-4
    for z in (-3.0, -1.0, -0.25, -0.125, 0.125, 0.25, 1.0, 3.0):
        ref = 0.5 * z * (1 + math.tanh(math.sqrt(2 / math.pi) * (z + 0.044715 * z ** 3)))
        assert abs(orc.gelu(z) - ref) <= 1e-6 * max(1.0, abs(z))


# ---------------------------------------------------------------- dequant

@pytest.mark.parametrize("bits", [4, 8])
def test_dequant_one_hot_columns(orc, bits):
    """W e_j = column j = s[r, j/64] * q[r, j] + b[r, j/64] exactly.

    The q pattern differs in every row and column, and the scales/biases in
    every group, so a wrong nibble order, group index or transpose fails."""
    rows, cols = 8, 192
    r = np.arange(rows)[:, None]
    c = np.arange(cols)[None, :]
    q = (r + 3 * c + (c // 8)) % (1 << bits)
    G = cols // 64
    s = np.array([[2.0 ** -(3 + rr + 2 * g) for g in range(G)] for rr in range(rows)])
    b = np.array([[-(rr + 1) * 2.0 ** -(6 + g) for g in range(G)] for rr in range(rows)])
    m = qmat_from(q, s, b, bits)
    for j in (0, 1, 5, 7, 8, 63, 64, 70, 127, 128, 191):
        x = np.zeros(cols, dtype=np.float32)
        x[j] = 1.0
        y = orc.qmatvec(m, x)
        want = s[:, j // 64] * q[:, j] + b[:, j // 64]
        assert np.array_equal(y, want.astype(np.float32)), (bits, j)


def test_all_zero_nibbles_closed_form(orc):
    """q = 0 everywhere: every weight is its group bias, W x = sum_g b_g X_g."""
    rng = np.random.default_rng(11)
    rows, cols = 16, 256
    q = np.zeros((rows, cols), dtype=np.int64)
    s = f32_to_bf16_bits(rng.uniform(0.005, 0.02, (rows, cols // 64)).astype(np.float32))
    b = f32_to_bf16_bits(rng.uniform(-0.08, 0, (rows, cols // 64)).astype(np.float32))
    m = qmat_from(q, bf16_bits_to_f32(s), bf16_bits_to_f32(b), 4)
    x = rng.standard_normal(cols).astype(np.float32)
    X = x.astype(np.float64).reshape(-1, 64).sum(axis=1)
    want = bf16_bits_to_f32(b).astype(np.float64) @ X
    y = orc.qmatvec(m, x)
    bound = 1e-6 * (np.abs(bf16_bits_to_f32(b)).astype(np.float64) @ np.abs(x).reshape(-1, 64).sum(1))
    assert np.all(np.abs(y - want) <= bound + 1e-30)


def test_all_fifteen_nibbles_exact_dyadic(orc):
    """q = 15, s = 2^-6, b = 0: w = 15/64; x = k/8 gives an exactly representable sum."""
    rows, cols = 4, 128
    m = qmat_from(np.full((rows, cols), 15), 2.0 ** -6, 0.0, 4)
    x = (np.arange(cols) % 9 - 4).astype(np.float32) / 8
    y = orc.qmatvec(m, x)
    want = 15 / 64 * x.astype(np.float64).sum()
    assert np.all(y == np.float32(want))


def test_qmatvec_against_dense_fp64(orc):
    rng = np.random.default_rng(5)
    m = synth.make_qmat(rng, 24, 320, 4, synth.EXPERT_S, synth.EXPERT_B)
    x = rng.standard_normal(320).astype(np.float32)
    ref = dequant64(m) @ x.astype(np.float64)
    y = orc.qmatvec(m, x)
    scale = np.abs(dequant64(m)) @ np.abs(x.astype(np.float64))
    assert np.all(np.abs(y - ref) <= 2e-6 * scale)


# ----------------------------------------------------------------- router

def _router_case(seed, E=16, D=256, T=6):
    rng = np.random.default_rng(seed)
    m = synth.make_qmat(rng, E, D, 8, synth.ROUTER_S, synth.ROUTER_B)
    x = rng.standard_normal((T, D)).astype(np.float32)
    return m, x


def test_router_logits_within_fp32_bound_of_exact(orc):
    m, x = _router_case(1)
    L = orc.router_logits(m, x)
    W = dequant64(m)
    ref = x.astype(np.float64) @ W.T
    scale = np.abs(x.astype(np.float64)) @ np.abs(W).T
    assert np.all(np.abs(L - ref) <= 4e-6 * scale)


def test_router_canonical_order_reproducible(orc):
    """Same bits on a permuted token order (the order is per token, fixed)."""
    m, x = _router_case(2, T=8)
    L = orc.router_logits(m, x)
    p = np.array([3, 0, 7, 1, 6, 2, 5, 4])
    assert np.array_equal(orc.router_logits(m, x[p]), L[p])


def test_topk_matches_full_sort_brute_force(orc):
    rng = np.random.default_rng(3)
    for E, K in ((16, 2), (128, 8), (256, 8), (7, 7), (9, 1)):
        logits = rng.standard_normal((20, E)).astype(np.float32)
        logits[:, 1] = logits[:, 4]                     # plant exact ties
        idx, w = orc.topk_softmax(logits, K)
        for t in range(logits.shape[0]):
            order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))
            assert list(idx[t]) == order[:K]


def test_topk_tie_selects_lower_index(orc):
    """Two identical router rows give equal logits; K=1 must pick the lower index."""
    rng = np.random.default_rng(4)
    m = synth.make_qmat(rng, 6, 128, 8, synth.ROUTER_S, synth.ROUTER_B)
    for arr in (m.w, m.s, m.b):
        arr[4] = arr[2]
    # make rows 2/4 the largest by giving them the largest scales and zero bias
    m.s[2] = m.s[4] = f32_to_bf16_bits(np.full(2, 4e-4, np.float32))
    m.b[2] = m.b[4] = 0
    x = np.abs(rng.standard_normal((3, 128))).astype(np.float32)
    L = orc.router_logits(m, x)
    assert np.array_equal(L[:, 2], L[:, 4])
    idx1, _ = orc.topk_softmax(L, 1)
    assert np.all(idx1[:, 0] == 2)
    idx2, w2 = orc.topk_softmax(L, 2)
    assert np.all(idx2 == [2, 4]) and np.all(w2[:, 0] == w2[:, 1])


def test_topk_nan_ranks_as_minus_infinity_and_degenerate_k(orc):
    """The reading for NaN logits: they rank as -inf (after every finite
    logit, ties among them to the lower index).  K = 1 gives weight exactly 1;
    K = E gives the softmax of the whole row."""
    logits = np.array([[0.5, np.nan, -3.0, np.nan, 2.0, -np.inf]], dtype=np.float32)
    idx, w = orc.topk_softmax(logits, 6)
    assert list(idx[0]) == [4, 0, 2, 1, 3, 5]   # finite desc, then NaN/-inf by index
    assert np.all(w[0, 3:] == 0.0)              # exp(-inf - max) = 0
    idx1, w1 = orc.topk_softmax(logits, 1)
    assert idx1[0, 0] == 4 and w1[0, 0] == 1.0
    rng = np.random.default_rng(8)
    full = rng.standard_normal((4, 9)).astype(np.float32)
    idx9, w9 = orc.topk_softmax(full, 9)
    ref = np.exp(full.astype(np.float64) - full.max(1, keepdims=True))
    ref /= ref.sum(1, keepdims=True)
    assert np.max(np.abs(w9 - np.take_along_axis(ref, idx9, 1))) <= 2e-7


def test_softmax_weights(orc):
    rng = np.random.default_rng(6)
    logits = (3 * rng.standard_normal((50, 128))).astype(np.float32)
    idx, w = orc.topk_softmax(logits, 8)
    assert np.all(np.abs(w.sum(1) - 1) <= 1e-6)
    assert np.all(np.diff(w, axis=1) <= 0)
    sel = np.take_along_axis(logits, idx, 1).astype(np.float64)
    want = np.exp(sel - sel[:, :1])
    want /= want.sum(1, keepdims=True)
    assert np.max(np.abs(w - want)) <= 2e-7
    # per-expert scale multiplies the selected weights
    pes = (1 + np.arange(128) / 64).astype(np.float32)
    idx2, w2 = orc.topk_softmax(logits, 8, pes)
    assert np.array_equal(idx2, idx)
    assert np.allclose(w2, w * pes[idx], rtol=1e-7, atol=0)


def test_permute_brute_force(orc):
    rng = np.random.default_rng(7)
    for T, K, E in ((1, 8, 128), (64, 8, 128), (33, 2, 16), (512, 8, 128)):
        idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
        counts, offsets, perm = orc.permute(idx, E)
        assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
        assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
        assert np.array_equal(perm, np.argsort(idx.ravel(), kind="stable"))


# ------------------------------------------------------------------ block

def two_expert_layer():
    D = I = S = 64
    one = np.ones((1, 64), dtype=np.int64)
    router = qmat_from(np.concatenate([2 * one, one]), 1 / 64, 0.0, 8)
    e0 = (qmat_from(np.ones((I, D)), 1 / 64, 0.0, 4), qmat_from(np.ones((I, D)), 1 / 64, 0.0, 4),
          qmat_from(np.ones((D, I)), 1 / 64, 0.0, 4))
    e1 = (qmat_from(2 * np.ones((I, D)), 1 / 64, 0.0, 4), qmat_from(np.ones((I, D)), 1 / 64, 0.0, 4),
          qmat_from(np.ones((D, I)), 1 / 64, 0.0, 4))
    sh = tuple(qmat_from(np.zeros((64, 64)), 1 / 64, 1 / 64, 4) for _ in range(3))
    return layer_from(router, sh, [e0, e1], D, I, S, K=2, lam=0.5)


def test_two_expert_hand_example(orc):
    g = read_golden(GOLDEN)
    layer = two_expert_layer()
    x = np.full((1, 64), 1 / 8, dtype=np.float32)
    L = orc.router_logits(layer.router, x)
    assert L[0, 0] == g["logit0"] and L[0, 1] == g["logit1"]
    out, idx, w = orc.block_forward(layer, x)
    assert list(idx[0]) == [int(v) for v in g["topk_idx"]]
    assert w[0, 0] == pytest.approx(g["w0"], rel=1e-6)
    assert w[0, 1] == pytest.approx(g["w1"], rel=1e-6)
    e0 = layer.expert(0)
    y0 = orc.expert_ffn(*e0, x[0])
    assert np.allclose(y0, g["y0"], rtol=1e-6, atol=0)
    y1 = orc.expert_ffn(*layer.expert(1), x[0])
    assert np.allclose(y1, g["y1"], rtol=1e-6, atol=0)
    assert np.allclose(out[0], g["out"], rtol=1e-6, atol=0)
    assert not np.allclose(out[0], g["out_erf_gelu"], rtol=1e-6, atol=0)
    # bf16 activations: same example, output rounded once
    xb = f32_to_bf16_bits(x)
    outb, idxb, _ = orc.block_forward(layer, xb)
    assert np.array_equal(idxb, idx)
    assert np.all(outb == f32_to_bf16_bits(np.float32(g["out"]) * np.ones(1, np.float32))[0])


def _tiny_layer(seed=0, **kw):
    cfg = synth.small_config(seed=seed, **kw)
    return cfg, synth.make_layer(cfg), synth.make_x(cfg)


def test_block_matches_dense_fp64_definition(orc):
    cfg, layer, x = _tiny_layer(0)
    out, idx, w = orc.block_forward(layer, x)
    xs = x.astype(np.float64)
    gelu = lambda z: 0.5 * z * (1 + np.tanh(np.sqrt(2 / np.pi) * (z + 0.044715 * z ** 3)))
    ffn = lambda g, u, d, v: dequant64(d) @ (gelu(dequant64(g) @ v) * (dequant64(u) @ v))
    for t in range(cfg.T):
        acc = ffn(layer.shared_gate, layer.shared_up, layer.shared_down, xs[t])
        for k in range(cfg.K):
            acc = acc + w[t, k] * ffn(*layer.expert(idx[t, k]), xs[t])
        ref = cfg.lam * acc
        assert rel_l2(out[t], ref) < 2e-6


def test_block_token_permutation_invariance(orc):
    cfg, layer, x = _tiny_layer(1, T=7)
    out, idx, w = orc.block_forward(layer, x)
    p = np.array([6, 2, 0, 5, 1, 4, 3])
    out_p, idx_p, w_p = orc.block_forward(layer, x[p])
    assert np.array_equal(out_p, out[p]) and np.array_equal(idx_p, idx[p]) and np.array_equal(w_p, w[p])


def test_block_linear_in_layer_scalar(orc):
    cfg, layer, x = _tiny_layer(2)
    out_half, _, _ = orc.block_forward(layer, x)
    layer.lam = 1.0
    out_one, _, _ = orc.block_forward(layer, x)
    assert np.array_equal(out_one, 2 * out_half)
    layer.lam = 0.0
    res = np.random.default_rng(0).standard_normal(x.shape).astype(np.float32)
    out_res, _, _ = orc.block_forward(layer, x, residual=res)
    assert np.array_equal(out_res, res)


def test_block_shared_branch_has_no_routing_weight(orc):
    """Zero routed down projections (w = 0): the output is lambda * shared exactly."""
    cfg, layer, x = _tiny_layer(3)
    wo, so, bo = layer.offsets["down"]
    D, I = cfg.D, cfg.I
    for e in range(cfg.E):
        rec = layer.blob[e * layer.stride:(e + 1) * layer.stride]
        rec[wo:wo + D * I // 2] = 0
        rec[so:so + D * (I // 64) * 2] = 0
        rec[bo:bo + D * (I // 64) * 2] = 0
    out, _, _ = orc.block_forward(layer, x)
    for t in range(cfg.T):
        sh = orc.expert_ffn(layer.shared_gate, layer.shared_up, layer.shared_down, x[t])
        assert np.array_equal(out[t], np.float32(cfg.lam) * sh)


def test_block_experts_selected_only(orc):
    """Changing an expert no token selects leaves the output unchanged."""
    cfg, layer, x = _tiny_layer(4)
    out, idx, _ = orc.block_forward(layer, x)
    unused = sorted(set(range(cfg.E)) - set(idx.ravel().tolist()))
    assert unused
    e = unused[0]
    layer.blob[e * layer.stride:(e + 1) * layer.stride] ^= 0x5A
    out2, idx2, _ = orc.block_forward(layer, x)
    assert np.array_equal(out2, out) and np.array_equal(idx2, idx)


# --------------------------------------------------------- rmsnorm / stack

def test_rmsnorm_closed_forms(orc):
    # constant rows: x / sqrt(x^2 + eps) ~ sign(x)
    x = f32_to_bf16_bits(np.array([[0.5] * 128, [-3.0] * 128], dtype=np.float32))
    y = bf16_bits_to_f32(orc.rmsnorm_bf16(x, 1e-6))
    assert np.all(np.abs(y[0] - 1) <= 2 ** -8) and np.all(np.abs(y[1] + 1) <= 2 ** -8)
    # eps = 0: scale invariance is exact (powers of two)
    rng = np.random.default_rng(8)
    xr = f32_to_bf16_bits(rng.standard_normal((3, 256)).astype(np.float32))
    x2 = f32_to_bf16_bits(2 * bf16_bits_to_f32(xr))
    assert np.array_equal(orc.rmsnorm_bf16(xr, 0.0), orc.rmsnorm_bf16(x2, 0.0))
    # against fp64 within one BF16 rounding
    xf = bf16_bits_to_f32(xr).astype(np.float64)
    ref = xf / np.sqrt((xf ** 2).mean(1, keepdims=True) + 1e-6)
    got = bf16_bits_to_f32(orc.rmsnorm_bf16(xr, 1e-6))
    assert np.all(np.abs(got - ref) <= 2 ** -8 * np.abs(ref) + 1e-30)


def test_stack_identity_when_scalar_zero_and_one_layer_match(orc):
    cfg = synth.small_config(T=2, act="bf16", seed=5)
    layers = [synth.make_layer(cfg, l) for l in range(3)]
    x = synth.make_x(cfg)
    xs, idx, w = orc.stack_forward(layers, x)
    # layer 0 of the stack = rmsnorm -> block -> residual
    xn = orc.rmsnorm_bf16(x)
    out0, idx0, w0 = orc.block_forward(layers[0], xn, residual=x)
    assert np.array_equal(xs[0], out0) and np.array_equal(idx[0], idx0)
    for l in layers:
        l.lam = 0.0
    xs0, _, _ = orc.stack_forward(layers, x)
    assert np.all(xs0 == x[None])


# ----------------------------------------------------------------- layout

def test_default_layout_sizes():
    for D, I, payload, stride in ((2816, 704, 3_345_408, 3_346_432), (4096, 1024, 7_077_888, 7_077_888),
                                  (256, 128, 55_296, 57_344)):
        off, st = synth.default_layout(D, I)
        assert synth.payload_bytes(D, I) == payload and st == stride and st % 4096 == 0
        for name in ("gate", "up", "down"):
            for o in off[name]:
                assert o % 256 == 0 and o < st
