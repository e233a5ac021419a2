"""Pins of the oracle's optional layer parts (CPU): the resident-set expert
table, the router's input scale, the post-FFN norm and the gated shared
expert.  Each is checked against what fixes it independently of the oracle:
an invariance (a permuted or reduced blob with a matching table), an exact
power-of-two scaling, or a closed form evaluated in fp64."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest

import synth
from synth import bf16_bits_to_f32, f32_to_bf16_bits


def _layer(T=3, D=256, E=16, K=2, I=128, S=128, act="f32", seed=5):
    cfg = synth.small_config(T=T, D=D, E=E, K=K, I=I, S=S, act=act, seed=seed)
    return cfg, synth.make_layer(cfg), synth.make_x(cfg)


def _with_blob(layer, order):
    """A copy of `layer` whose blob holds the records of experts `order` (in
    that order), with the matching expert -> record table."""
    st = layer.stride
    blob = np.concatenate([layer.blob[e * st:(e + 1) * st] for e in order])
    slot = np.full(layer.E, -1, dtype=np.int16)
    for r, e in enumerate(order):
        slot[e] = r
    return dataclasses.replace(layer, blob=blob, expert_slot=slot, n_slots=len(order))


# ------------------------------------------------------------ expert table

def test_identity_table_equals_no_table(orc):
    cfg, layer, x = _layer()
    a = orc.block_forward(layer, x)
    b = orc.block_forward(_with_blob(layer, list(range(layer.E))), x)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_permuted_records_with_their_table(orc):
    cfg, layer, x = _layer(seed=6)
    order = list(np.random.default_rng(0).permutation(layer.E))
    a = orc.block_forward(layer, x)
    b = orc.block_forward(_with_blob(layer, order), x)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_resident_subset_and_absent_expert(orc):
    """A blob holding only the experts the tokens select gives the same
    result; removing one selected expert is reported."""
    cfg, layer, x = _layer(seed=7)
    out, idx, w = orc.block_forward(layer, x)
    chosen = sorted(set(int(e) for e in idx.ravel()))
    sub = _with_blob(layer, chosen[::-1])
    for u, v in zip((out, idx, w), orc.block_forward(sub, x)):
        assert np.array_equal(u, v)
    missing = _with_blob(layer, chosen[1:])
    with pytest.raises(orc.ExpertNotResident):
        orc.block_forward(missing, x)


# ------------------------------------------------------------ router scale

def test_router_scale_sqrt_d_is_the_identity(orc):
    """D = 64: router_scale = 8 = sqrt(D) and 1/sqrt(D) = 1/8 exactly, so the
    router reads x itself."""
    cfg, layer, x = _layer(D=64, I=64, S=64)
    a = orc.block_forward(layer, x)
    scaled = dataclasses.replace(layer, router_scale=f32_to_bf16_bits(np.full(64, 8.0, np.float32)))
    for u, v in zip(a, orc.block_forward(scaled, x)):
        assert np.array_equal(u, v)


def test_router_scale_doubles_the_logits(orc):
    """router_scale = 2 sqrt(D) doubles every router input exactly, hence every
    logit: the same top-k, and weights softmax(2 l) of the selected logits."""
    cfg, layer, x = _layer(D=64, I=64, S=64, seed=8)
    l1 = orc.router_logits(layer.router, x)
    scaled = dataclasses.replace(layer, router_scale=f32_to_bf16_bits(np.full(64, 16.0, np.float32)))
    _, idx, w = orc.block_forward(scaled, x)
    ridx, _ = orc.topk_softmax(l1, cfg.K)
    assert np.array_equal(idx, ridx)
    sel = np.take_along_axis(l1.astype(np.float64), ridx, axis=1) * 2.0
    ew = np.exp(sel - sel[:, :1])
    assert np.allclose(w, ew / ew.sum(1, keepdims=True), rtol=1e-6, atol=1e-7)


# --------------------------------------------------------------- post norm

def test_post_norm_closed_form(orc):
    """fp32 activations, lambda = 0.5 (exact): the plain block gives y = 2 out;
    with the post-FFN norm (weights w) out becomes 0.5 * y / rms(y) * w
    (fp64 closed form, fp32 rounding)."""
    cfg, layer, x = _layer(seed=9)
    out, _, _ = orc.block_forward(layer, x)
    y = 2.0 * out.astype(np.float64)
    wv = np.random.default_rng(1).uniform(0.5, 1.5, cfg.D).astype(np.float32)
    wb = f32_to_bf16_bits(wv)
    normed = dataclasses.replace(layer, post_norm=wb, post_eps=1e-6)
    got, _, _ = orc.block_forward(normed, x)
    r = 1.0 / np.sqrt((y * y).mean(axis=1, keepdims=True) + 1e-6)
    ref = 0.5 * y * r * bf16_bits_to_f32(wb).astype(np.float64)
    assert np.max(np.abs(got - ref) / (np.abs(ref) + 1e-6)) < 2e-5


def test_post_norm_weight_two_doubles_unit_weight(orc):
    cfg, layer, x = _layer(seed=10)
    one = dataclasses.replace(layer, post_norm=f32_to_bf16_bits(np.ones(cfg.D, np.float32)))
    two = dataclasses.replace(layer, post_norm=f32_to_bf16_bits(np.full(cfg.D, 2.0, np.float32)))
    a, _, _ = orc.block_forward(one, x)
    b, _, _ = orc.block_forward(two, x)
    assert np.array_equal(b, 2.0 * a)


# ---------------------------------------------------- gated shared expert

def test_zero_gate_halves_the_shared_branch(orc):
    """With every routing weight 0 (per-expert scale 0) the output is the
    shared branch alone; a zero gate vector gives sigmoid(0) = 1/2 exactly."""
    cfg, layer, x = _layer(seed=11)
    quiet = dataclasses.replace(layer, per_expert_scale=np.zeros(cfg.E, np.float32))
    a, _, _ = orc.block_forward(quiet, x)
    gated = dataclasses.replace(quiet, shared_expert_gate=np.zeros(cfg.D, np.uint16))
    b, _, _ = orc.block_forward(gated, x)
    assert np.array_equal(b, 0.5 * a)


def test_gate_value_closed_form(orc):
    """x = 1/8 everywhere, gate vector 1/64 everywhere (D = 64): the gate is
    sigmoid(1/8); the gated shared-only output is that multiple of the plain
    one (fp64 sigmoid, fp32 rounding)."""
    cfg, layer, _ = _layer(T=1, D=64, I=64, S=64, seed=12)
    x = np.full((1, 64), 0.125, np.float32)
    quiet = dataclasses.replace(layer, per_expert_scale=np.zeros(cfg.E, np.float32))
    a, _, _ = orc.block_forward(quiet, x)
    gated = dataclasses.replace(quiet, shared_expert_gate=f32_to_bf16_bits(np.full(64, 1 / 64, np.float32)))
    b, _, _ = orc.block_forward(gated, x)
    g = 1.0 / (1.0 + np.exp(-0.125))
    assert np.allclose(b, g * a.astype(np.float64), rtol=3e-7, atol=1e-12)
