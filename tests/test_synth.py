"""The seeded generator: determinism, the distributions it states, the layout
it writes, and the calibration of the skewed-routing workload."""
from __future__ import annotations

import numpy as np

import synth


def test_generator_is_deterministic_and_keyed():
    cfg = synth.small_config(T=3, D=128, E=4, K=2, I=64, S=64, act="bf16", seed=5)
    a, b = synth.make_layer(cfg), synth.make_layer(cfg)
    assert np.array_equal(a.blob, b.blob) and np.array_equal(a.router.w, b.router.w)
    c = synth.make_layer(cfg, layer=1)
    assert not np.array_equal(a.blob, c.blob)
    assert np.array_equal(synth.make_x(cfg), synth.make_x(cfg))


def test_stated_distributions():
    cfg = synth.small_config(T=64, D=512, E=8, K=2, I=128, S=128, act="bf16", seed=1)
    layer = synth.make_layer(cfg)
    s = synth.bf16_bits_to_f32(layer.shared_gate.s)
    b = synth.bf16_bits_to_f32(layer.shared_gate.b)
    assert s.min() >= 0.005 * (1 - 2 ** -8) and s.max() <= 0.02 * (1 + 2 ** -8)
    assert b.min() >= -0.08 * (1 + 2 ** -8) and b.max() <= 0.0
    q = np.stack([(layer.shared_gate.w >> (4 * j)) & 15 for j in range(8)])
    counts = np.bincount(q.ravel(), minlength=16) / q.size
    assert np.all(np.abs(counts - 1 / 16) < 0.01)
    x = synth.bf16_bits_to_f32(synth.make_x(cfg))
    assert abs(x.mean()) < 0.05 and abs(x.std() - 1) < 0.05


def test_skewed_routing_calibration(orc):
    """The skewed-decode workload puts about 30% of its T*K slots on the 8
    most popular experts (the workload's own description)."""
    cfg = synth.CONFIGS[3]
    layer = synth.make_layer(cfg)
    x = synth.bf16_bits_to_f32(synth.make_x(cfg))
    idx, _ = orc.topk_softmax(orc.router_logits(layer.router, x), cfg.K)
    cnt = np.bincount(idx.ravel(), minlength=cfg.E)
    share = np.sort(cnt)[::-1][:8].sum() / idx.size
    assert 0.27 <= share <= 0.33, share
    assert 100 <= (cnt > 0).sum() <= 126
