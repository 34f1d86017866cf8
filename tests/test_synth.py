"""The seeded input generator: determinism, shapes, and the workload
properties its recipe promises (near-tie margin, hot experts, Zipf skew)."""
import numpy as np
import pytest
import torch

import oracle
from top_routing_expert_02_b300 import synth


def test_routing_inputs_are_deterministic():
    cfg = synth.workload("tiny_fp32")
    a, b = synth.make_routing_inputs(cfg), synth.make_routing_inputs(cfg)
    assert torch.equal(a.x, b.x) and torch.equal(a.W, b.W) and a.b is None
    assert a.x.shape == (64, 128) and a.x.dtype == torch.float32 and a.W.shape == (8, 128)
    assert abs(float(a.W.std()) - 0.02) < 0.003


def test_expert_weights_deterministic_and_scaled():
    cfg = synth.workload("tiny_fp32")
    w1, w2 = synth.make_expert_weights(cfg)
    v1, v2 = synth.make_expert_weights(cfg)
    assert torch.equal(w1, v1) and torch.equal(w2, v2)
    assert w1.shape == (8, 256, 128) and w2.shape == (8, 128, 256)
    assert abs(float(w1.std()) * 128 ** 0.5 - 1) < 0.02
    assert abs(float(w2.std()) * 256 ** 0.5 - 1) < 0.02
    cfg2 = cfg.replace(act="swiglu", dtype="bf16")
    u1, u2 = synth.make_expert_weights(cfg2)
    assert u1.shape == (8, 512, 128) and u1.dtype == torch.bfloat16


def test_bf16_rounding_is_nearest_even():
    cfg = synth.workload("tiny_fp32").replace(dtype="bf16")
    x32 = synth.make_routing_inputs(synth.workload("tiny_fp32")).x
    xb = synth.make_routing_inputs(cfg).x
    assert xb.dtype == torch.bfloat16
    assert torch.equal(xb, x32.to(torch.bfloat16))


@pytest.mark.parametrize("name", ["tiny_fp32", "e64_zipf"])
def test_near_tie_conditioning_leaves_margin(name):
    cfg = synth.workload(name)
    ri = synth.condition_near_ties(cfg, synth.make_routing_inputs(cfg), oracle.router_logits)
    L = oracle.router_logits(ri.x, ri.W, ri.b)
    top = -np.sort(-L, axis=1)[:, :cfg.k + 1]
    assert (np.diff(-top, axis=1) >= 1e-3).all()
    again = synth.condition_near_ties(cfg, synth.make_routing_inputs(cfg), oracle.router_logits)
    assert torch.equal(again.x, ri.x) and again.redrawn == ri.redrawn


def test_hot_experts_get_three_times_mean_load():
    cfg = synth.workload("e16_gelu_hot2")
    ri = synth.make_routing_inputs(cfg)
    idx, _, _ = oracle.route(oracle.router_logits(ri.x, ri.W, ri.b), cfg.k)
    counts = np.bincount(idx.ravel(), minlength=cfg.E)
    mean = cfg.T * cfg.k / cfg.E
    assert 2.8 < counts[:2].mean() / mean < 3.2
    cap = oracle.capacity(cfg.T, cfg.E, cfg.cf)
    assert cap == 512 and (counts > cap).all()         # every expert saturates


def test_zipf_skew_is_heavy():
    cfg = synth.workload("e64_zipf")
    ri = synth.make_routing_inputs(cfg)
    idx, _, _ = oracle.route(oracle.router_logits(ri.x, ri.W, ri.b), cfg.k)
    counts = np.bincount(idx.ravel(), minlength=cfg.E)
    assert counts.argmax() == 0
    assert counts.max() / counts.mean() > 10


def test_near_tie_conditioning_for_group_limited_routing():
    """With a routing variant's own gap function, every decision it takes
    (group scores, then the logits inside the kept groups) clears the margin."""
    cfg = synth.MoEConfig("grp", 512, 128, 32, 4, 128, "swiglu", 1.25, "bf16")
    gaps = lambda L: oracle.decision_gaps(L, cfg.k, 8, 2)
    ri = synth.condition_near_ties(cfg, synth.make_routing_inputs(cfg), oracle.router_logits, gaps_fn=gaps)
    L = oracle.router_logits(ri.x, ri.W, ri.b)
    assert (gaps(L) >= 1e-3).all()
    assert ri.redrawn > 0
    # decision_gaps without groups is the plain top-(k+1) test
    top = -np.sort(-L, axis=1)[:, :cfg.k + 1]
    np.testing.assert_array_equal(oracle.decision_gaps(L, cfg.k), np.diff(-top, axis=1).min(axis=1))
