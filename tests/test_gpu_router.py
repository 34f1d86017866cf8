"""GPU parity of the bf16 router (moe_route) on its own, on shapes chosen for
the fused tensor-core kernel's code paths: one CTA per tile with many K
blocks (the accumulators drained in chunks of four K blocks, including a
ragged last chunk), clusters of 2 to 4 CTAs splitting d, one or two 128-token
tiles per CTA in both accumulator layouts (three parts in one MMA, E <= 32;
one MMA per part above), expert counts that are not multiples of 16
(zero-padded weight rows), ragged token tails, a bias, and the largest
expert count (128) at top-8.  Indices bit-exact,
gates and probability sums within the gate bar of moe_cases, against the
oracle's fp64 router on the same stored inputs."""
import numpy as np
import pytest
import torch

import oracle
import top_routing_expert_02_b300 as moe
from top_routing_expert_02_b300 import synth

from moe_cases import GATE_RTOL

pytestmark = pytest.mark.gpu

C = synth.MoEConfig

CASES = {
    # 157 tiles > 148 SMs: one CTA per tile, 16 K blocks = 4 chunks
    "e64_chunks": C("r_e64_chunks", 20000, 1024, 64, 2, 64, "gelu", 0.0, "bf16"),
    # E = 128, top-8, 20 K blocks: 5 chunks, 150 tiles
    "e128_top8_chunks": C("r_e128_chunks", 19100, 1280, 128, 8, 64, "gelu", 0.0, "bf16"),
    # 8 tiles: clusters of 4 CTAs, 16 K blocks each (4 chunks), ragged tail of 104 tokens
    "e8_cluster8": C("r_e8_cl8", 1000, 4096, 8, 2, 64, "gelu", 0.0, "bf16"),
    # 10 K blocks over a cluster of 4: K ranges of 2 and 3 blocks
    "e16_cluster4_ragged_k": C("r_e16_cl4", 777, 640, 16, 2, 64, "gelu", 0.0, "bf16", bias="hot2"),
    # E = 40 (padded to 48 weight rows), 10 K blocks over one CTA: chunks 4, 4, 2
    "e40_pad": C("r_e40", 19000, 640, 40, 3, 64, "gelu", 0.0, "bf16"),
    # E = 100 (padded to 112), Zipf bias, top-6
    "e100_zipf": C("r_e100", 5000, 2048, 100, 6, 64, "gelu", 0.0, "bf16", bias="zipf"),
    # one token
    "one_token": C("r_one", 1, 512, 32, 4, 64, "gelu", 0.0, "bf16"),
    # two 128-token tiles per CTA, all three parts in one MMA (E <= 32)
    "e16_two_tiles": C("r_e16_2t", 8100, 512, 16, 2, 64, "gelu", 0.0, "bf16"),
    # two tiles per CTA, one MMA per part (32 < E <= 64), ragged last tile pair
    "e48_two_tiles": C("r_e48_2t", 16000, 1024, 48, 4, 64, "gelu", 0.0, "bf16", bias="zipf"),
}


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("renorm", [True, False])
def test_router_against_oracle(name, renorm):
    cfg = CASES[name]
    ri = synth.condition_near_ties(cfg, synth.make_routing_inputs(cfg), oracle.router_logits)
    x, W = ri.x.cuda(), ri.W.cuda()
    b = None if ri.b is None else ri.b.cuda()
    idx, gate, ps = moe.route(x, W, b, cfg.k, renorm)
    moe.check()
    ref_idx, ref_gate, ref_ps = oracle.route(oracle.router_logits(ri.x, ri.W, ri.b), cfg.k, renorm)
    assert np.array_equal(idx.cpu().numpy(), ref_idx), "top-k indices differ"
    g = gate.cpu().numpy().astype(np.float64)
    p = ps.cpu().numpy().astype(np.float64)
    eg = float(np.max(np.abs(g - ref_gate) / np.abs(ref_gate)))
    ep = float(np.max(np.abs(p - ref_ps) / np.abs(ref_ps)))
    print(f"[router] {name} renorm={renorm}: gate max rel err {eg:.3e}, prob_sum max rel err {ep:.3e}")
    np.testing.assert_allclose(g, ref_gate, rtol=GATE_RTOL["bf16"], atol=0)
    np.testing.assert_allclose(p, ref_ps, rtol=GATE_RTOL["bf16"], atol=1e-30)


def test_router_bitwise_run_to_run_and_logits_output():
    """Two calls give the same bits; the logits and log-sum-exp outputs of
    moe_route_ex match the oracle's fp64 logits within the gate bar."""
    cfg = CASES["e64_chunks"]
    ri = synth.condition_near_ties(cfg, synth.make_routing_inputs(cfg), oracle.router_logits)
    x, W = ri.x.cuda(), ri.W.cuda()
    T, E = cfg.T, cfg.E
    logits = torch.empty(T, E, device="cuda")
    lse = torch.empty(T, device="cuda")
    a = moe.route(x, W, None, cfg.k, True, logits=logits, lse=lse)
    a = [t.clone() for t in a]
    b = moe.route(x, W, None, cfg.k, True)
    moe.check()
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    L = oracle.router_logits(ri.x, ri.W)
    got = logits.cpu().numpy().astype(np.float64)
    err = np.max(np.abs(got - L)) / np.max(np.abs(L))
    print(f"[router] logits max abs err / max |l| {err:.3e}")
    assert err <= 1e-6
    np.testing.assert_allclose(lse.cpu().numpy(), oracle.logsumexp(L), rtol=GATE_RTOL["bf16"], atol=1e-6)


@pytest.mark.parametrize("kind", [1, 2])
def test_small_e_logits_and_lse_outputs_on_both_router_kernels(kind):
    """At E = 8 (with a bias) the tensor-core router (1) and the CUDA-core
    E <= 8 router (2) both write logits within 1e-6 of max |l| of the oracle's
    fp64 logits and the log-sum-exp within the gate bar, and repeat their
    bits run to run."""
    cfg = synth.MoEConfig("e8_logits", 1000, 512, 8, 2, 128, "gelu", 1.25, "bf16", bias="hot2")
    ri = synth.condition_near_ties(cfg, synth.make_routing_inputs(cfg), oracle.router_logits)
    x, W, b = ri.x.cuda(), ri.W.cuda(), ri.b.cuda()
    T, E = cfg.T, cfg.E
    moe.set_router_kernel(kind)
    try:
        outs = []
        for _ in range(2):
            logits = torch.empty(T, E, device="cuda")
            lse = torch.empty(T, device="cuda")
            r = moe.route(x, W, b, cfg.k, True, logits=logits, lse=lse)
            outs.append([t.clone() for t in r] + [logits, lse])
        moe.check()
    finally:
        moe.set_router_kernel(0)
    for u, v in zip(outs[0], outs[1]):
        assert torch.equal(u, v)
    L = oracle.router_logits(ri.x, ri.W, ri.b)
    got = outs[0][3].cpu().numpy().astype(np.float64)
    err = np.max(np.abs(got - L)) / np.max(np.abs(L))
    print(f"[router] kind {kind}: logits max abs err / max |l| {err:.3e}")
    assert err <= 1e-6
    np.testing.assert_allclose(outs[0][4].cpu().numpy(), oracle.logsumexp(L), rtol=GATE_RTOL["bf16"], atol=1e-6)
    ref_idx, ref_gate, _ = oracle.route(L, cfg.k, True)
    assert np.array_equal(outs[0][0].cpu().numpy(), ref_idx)
