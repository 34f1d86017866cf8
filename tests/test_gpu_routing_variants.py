"""GPU parity of the routing variants against the oracle: group-limited
top-k (every router kernel: the tensor-core router finished in its logits
kernel for E <= 64 and by the finishing kernel above, the CUDA-core E <= 8
router for bf16 x on request, the fused CUDA-core router for fp32 x and for
more than 128 experts), the per-token log-sum-exp and the router z-loss,
and the post-drop f_i aux loss.  Bars are in moe_cases."""
import numpy as np
import pytest
import torch

import top_routing_expert_02_b300 as moe
from top_routing_expert_02_b300 import synth

from moe_cases import (compare_dispatch, compare_output, compare_routing, compare_z_loss, make_case, run_gpu,
                       run_oracle)

pytestmark = pytest.mark.gpu

C = synth.MoEConfig

# name: (config, n_group, topk_group, post-drop aux)
CASES = {
    # E = 8: the tensor-core router finished in the logits kernel (and the CUDA-core E <= 8 router:
    # test_e8_variants_on_both_router_kernels), 2 groups of 4, one kept
    "e8_g2m1": (C("e8_g2m1", 2000, 256, 8, 2, 384, "swiglu", 1.25, "bf16"), 2, 1, False),
    # E = 32 (one MMA for the three weight parts), one group of 4 kept, no renormalisation, post-drop aux
    "e32_g8m1": (C("e32_g8m1", 1500, 128, 32, 4, 256, "gelu", 1.5, "bf16", renorm=False), 8, 1, True),
    # E = 64 (two MMAs per K step, still finished in the logits kernel), Zipf skew, 3 of 32 groups of 2,
    # k = 6 (every kept expert chosen)
    "e64_g32m3_zipf": (C("e64_g32m3_zipf", 3000, 128, 64, 6, 192, "swiglu", 1.25, "bf16", bias="zipf"), 32, 3,
                       True),
    # E = 128: logits kernel + the separate finishing kernel, 4 of 8 groups, top-8, dropless
    "e128_g8m4": (C("e128_g8m4", 600, 256, 128, 8, 128, "swiglu", 0.0, "bf16"), 8, 4, False),
    # E = 160 (above the tensor-core router: CUDA-core router), 32 groups of 5, 4 kept, top-16
    "e160_g32m4": (C("e160_g32m4", 300, 192, 160, 16, 128, "swiglu", 0.0, "bf16", renorm=False), 32, 4, False),
    # fused CUDA-core router, fp32 x: 4 groups of 16, 2 kept
    "f32_e64_g4m2": (C("f32_e64_g4m2", 700, 128, 64, 4, 128, "gelu", 1.25, "f32"), 4, 2, True),
    # CUDA-core router, bf16 x with E = 200: 8 groups of 25, 3 kept
    "bf16_e200_g8m3": (C("bf16_e200_g8m3", 400, 128, 200, 4, 128, "gelu", 2.0, "bf16"), 8, 3, False),
}

Z_BETA = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "these tests need a CUDA device"
    moe.lib()
    yield


def _plan(case, G, M, post):
    cfg = case["cfg"]
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    return moe.MoEPlan(cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.act, tdt, case["cap"], case["x"].device, cfg.alpha,
                       cfg.renorm, n_group=G, topk_group=M, z_beta=Z_BETA, aux_post_drop=post)


@pytest.mark.parametrize("name", list(CASES))
def test_routing_variant_layer(name):
    cfg, G, M, post = CASES[name]
    case = make_case(cfg, n_group=G, topk_group=M)
    plan = run_gpu(case, _plan(case, G, M, post))
    ref = run_oracle(case, n_group=G, topk_group=M, z_beta=Z_BETA, aux_post_drop=post)
    compare_routing(plan, ref, cfg.dtype)
    compare_dispatch(plan, ref, case["x_h"])
    compare_output(plan, ref, cfg.dtype)
    compare_z_loss(plan, ref, cfg.dtype)
    # the restriction really bites: some token's choice differs from plain top-k
    plain = run_oracle(case, tokens=[0])
    assert not np.array_equal(plain["idx"], ref["idx"])


@pytest.mark.parametrize("kind", [1, 2])
def test_e8_variants_on_both_router_kernels(kind):
    """The E = 8 group-limited case (with the log-sum-exp and the z-loss) on the
    tensor-core router (1) and on the CUDA-core E <= 8 router (2)."""
    cfg, G, M, post = CASES["e8_g2m1"]
    case = make_case(cfg, n_group=G, topk_group=M)
    moe.set_router_kernel(kind)
    try:
        plan = run_gpu(case, _plan(case, G, M, post))
    finally:
        moe.set_router_kernel(0)
    ref = run_oracle(case, n_group=G, topk_group=M, z_beta=Z_BETA, aux_post_drop=post)
    compare_routing(plan, ref, cfg.dtype)
    compare_dispatch(plan, ref, case["x_h"])
    compare_output(plan, ref, cfg.dtype)
    compare_z_loss(plan, ref, cfg.dtype)


def test_one_group_equals_moe_route_bitwise():
    """moe_route_ex with n_group = 1 (and with every group kept) writes what
    moe_route writes, bit for bit; lse is written either way."""
    cfg = CASES["e64_g32m3_zipf"][0]
    case = make_case(cfg)
    x, W, b = case["x"], case["W"], case["b"]
    base = moe.route(x, W, b, cfg.k)
    lse = torch.empty(cfg.T, dtype=torch.float32, device=x.device)
    for G, M in [(1, 1), (8, 8)]:
        got = moe.route(x, W, b, cfg.k, n_group=G, topk_group=M, lse=lse)
        for a, c in zip(base, got):
            assert torch.equal(a, c)
    moe.check()
    ref = run_oracle(case, tokens=[0])
    np.testing.assert_allclose(lse.cpu().numpy(), ref["lse"], rtol=2e-4)


def test_z_loss_of_zero_router_is_closed_form():
    """W = 0: every logit is 0, lse = ln E, z-loss = beta (ln E)^2."""
    T, d, E = 1000, 128, 64
    x = torch.randn(T, d, device="cuda").to(torch.bfloat16)
    W = torch.zeros(E, d, device="cuda")
    lse = torch.empty(T, dtype=torch.float32, device="cuda")
    moe.route(x, W, None, 2, lse=lse)
    z = moe.z_loss(lse, 0.5)
    moe.check()
    assert torch.allclose(lse, torch.full_like(lse, float(np.log(E))), rtol=1e-6)
    assert abs(z.item() - 0.5 * np.log(E) ** 2) <= 1e-6 * 0.5 * np.log(E) ** 2


def test_routing_variant_full_size_e128_top8_T8192():
    """Group-limited top-8 (8 groups of 16, 4 kept) with the z-loss on the
    128-expert, T = 8192 workload: routing and dispatch over every token,
    sampled outputs, both losses."""
    cfg = synth.workload("e128_top8_T8192")
    G, M = 8, 4
    case = make_case(cfg, n_group=G, topk_group=M)
    plan = run_gpu(case, _plan(case, G, M, False))
    slot = plan.disp.slot_row.cpu().numpy()
    toks = sorted(set(np.linspace(0, cfg.T - 1, 12).astype(int).tolist()))
    ref = run_oracle(case, tokens=toks, n_group=G, topk_group=M, z_beta=Z_BETA)
    compare_routing(plan, ref, cfg.dtype)
    compare_dispatch(plan, ref, case["x_h"])
    compare_output(plan, ref, cfg.dtype)
    compare_z_loss(plan, ref, cfg.dtype)
    assert (slot >= 0).all()


@pytest.mark.parametrize("T,offset", [(1, 0), (4097, 0), (4097, 1), (32768, 0), (33, 3)])
def test_z_loss_kernel_against_oracle_on_given_values(T, offset):
    """moe_z_loss on stored log-sum-exp values (aligned or not, any length)
    equals the oracle's z-loss of the same fp32 values."""
    import oracle
    g = torch.Generator().manual_seed(T + offset)
    host = (torch.rand(T + offset, generator=g) * 6.0 - 1.0).float()
    dev = host.cuda()[offset:]
    z = moe.z_loss(dev, 1e-3)
    moe.check()
    ref = oracle.z_loss(host[offset:].double().numpy(), 1e-3)
    assert abs(z.item() - ref) <= 1e-6 * abs(ref)
