"""The expert-parallel layer (top_routing_expert_02_b300.ep) through the CUDA
library on one GPU: a one-rank NCCL group, where the exchange is a copy and
the regrouping an identity permutation, must reproduce MoEPlan bit for bit
and the oracle's layer within the bf16 bar; and moe_permute_rows against
torch indexing."""
import pytest
import torch
import torch.distributed as dist

import top_routing_expert_02_b300 as moe
from top_routing_expert_02_b300 import synth
from top_routing_expert_02_b300.ep import ep_forward

from moe_cases import compare_output, make_case, run_oracle

pytestmark = pytest.mark.gpu


def test_permute_rows_is_exact():
    g = torch.Generator(device="cuda").manual_seed(3)
    src = torch.randn(300, 256, device="cuda", generator=g).to(torch.bfloat16)
    index = torch.randint(0, 300, (517,), device="cuda", generator=g, dtype=torch.int64).to(torch.int32)
    out = moe.permute_rows(src, index)
    moe.check()
    assert torch.equal(out, src[index.long()])
    wide = torch.randn(50, 4, device="cuda", generator=g)
    idx2 = torch.randperm(50, device="cuda", generator=g).to(torch.int32)
    assert torch.equal(moe.permute_rows(wide, idx2), wide[idx2.long()])


def test_one_rank_expert_parallel_layer_equals_the_plan():
    cfg = synth.MoEConfig("ep1", 1500, 256, 8, 2, 384, "swiglu", 1.25, "bf16")
    case = make_case(cfg)
    store = dist.HashStore()
    dist.init_process_group("nccl", store=store, rank=0, world_size=1)
    try:
        res = ep_forward(case["x"], case["W"], case["b"], case["w1"], case["w2"], k=cfg.k, cap=case["cap"],
                         act=cfg.act)
        moe.check()
    finally:
        dist.destroy_process_group()
    plan = moe.MoEPlan(cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.act, torch.bfloat16, case["cap"], "cuda", cfg.alpha,
                       cfg.renorm)
    plan.run(case["x"], case["W"], case["b"], case["w1"], case["w2"])
    moe.check()
    assert torch.equal(res.y, plan.y)
    assert abs(float(res.loss) - float(plan.loss.item())) <= 1e-6 * float(plan.loss.item())
    assert res.recv_rows == int(plan.disp.offsets[-1].item())
    ref = run_oracle(case)                       # and directly against the oracle's layer
    assert res.recv_rows == int(ref["kept"].sum())
    compare_output(plan, ref, cfg.dtype)
