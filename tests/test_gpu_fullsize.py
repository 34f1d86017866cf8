"""Full-size parity on every workload, in the launch configuration bench.py
times (MoEPlan.run): routing and dispatch bit-exact over all T tokens; the
layer output against the oracle (which computes tokens one by one) on tokens
that cover every 128-row tile of every expert segment (up to a budget; the
largest workload samples the tiles evenly) plus tokens with dropped slots and
one with none kept, pooled and token by token; every kept row of h and y_perm
against a per-expert fp32 reference on the device, row by row; y against the
sum of its y_perm rows bit for bit; and the aux loss."""
import numpy as np
import pytest
import torch

import top_routing_expert_02_b300 as moe
from top_routing_expert_02_b300 import synth

from moe_cases import (check_expert_rows_on_device, compare_dispatch, compare_output, compare_routing, make_case,
                       run_gpu, run_oracle, tile_tokens)

pytestmark = pytest.mark.gpu

FULL = ["e8_swiglu", "e16_gelu_hot2", "e64_zipf", "e128_top8_T512", "e128_top8_T2048", "e128_top8_T8192",
        "e128_top8_T32768"]


# the oracle's cost per token grows with k*d*F; keep each test near a minute
ORACLE_TOKENS = {"e8_swiglu": 400, "e16_gelu_hot2": 400, "e64_zipf": 1200, "e128_top8_T512": 600,
                 "e128_top8_T2048": 300, "e128_top8_T8192": 200, "e128_top8_T32768": 160}


def sample_tokens(plan, budget: int):
    """One token from every 128-row GEMM tile of every expert (evenly thinned
    to the budget when there are more tiles), plus a few tokens with dropped
    slots and one with none kept."""
    slot_row = plan.disp.slot_row.cpu().numpy()
    tiles = tile_tokens(plan)
    if len(tiles) > budget:
        tiles = [tiles[i] for i in np.linspace(0, len(tiles) - 1, budget).astype(int)]
    toks = set(tiles)
    partial = np.nonzero((slot_row < 0).any(1) & (slot_row >= 0).any(1))[0]
    none = np.nonzero((slot_row < 0).all(1))[0]
    toks.update(partial[:3].tolist())
    toks.update(none[:1].tolist())
    return sorted(toks)


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name):
    cfg = synth.workload(name)
    case = make_case(cfg)
    plan = run_gpu(case)
    check_expert_rows_on_device(plan, case["x"], case["w1"], case["w2"], cfg.act)
    toks = sample_tokens(plan, ORACLE_TOKENS[name])
    ref = run_oracle(case, tokens=toks)
    compare_routing(plan, ref, cfg.dtype)
    compare_dispatch(plan, ref, case["x_h"])
    compare_output(plan, ref, cfg.dtype)
    del plan, case
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["e8_swiglu", "e128_top8_T32768"])
def test_full_size_gathered_up_projection(name):
    """The fused-gather layer (no x_perm) at full size: same checks."""
    cfg = synth.workload(name)
    case = make_case(cfg)
    plan = moe.MoEPlan(cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.act, torch.bfloat16, case["cap"], case["x"].device,
                       cfg.alpha, cfg.renorm, gather=True)
    run_gpu(case, plan)
    toks = sample_tokens(plan, ORACLE_TOKENS[name] // 2)
    ref = run_oracle(case, tokens=toks)
    compare_routing(plan, ref, cfg.dtype)
    compare_dispatch(plan, ref)
    compare_output(plan, ref, cfg.dtype)
    del plan, case
    torch.cuda.empty_cache()
