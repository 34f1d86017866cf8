"""Full-size parity on every workload, in the launch configuration bench.py
times (MoEPlan.run): routing and dispatch bit-exact over all T tokens, the
layer output on sampled tokens against the oracle (which computes them one by
one), and the aux loss."""
import numpy as np
import pytest
import torch

import top_routing_expert_02_b300 as moe
from top_routing_expert_02_b300 import synth

from moe_cases import compare_dispatch, compare_output, compare_routing, make_case, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

FULL = ["e8_swiglu", "e16_gelu_hot2", "e64_zipf", "e128_top8_T512", "e128_top8_T2048", "e128_top8_T8192",
        "e128_top8_T32768"]


def sample_tokens(slot_row: np.ndarray, n: int = 16):
    """Evenly spread tokens plus a few with dropped slots and one with none kept."""
    T = slot_row.shape[0]
    toks = set(np.linspace(0, T - 1, n).astype(int).tolist())
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
    toks = sample_tokens(plan.disp.slot_row.cpu().numpy())
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
    toks = sample_tokens(plan.disp.slot_row.cpu().numpy())
    ref = run_oracle(case, tokens=toks)
    compare_routing(plan, ref, cfg.dtype)
    compare_dispatch(plan, ref)
    compare_output(plan, ref, cfg.dtype)
    del plan, case
    torch.cuda.empty_cache()
