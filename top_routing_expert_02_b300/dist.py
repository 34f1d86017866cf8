"""Token-sharded data parallelism across GPUs (host side, torch.distributed).

Each rank runs the whole layer forward on its own shard of tokens; routing,
dispatch, the expert FFN and the combine are per token and need no exchange.
Capacity is then per shard (round(T_shard / E * cf)).  The one quantity that
spans shards is the auxiliary load-balance loss of the expert-parallelism
tutorial "专家并行：混合专家模型的分布式训练方案" §5.1: f_i and P_i are means over
all tokens, so the per-expert assignment counts, the per-expert probability
sums and the token count are summed over ranks (one all-reduce of 2E + 1
numbers) before L = alpha * E * sum_i f_i P_i is formed.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

__all__ = ["global_aux_inputs", "global_aux_loss", "max_over_ranks"]


def global_aux_inputs(counts: torch.Tensor, prob_sum: torch.Tensor, T: int, group=None, T_total=None):
    """Sum this rank's counts [E], prob_sum [E] and T over all ranks.

    Returns (counts int32 [E], prob_sum fp32 [E], T_total) on the inputs' device.
    The probability sums travel as fp64 so the reduction adds no rounding of
    its own beyond the final conversion.  A caller that knows the total token
    count passes ``T_total``: then only the 2E sums are reduced and nothing
    waits on the host (no device-to-host read), so the step stays asynchronous."""
    parts = [counts.to(torch.float64), prob_sum.to(torch.float64)]
    if T_total is None:
        parts.append(torch.tensor([float(T)], dtype=torch.float64, device=counts.device))
    packed = torch.cat(parts)
    dist.all_reduce(packed, op=dist.ReduceOp.SUM, group=group)
    E = counts.numel()
    total = int(packed[2 * E].item()) if T_total is None else int(T_total)
    return packed[:E].round().to(torch.int32), packed[E:2 * E].to(torch.float32), total


def global_aux_loss(counts: torch.Tensor, prob_sum: torch.Tensor, T: int, alpha: float, group=None):
    """Aux loss of the union of all ranks' shards, computed by the library's
    moe_aux_loss on the reduced sums (device tensors)."""
    from . import aux_loss
    c, p, t = global_aux_inputs(counts, prob_sum, T, group)
    return aux_loss(c.contiguous(), p.contiguous(), t, alpha)


def max_over_ranks(value: float, device=None, group=None) -> float:
    """The largest of one float over all ranks (e.g. a step time)."""
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())
