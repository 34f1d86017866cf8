"""Expert-parallel MoE layer forward across ranks (host side, torch.distributed).

The expert-parallelism tutorial "专家并行：混合专家模型的分布式训练方案" §2.1 splits
the forward into gate decision, dispatch plan, All-to-All dispatch, local
expert compute and All-to-All combine; the fine-grained EP deployment guide
"细粒度专家并行部署实践与优化指南" §七 gives the same steps as pseudo-code.  Here:

  * rank r owns the contiguous expert block [r*E_loc, (r+1)*E_loc), E_loc = E/G,
    so the rows a rank sends to one destination are one contiguous slice of
    its expert-major x_perm (no packing before the exchange);
  * every rank routes and dispatches its own tokens with a per-rank capacity
    (round(T_local / E * cf): the token-group reading of capacity);
  * exchange 1: per-expert row counts (all_to_all of G*E_loc ints);
  * exchange 2: the x_perm rows and their gates (all_to_all_single with
    uneven splits); the received rows come grouped by source rank and are
    regrouped by local expert with one row permutation;
  * the local experts run the grouped GEMMs on their rows;
  * the inverse permutation and the reverse all_to_all_single return each
    y_perm row to the rank and the slot it came from; the combine is local;
  * the aux loss is global: one all-reduce of 2E + 1 numbers (dist.py).

The local steps go through an ``ops`` object (route, dispatch, permute_rows,
expert_ffn, combine, aux_loss): :class:`LibraryOps` runs the CUDA library;
tests may supply another implementation of the same six calls.  Host synchronisation
happens once per layer, to turn the received counts into split sizes.

``host_exchange=True`` stages every exchange through host memory (device
tensors are copied to the host, exchanged, and copied back), for process
groups whose backend moves host tensors only (gloo); the device-side steps
are unchanged.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch
import torch.distributed as dist

from .dist import global_aux_inputs

__all__ = ["LibraryOps", "EPResult", "ep_forward", "expert_block"]


class LibraryOps:
    """The local steps on the GPU through the CUDA library."""

    def route(self, x, W, b, k, renorm):
        from . import route
        return route(x, W, b, k, renorm)

    def dispatch(self, idx, gate, x, E, cap):
        from . import dispatch
        D = dispatch(idx, gate, x, E, cap)
        return dict(counts=D.counts, kept=D.kept, offsets=D.offsets, slot_row=D.slot_row, row_token=D.row_token,
                    row_gate=D.row_gate, x_perm=D.x_perm)

    def permute_rows(self, src, index):
        from . import permute_rows
        return permute_rows(src.contiguous(), index.to(device=src.device, dtype=torch.int32).contiguous())

    def expert_ffn(self, rows, offsets, kept, w1, w2, gate, act):
        from . import expert_ffn
        R = rows.shape[0]
        _, y = expert_ffn(rows, offsets.to(rows.device), kept.to(rows.device), w1, w2, gate, act, R)
        return y[:R]

    def combine(self, y_perm, slot_row):
        from . import combine
        return combine(y_perm, slot_row)

    def aux_loss(self, counts, prob_sum, T, alpha):
        from . import aux_loss
        return aux_loss(counts.contiguous(), prob_sum.contiguous(), T, alpha)


def expert_block(E: int, world: int, rank: int):
    """The experts rank `rank` owns: [lo, hi)."""
    if E % world:
        raise ValueError("the expert count must divide evenly over the ranks")
    n = E // world
    return rank * n, (rank + 1) * n


@dataclass
class EPResult:
    y: torch.Tensor            # [T_local, d] this rank's layer output
    loss: torch.Tensor         # global aux loss (fp32 scalar tensor)
    counts: torch.Tensor       # this rank's per-expert assignment counts (before drops)
    recv_rows: int             # rows this rank's experts processed


def _bytes_view(t: torch.Tensor) -> torch.Tensor:
    """Rows of t as raw bytes [rows, row_bytes] (keeps the row split sizes)."""
    row_bytes = t.element_size() * (math.prod(t.shape[1:]) if t.dim() > 1 else 1)
    return t.contiguous().view(torch.uint8).reshape(t.shape[0], row_bytes)


def _a2a(out, inp, out_splits, in_splits, group, host=False):
    if not host:
        dist.all_to_all_single(out, inp, out_splits, in_splits, group=group)
        return
    src = _bytes_view(inp).cpu()
    dst = torch.empty((out.shape[0], src.shape[1]), dtype=torch.uint8)
    dist.all_to_all_single(dst, src, out_splits, in_splits, group=group)
    out.copy_(dst.view(out.dtype).reshape(out.shape))


def ep_forward(x, W, b, w1_local, w2_local, *, k: int, cap: int, act: str, renorm: bool = True, alpha: float = 0.01,
               group=None, ops=None, host_exchange: bool = False) -> EPResult:
    """One expert-parallel layer forward (module docstring).  x [T_local, d] is
    this rank's tokens; W [E, d] (and b) the router, the same on every rank;
    w1_local / w2_local this rank's expert block of w1 [E, N1, d] / w2 [E, d, F]."""
    ops = ops or LibraryOps()
    G = dist.get_world_size(group)
    rank = dist.get_rank(group)
    E = W.shape[0]
    lo, hi = expert_block(E, G, rank)
    El = hi - lo
    if w1_local.shape[0] != El or w2_local.shape[0] != El:
        raise ValueError("w1_local / w2_local must hold this rank's expert block")
    T = x.shape[0]
    dev = x.device

    # local gate decision and dispatch plan (per-rank capacity)
    idx, gate, prob_sum = ops.route(x, W, b, k, renorm)
    D = ops.dispatch(idx, gate, x, E, cap)
    kept = D["kept"].to("cpu", torch.int64)
    offsets = D["offsets"].to("cpu", torch.int64)

    # exchange 1: how many rows of each of its experts every rank receives from us
    if host_exchange:
        recv_counts = torch.empty((G, El), dtype=torch.int64)
        dist.all_to_all_single(recv_counts, kept.view(G, El).contiguous(), group=group)
    else:
        send_counts = kept.view(G, El).to(dev)
        recv_dev = torch.empty_like(send_counts)
        dist.all_to_all_single(recv_dev, send_counts, group=group)   # equal splits: El counts per rank
        recv_counts = recv_dev.to("cpu")                              # [source rank, local expert]

    in_splits = [int(offsets[(r + 1) * El] - offsets[r * El]) for r in range(G)]
    out_splits = [int(recv_counts[s].sum()) for s in range(G)]
    n_recv = sum(out_splits)
    A = int(offsets[E])

    # exchange 2: rows and their gates (x_perm is expert-major, so each destination is one slice)
    d = x.shape[1]
    x_send = D["x_perm"][:A].contiguous()
    g_send = D["row_gate"][:A].contiguous()
    rdt = x_send.dtype
    x_recv = torch.empty((n_recv, d), dtype=rdt, device=dev)
    g_recv = torch.empty((n_recv,), dtype=g_send.dtype, device=dev)
    _a2a(x_recv, x_send, out_splits, in_splits, group, host_exchange)
    _a2a(g_recv, g_send, out_splits, in_splits, group, host_exchange)

    # regroup: received [src][local expert] blocks -> [local expert][src] segments;
    # every received row gets the key (local expert, src) of its block, and a
    # stable sort of the keys is the permutation (rows keep their order inside a block)
    block_key = (torch.arange(El, dtype=torch.int64)[None, :] * G + torch.arange(G, dtype=torch.int64)[:, None])
    row_key = torch.repeat_interleave(block_key.reshape(-1), recv_counts.reshape(-1).to(torch.int64))
    perm = torch.argsort(row_key, stable=True)
    kept_loc = recv_counts.sum(0).to(torch.int32)
    off_loc = torch.zeros(El + 1, dtype=torch.int32)
    off_loc[1:] = torch.cumsum(kept_loc, 0)

    if n_recv > 0:
        pdev = perm.to(dev)
        rows = ops.permute_rows(x_recv, pdev)
        # the gates ride the same permutation as 16-byte rows (gate, 0, 0, 0)
        wide = torch.zeros((n_recv, 4), dtype=g_recv.dtype, device=dev)
        wide[:, 0] = g_recv
        gates = ops.permute_rows(wide, pdev)[:, 0].contiguous()
        y_loc = ops.expert_ffn(rows, off_loc.to(dev), kept_loc.to(dev), w1_local, w2_local, gates, act)
        inv = torch.empty_like(perm)
        inv[perm] = torch.arange(n_recv, dtype=torch.int64)
        y_back = ops.permute_rows(y_loc.contiguous(), inv.to(dev))
    else:
        y_back = torch.empty((0, d), dtype=rdt, device=dev)

    # reverse exchange: every row returns to its sender, in the order it was sent
    y_perm = torch.empty((max(A, 1), d), dtype=y_back.dtype, device=dev)
    _a2a(y_perm[:A], y_back.contiguous(), in_splits, out_splits, group, host_exchange)
    y = ops.combine(y_perm, D["slot_row"])

    # global aux loss over every rank's tokens
    if host_exchange:
        c, p, t = global_aux_inputs(D["counts"].cpu(), prob_sum.cpu(), T, group)
        c, p = c.to(D["counts"].device), p.to(prob_sum.device)
    else:
        c, p, t = global_aux_inputs(D["counts"], prob_sum, T, group)
    loss = ops.aux_loss(c, p, t, alpha)
    return EPResult(y=y, loss=loss, counts=D["counts"], recv_rows=n_recv)
