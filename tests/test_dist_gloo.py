"""Token-sharded multi-rank path on CPU: two gloo ranks, each with its own
shard.  The all-reduced per-expert sums must reproduce the aux loss of the
whole batch (f_i counts every choice before drops, so sharding the tokens
and their capacities does not change it), and the step-time reduction is
the maximum over ranks."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shard(seed, T, d, E):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, d, generator=g)
    W = torch.randn(E, d, generator=g) * 0.3
    return x, W


def _worker(rank, world, port, out_dir):
    import oracle
    from top_routing_expert_02_b300 import dist as mdist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    T, d, E, k, alpha = 50 + 7 * rank, 16, 8, 2, 0.01
    x, _ = _shard(100 + rank, T, d, E)
    _, W = _shard(7, 1, d, E)                       # same router on every rank
    idx, _, ps = oracle.route(oracle.router_logits(x, W), k)
    cap = oracle.capacity(T, E, 1.0)                # per-shard capacity
    counts, _, _, _ = oracle.dispatch(idx, E, cap)
    c, p, t = mdist.global_aux_inputs(torch.from_numpy(counts), torch.from_numpy(ps), T)
    loss = oracle.aux_loss(c.numpy(), p.numpy().astype(np.float64), t, alpha)
    # the host-sync-free form (total token count known): the same sums
    c2, p2, t2 = mdist.global_aux_inputs(torch.from_numpy(counts), torch.from_numpy(ps), T, T_total=50 + 57)
    same = float(torch.equal(c, c2) and torch.equal(p, p2) and t2 == t)
    worst = mdist.max_over_ranks(1.0 + rank)
    np.save(os.path.join(out_dir, f"r{rank}.npy"), np.array([loss, t, worst, same]))
    dist.destroy_process_group()


def test_two_gloo_ranks_reproduce_whole_batch_aux_loss(tmp_path):
    import oracle
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    res = [np.load(tmp_path / f"r{r}.npy") for r in range(world)]
    d, E, k, alpha = 16, 8, 2, 0.01
    xs = [_shard(100 + r, 50 + 7 * r, d, E)[0] for r in range(world)]
    _, W = _shard(7, 1, d, E)
    x = torch.cat(xs)
    idx, _, ps = oracle.route(oracle.router_logits(x, W), k)
    counts, _, _, _ = oracle.dispatch(idx, E, x.shape[0])
    whole = oracle.aux_loss(counts, ps, x.shape[0], alpha)
    for r in res:
        assert int(r[1]) == x.shape[0]
        assert abs(r[0] - whole) <= 1e-6 * whole     # prob sums cross ranks in fp32
        assert r[2] == 2.0
        assert r[3] == 1.0
