"""The expert-parallel layer (top_routing_expert_02_b300.ep) with the CUDA
library doing every local step on both sides of a real two-rank exchange:
two processes share cuda:0, join a gloo group, and stage the all-to-all
exchanges through host memory (ep_forward(host_exchange=True)); their kernels
never wait on one another.  Each rank's output must equal the oracle's layer
on that rank's tokens (per-rank capacity) within the bf16 bar, pooled and per
token, and the aux loss the oracle's over both ranks' tokens; every kept row
is processed by exactly one expert owner.  Not measured on more than one GPU:
each box of this pool has one."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu

WORLD = 2
CFG = dict(name="ep2", T=1200, d=256, E=8, k=2, F=384, act="swiglu", cf=1.25, dtype="bf16")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(rank):
    """Rank-local tokens (seed 100 + rank; more tokens on rank 1), the shared
    router and the full expert weights (identical on every rank)."""
    import oracle
    from top_routing_expert_02_b300 import synth
    cfg = synth.MoEConfig(**CFG).replace(T=CFG["T"] + 137 * rank, seed=100 + rank)
    ri = synth.condition_near_ties(cfg, synth.make_routing_inputs(cfg), oracle.router_logits)
    shared = synth.MoEConfig(**CFG)
    r0 = synth.make_routing_inputs(shared)
    w1, w2 = synth.make_expert_weights(shared, device="cuda")
    return cfg, ri.x, r0.W, w1, w2


def _worker(rank, port, out_dir):
    import torch.distributed as dist
    import top_routing_expert_02_b300 as moe
    from top_routing_expert_02_b300.ep import ep_forward, expert_block
    torch.cuda.set_device(0)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        cfg, x, W, w1, w2 = _inputs(rank)
        lo, hi = expert_block(cfg.E, WORLD, rank)
        cap = moe.capacity(cfg.T, cfg.E, cfg.cf)
        res = ep_forward(x.cuda(), W.cuda(), None, w1[lo:hi].contiguous(), w2[lo:hi].contiguous(), k=cfg.k,
                         cap=cap, act=cfg.act, host_exchange=True)
        moe.check()
        np.save(os.path.join(out_dir, f"y{rank}.npy"), res.y.float().cpu().numpy())
        np.save(os.path.join(out_dir, f"m{rank}.npy"), np.array([float(res.loss), res.recv_rows]))
    finally:
        dist.destroy_process_group()


def test_two_rank_expert_parallel_layer_through_the_library(tmp_path):
    import oracle
    import top_routing_expert_02_b300 as moe
    mp.start_processes(_worker, args=(_free_port(), str(tmp_path)), nprocs=WORLD, start_method="spawn")
    shards = [_inputs(r) for r in range(WORLD)]
    W, w1h, w2h = shards[0][2], shards[0][3].cpu(), shards[0][4].cpu()
    whole = torch.cat([s[1] for s in shards])
    idx, _, ps = oracle.route(oracle.router_logits(whole, W), CFG["k"])
    counts, _, _, _ = oracle.dispatch(idx, CFG["E"], whole.shape[0])
    loss_whole = oracle.aux_loss(counts, ps, whole.shape[0], 0.01)
    recv_total = kept_total = 0
    for r, (cfg, x, _, _, _) in enumerate(shards):
        cap = moe.capacity(cfg.T, cfg.E, cfg.cf)
        ref = oracle.forward(x, W, None, w1h, w2h, k=cfg.k, cap=cap, act=cfg.act)
        y = np.load(tmp_path / f"y{r}.npy").astype(np.float64)
        err = np.linalg.norm(y - ref["y"]) / np.linalg.norm(ref["y"])
        norms = np.linalg.norm(ref["y"], axis=1)
        live = norms > 0
        worst = float((np.linalg.norm(y - ref["y"], axis=1)[live] / norms[live]).max())
        print(f"[ep2] rank {r}: y rel Frobenius err {err:.3e}, worst token {worst:.3e}")
        assert err <= 2e-2 and worst <= 2e-2
        assert not np.any(y[~live])                     # fully dropped tokens: zero rows
        assert ref["n_dropped"] > 0                     # the per-rank capacity bites
        loss, recv = np.load(tmp_path / f"m{r}.npy")
        assert abs(loss - loss_whole) <= 1e-5 * loss_whole
        recv_total += int(recv)
        kept_total += int(ref["kept"].sum())
    assert recv_total == kept_total
