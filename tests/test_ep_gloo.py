"""Expert-parallel layer forward (top_routing_expert_02_b300.ep) on CPU gloo
ranks.  The local steps run through a CPU implementation built on the oracle
(route, dispatch, per-row expert FFN, combine), so what is tested here is the
exchange: per-expert counts, the uneven row all-to-all, the regrouping by
local expert, the reverse exchange back to the sending slots and the global
aux loss.  Every rank's output must equal the oracle's whole layer on that
rank's tokens (expert parallelism only moves where an expert runs)."""
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


class OracleOps:
    """The six local steps of ep_forward in float64 on the CPU, from the oracle."""

    def route(self, x, W, b, k, renorm):
        import oracle
        L = oracle.router_logits(x.float(), W, b)
        idx, gate, ps = oracle.route(L, k, renorm)
        return torch.from_numpy(idx), torch.from_numpy(gate), torch.from_numpy(ps)

    def dispatch(self, idx, gate, x, E, cap):
        import oracle
        counts, kept, pos, _ = oracle.dispatch(idx.numpy(), E, cap)
        offsets = np.concatenate([[0], np.cumsum(kept)]).astype(np.int64)
        T, k = idx.shape
        A = int(offsets[-1])
        slot = np.full((T, k), -1, dtype=np.int64)
        row_token = np.zeros(max(A, 1), dtype=np.int64)
        row_gate = torch.zeros(max(A, 1), dtype=torch.float64)
        for t in range(T):
            for j in range(k):
                if pos[t, j] >= 0:
                    r = offsets[idx[t, j]] + pos[t, j]
                    slot[t, j] = r
                    row_token[r] = t
                    row_gate[r] = gate[t, j]
        x_perm = x.double()[torch.from_numpy(row_token)]
        return dict(counts=torch.from_numpy(counts), kept=torch.from_numpy(kept),
                    offsets=torch.from_numpy(offsets.astype(np.int32)), slot_row=torch.from_numpy(slot),
                    row_token=torch.from_numpy(row_token), row_gate=row_gate, x_perm=x_perm)

    def permute_rows(self, src, index):
        return src[index.long()]

    def expert_ffn(self, rows, offsets, kept, w1, w2, gate, act):
        import oracle
        out = torch.zeros(rows.shape[0], w2.shape[1], dtype=torch.float64)
        for e in range(kept.shape[0]):
            for r in range(int(offsets[e]), int(offsets[e]) + int(kept[e])):
                _, f = oracle.expert_ffn_row(rows[r].float().numpy(), w1, w2, e, act)
                out[r] = float(gate[r]) * torch.from_numpy(f)
        return out

    def combine(self, y_perm, slot_row):
        T, k = slot_row.shape
        y = torch.zeros(T, y_perm.shape[1], dtype=torch.float64)
        for t in range(T):
            for j in range(k):
                r = int(slot_row[t, j])
                if r >= 0:
                    y[t] += y_perm[r]
        return y

    def aux_loss(self, counts, prob_sum, T, alpha):
        import oracle
        return torch.tensor(oracle.aux_loss(counts.numpy(), prob_sum.numpy().astype(np.float64), T, alpha))


D, E, K, F, ACT = 16, 8, 2, 8, "swiglu"


def _weights():
    g = torch.Generator().manual_seed(11)
    W = torch.randn(E, D, generator=g) * 0.5
    w1 = torch.randn(E, 2 * F, D, generator=g) / 4
    w2 = torch.randn(E, D, F, generator=g) / 3
    return W, w1, w2


def _tokens(rank):
    g = torch.Generator().manual_seed(100 + rank)
    return torch.randn(40 + 9 * rank, D, generator=g)


def _worker(rank, world, port, out_dir, host_exchange=False):
    import oracle
    from top_routing_expert_02_b300.ep import ep_forward, expert_block
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    W, w1, w2 = _weights()
    x = _tokens(rank)
    lo, hi = expert_block(E, world, rank)
    cap = oracle.capacity(x.shape[0], E, 1.0)
    res = ep_forward(x, W, None, w1[lo:hi].contiguous(), w2[lo:hi].contiguous(), k=K, cap=cap, act=ACT,
                     ops=OracleOps(), host_exchange=host_exchange)
    np.save(os.path.join(out_dir, f"y{rank}.npy"), res.y.numpy())
    np.save(os.path.join(out_dir, f"m{rank}.npy"), np.array([float(res.loss), res.recv_rows]))
    dist.destroy_process_group()


@pytest.mark.parametrize("world,host_exchange", [(2, False), (4, False), (2, True)])
def test_expert_parallel_forward_matches_the_layer_on_each_shard(world, host_exchange, tmp_path):
    """host_exchange=True stages the exchanges as raw bytes through host
    tensors (the path the two-rank GPU test takes over gloo)."""
    import oracle
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path), host_exchange), nprocs=world,
                       start_method="spawn")
    W, w1, w2 = _weights()
    xs = [_tokens(r) for r in range(world)]
    whole = torch.cat(xs)
    idx, _, ps = oracle.route(oracle.router_logits(whole, W), K)
    counts, _, _, _ = oracle.dispatch(idx, E, whole.shape[0])
    loss_whole = oracle.aux_loss(counts, ps, whole.shape[0], 0.01)
    recv_total = kept_total = 0
    for r in range(world):
        cap = oracle.capacity(xs[r].shape[0], E, 1.0)
        ref = oracle.forward(xs[r], W, None, w1, w2, k=K, cap=cap, act=ACT)
        y = np.load(tmp_path / f"y{r}.npy")
        np.testing.assert_allclose(y, ref["y"], rtol=1e-12, atol=1e-12)
        assert ref["n_dropped"] > 0                        # capacity bites on every shard
        loss, recv = np.load(tmp_path / f"m{r}.npy")
        assert abs(loss - loss_whole) <= 1e-6 * loss_whole
        recv_total += int(recv)
        kept_total += int(ref["kept"].sum())
    assert recv_total == kept_total                        # every kept row ran on exactly one expert owner
