"""Shared helpers of the GPU parity tests: build a seeded case, run the CUDA
path through the C ABI, run the oracle, compare.

Bars (written here once, used by every parity test):
  routing indices, counts, kept, offsets, slot places, drops: bit-exact
  gates, prob sums, aux loss:         relative error <= 1e-5 for fp32 x (router logits are
                                      one fp32 FMA chain each) and for bf16 x (tensor-core
                                      router: exact bf16 products of the three weight parts;
                                      the large part accumulates over at most 4 K blocks of 64
                                      columns in the tensor core before an fp32 add into the
                                      running sum, which bounds the accumulator's drift to
                                      about 16 steps of 2^-23 of a chunk sum)
  layer output y:                     relative Frobenius error <= 1e-5 (fp32 layer),
                                      <= 2e-2 (bf16 layer), pooled over the compared tokens
                                      and for every token on its own (a token whose every
                                      slot was dropped must be exactly zero)
  per-token log-sum-exp:              as the gates (it carries the same logit error, atol 1e-6)
  router z-loss:                      twice the gates' bar (it squares the log-sum-exp)
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import top_routing_expert_02_b300 as moe
from top_routing_expert_02_b300 import synth

GATE_RTOL = {"f32": 1e-5, "bf16": 1e-5}
Y_TOL = {"f32": 1e-5, "bf16": 2e-2}


def make_case(cfg: synth.MoEConfig, device="cuda", condition=True, routing=None, n_group=1, topk_group=1):
    """Inputs of one workload: host copies for the oracle, device copies for the
    kernels.  With groups, the near-tie margin covers the group decisions too."""
    ri = routing if routing is not None else synth.make_routing_inputs(cfg)
    if condition:
        gaps = None if n_group == 1 else (lambda L: oracle.decision_gaps(L, cfg.k, n_group, topk_group))
        ri = synth.condition_near_ties(cfg, ri, oracle.router_logits, gaps_fn=gaps)
    w1, w2 = synth.make_expert_weights(cfg, device=device)
    cap = moe.capacity(cfg.T, cfg.E, cfg.cf)
    return dict(cfg=cfg, cap=cap, x_h=ri.x, W_h=ri.W, b_h=ri.b, x=ri.x.to(device), W=ri.W.to(device),
                b=None if ri.b is None else ri.b.to(device), w1=w1, w2=w2)


def run_gpu(case, plan=None):
    cfg = case["cfg"]
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    if plan is None:
        plan = moe.MoEPlan(cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.act, tdt, case["cap"], case["x"].device,
                           cfg.alpha, cfg.renorm)
    plan.run(case["x"], case["W"], case["b"], case["w1"], case["w2"])
    moe.check()
    return plan


def run_oracle(case, tokens=None, w_host=None, **variant):
    """The oracle's layer on the case's inputs; ``variant`` passes the routing
    variants (n_group, topk_group, z_beta, aux_post_drop) through."""
    cfg = case["cfg"]
    if w_host is None:
        w_host = (case["w1"].cpu(), case["w2"].cpu())
    return oracle.forward(case["x_h"], case["W_h"], case["b_h"], w_host[0], w_host[1], k=cfg.k, cap=case["cap"],
                          act=cfg.act, renorm=cfg.renorm, alpha=cfg.alpha, tokens=tokens, **variant)


def rel_fro(a: np.ndarray, b: np.ndarray) -> float:
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def compare_routing(plan, ref, dtype: str):
    idx = plan.topk_idx.cpu().numpy()
    assert np.array_equal(idx, ref["idx"]), "top-k indices differ"
    g = plan.topk_gate.cpu().numpy().astype(np.float64)
    ps = plan.prob_sum.cpu().numpy().astype(np.float64)
    print(f"[parity] gate max rel err {np.max(np.abs(g - ref['gate']) / np.abs(ref['gate'])):.3e}, "
          f"prob_sum max rel err {np.max(np.abs(ps - ref['prob_sum']) / np.maximum(np.abs(ref['prob_sum']), 1e-300)):.3e}")
    np.testing.assert_allclose(g, ref["gate"], rtol=GATE_RTOL[dtype], atol=0)
    np.testing.assert_allclose(ps, ref["prob_sum"], rtol=GATE_RTOL[dtype], atol=1e-30)


def compare_dispatch(plan, ref, x_h=None, check_rows=256):
    D = plan.disp
    counts, kept = D.counts.cpu().numpy(), D.kept.cpu().numpy()
    offsets, slot = D.offsets.cpu().numpy(), D.slot_row.cpu().numpy()
    assert np.array_equal(counts, ref["counts"])
    assert np.array_equal(kept, ref["kept"])
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(ref["kept"])]))
    assert int(D.n_dropped.item()) == ref["n_dropped"]
    idx = ref["idx"]
    pos = np.where(slot >= 0, slot - offsets[idx], -1)
    assert np.array_equal(pos, ref["pos"]), "slot places differ"
    A = int(offsets[-1])
    if A:
        row_token = D.row_token[:A].cpu().numpy()
        row_gate = D.row_gate[:A].cpu().numpy()
        t, j = np.nonzero(slot >= 0)
        rows = slot[t, j]
        assert np.array_equal(np.sort(rows), np.arange(A))        # bijection onto 0..A-1
        assert np.array_equal(row_token[rows], t)
        assert np.array_equal(row_gate[rows], plan.topk_gate.cpu().numpy()[t, j])
        if x_h is not None:
            sel = np.linspace(0, A - 1, num=min(A, check_rows)).astype(np.int64)
            xp = D.x_perm[torch.from_numpy(sel).to(D.x_perm.device)].cpu()
            assert torch.equal(xp, x_h[torch.from_numpy(row_token[sel]).long()])


def compare_output(plan, ref, dtype: str):
    toks = torch.from_numpy(ref["tokens"]).long().to(plan.y.device)
    y = plan.y[toks].float().cpu().numpy().astype(np.float64)
    err = rel_fro(y, ref["y"])
    norms = np.linalg.norm(ref["y"], axis=1)
    live = norms > 0
    per_tok = np.linalg.norm(y - ref["y"], axis=1)[live] / norms[live]
    worst = float(per_tok.max()) if per_tok.size else 0.0
    print(f"[parity] y rel Frobenius err {err:.3e} over {len(ref['tokens'])} tokens, worst token {worst:.3e}; "
          f"loss {float(plan.loss.item()):.7f} vs {ref['loss']:.7f}")
    assert err <= Y_TOL[dtype], f"relative Frobenius error {err:.3e} > {Y_TOL[dtype]}"
    assert worst <= Y_TOL[dtype], f"a token's relative error {worst:.3e} > {Y_TOL[dtype]}"
    assert not np.any(y[~live]), "a token with every slot dropped must get a zero row"
    loss = float(plan.loss.item())
    assert abs(loss - ref["loss"]) <= GATE_RTOL[dtype] * abs(ref["loss"]) + 1e-12, (loss, ref["loss"])
    return err


def compare_z_loss(plan, ref, dtype: str):
    """Per-token log-sum-exp and the router z-loss against the oracle."""
    T = plan.T
    lse = plan.lse[:T].cpu().numpy().astype(np.float64)
    err = np.max(np.abs(lse - ref["lse"]) / np.maximum(np.abs(ref["lse"]), 1e-30)) if T else 0.0
    z = float(plan.z_loss.item())
    print(f"[parity] lse max rel err {err:.3e}; z-loss {z:.8f} vs {ref['z_loss']:.8f}")
    np.testing.assert_allclose(lse, ref["lse"], rtol=GATE_RTOL[dtype], atol=1e-6)
    assert abs(z - ref["z_loss"]) <= 2 * GATE_RTOL[dtype] * abs(ref["z_loss"]) + 1e-12, (z, ref["z_loss"])


def tile_tokens(plan, per_tile: int = 1):
    """Tokens that cover every 128-row tile of every expert segment of the
    grouped GEMMs (``per_tile`` rows from each, spread over the tile), for
    comparing y with the oracle at sizes where it cannot compute every token."""
    D = plan.disp
    offsets, kept = D.offsets.cpu().numpy(), D.kept.cpu().numpy()
    row_token = D.row_token.cpu().numpy()
    toks = set()
    for e in range(plan.E):
        for m0 in range(0, int(kept[e]), 128):
            n = min(128, int(kept[e]) - m0)
            for i in range(per_tile):
                r = int(offsets[e]) + m0 + (i * (n - 1)) // max(per_tile - 1, 1)
                toks.add(int(row_token[r]))
    return sorted(toks)


def check_expert_rows_on_device(plan, x, w1, w2, act: str, tol: float = 2e-2):
    """Every kept row of h and y_perm against a per-expert fp32 reference
    computed with torch on the device (no TF32), row by row: h = act(x_perm w1^T)
    and y_perm = gate * (h w2^T) with the kernel's own h, so each GEMM is
    checked on its own; and y against the sum of the kernel's y_perm rows in
    j order (fp32, one rounding), which must match bit for bit.  Returns the
    worst per-row relative errors of h and y_perm."""
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        D = plan.disp
        offsets, kept = D.offsets.cpu().tolist(), D.kept.cpu().tolist()
        F, E = plan.F, plan.E
        worst_h = worst_y = 0.0
        for e in range(E):
            r0, n = offsets[e], kept[e]
            if n == 0:
                continue
            xp = D.x_perm[r0:r0 + n].float()
            assert torch.equal(D.x_perm[r0:r0 + n], x[D.row_token[r0:r0 + n].long()])
            z = xp @ w1[e].float().t()
            if act == "swiglu":
                a = torch.nn.functional.silu(z[:, :F]) * z[:, F:]
            elif act == "gelu":
                a = torch.nn.functional.gelu(z)
            else:
                a = z
            h = plan.h[r0:r0 + n].float()
            eh = (torch.linalg.vector_norm(h - a, dim=1) / torch.linalg.vector_norm(a, dim=1).clamp_min(1e-30)).max()
            yref = (h @ w2[e].float().t()) * D.row_gate[r0:r0 + n, None]
            yp = plan.y_perm[r0:r0 + n].float()
            ey = (torch.linalg.vector_norm(yp - yref, dim=1) /
                  torch.linalg.vector_norm(yref, dim=1).clamp_min(1e-30)).max()
            worst_h, worst_y = max(worst_h, float(eh)), max(worst_y, float(ey))
        assert worst_h <= tol, f"an h row's relative error {worst_h:.3e} > {tol}"
        assert worst_y <= tol, f"a y_perm row's relative error {worst_y:.3e} > {tol}"
        # the combine: y[t] = sum over kept j of y_perm[slot_row[t, j]] (fp32, j order, one rounding)
        slot = D.slot_row.long()
        acc = torch.zeros(plan.T, plan.d, dtype=torch.float32, device=x.device)
        for j in range(plan.k):
            rows = slot[:, j]
            keep = rows >= 0
            acc[keep] += plan.y_perm[rows[keep]].float()
        assert torch.equal(plan.y, acc.to(plan.y.dtype)), "y differs from the j-ordered sum of its y_perm rows"
        print(f"[parity] every kept row: worst h rel err {worst_h:.3e}, worst y_perm rel err {worst_y:.3e}")
        return worst_h, worst_y
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
