"""GPU parity of the layer backward against the fp64 backward oracle
(oracle/backward.py), through the C ABI (MoEPlan.backward), on seeded
inputs spanning several tiles with ragged expert segments, drops, empty
experts, both activations, renormalised and raw gates, the z-loss and the
post-drop aux loss; plus the data-movement kernels bit for bit and the
weight-gradient GEMM against torch fp32 per expert.

Bar (bf16 layers): relative Frobenius error <= 2e-2 for dx, dW, db, dw1,
dw2, dgate and dl, the bar of the bf16 forward output.  The path rounds
to bf16 at do, z, da, dz and dx_perm (each ~2^-9 relative), so the
expected error is a few 1e-3."""
import math

import numpy as np
import pytest
import torch

import top_routing_expert_02_b300 as moe
from oracle import backward as OB
from top_routing_expert_02_b300 import synth

from moe_cases import make_case, rel_fro

pytestmark = pytest.mark.gpu

C = synth.MoEConfig
TOL = 2e-2

# name: (config, z_beta, post-drop aux)
CASES = {
    "swiglu_e8": (C("swiglu_e8", 2000, 256, 8, 2, 384, "swiglu", 1.25, "bf16"), 0.0, False),
    "gelu_e16_hot": (C("gelu_e16_hot", 1500, 192, 16, 2, 320, "gelu", 1.0, "bf16", bias="hot2"), 1e-3, True),
    "swiglu_e64_zipf": (C("swiglu_e64_zipf", 3000, 128, 64, 2, 192, "swiglu", 1.25, "bf16", bias="zipf"), 1e-3,
                        False),
    "swiglu_e128_top8": (C("swiglu_e128_top8", 300, 256, 128, 8, 128, "swiglu", 0.0, "bf16"), 1e-2, False),
    "gelu_e32_norenorm": (C("gelu_e32_norenorm", 900, 128, 32, 4, 256, "gelu", 1.5, "bf16", renorm=False), 0.0,
                          True),
    "small_T": (C("small_T", 50, 128, 8, 2, 128, "swiglu", 1.25, "bf16"), 0.0, False),
    "e256_top16": (C("e256_top16", 600, 128, 256, 16, 64, "swiglu", 0.0, "bf16"), 1e-3, False),
    "min_d64_f64": (C("min_d64_f64", 3, 64, 2, 1, 64, "gelu", 0.0, "bf16"), 0.0, False),
}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "these tests need a CUDA device"
    moe.lib()
    yield


def _dy(cfg):
    g = torch.Generator().manual_seed(1234 + cfg.T)
    return torch.randn(cfg.T, cfg.d, generator=g).to(torch.bfloat16)


def _run(cfg, z_beta, post, aux_weight=1.0, z_weight=1.0, grad_dtype=torch.float32, n_group=1, topk_group=1):
    case = make_case(cfg, n_group=n_group, topk_group=topk_group)
    plan = moe.MoEPlan(cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.act, torch.bfloat16, case["cap"], case["x"].device,
                       cfg.alpha, cfg.renorm, z_beta=z_beta if z_beta else None, aux_post_drop=post, train=True,
                       grad_dtype=grad_dtype, n_group=n_group, topk_group=topk_group)
    moe.set_wait_limit(400_000_000)
    try:
        plan.run(case["x"], case["W"], case["b"], case["w1"], case["w2"])
        dy = _dy(cfg)
        g = plan.backward(case["x"], case["W"], case["w1"], case["w2"], dy.cuda(), aux_weight=aux_weight,
                          z_weight=z_weight)
        moe.check()
    finally:
        moe.set_wait_limit(0)
    ref = OB.backward(case["x_h"], case["W_h"], case["b_h"], case["w1"].cpu(), case["w2"].cpu(), dy, k=cfg.k,
                      cap=case["cap"], act=cfg.act, renorm=cfg.renorm, alpha=cfg.alpha, aux_weight=aux_weight,
                      z_beta=z_beta, z_weight=z_weight, aux_post_drop=post, n_group=n_group, topk_group=topk_group)
    return plan, g, ref, case


@pytest.mark.parametrize("name,grad_dtype", [(n, torch.float32) for n in CASES] +
                         [("swiglu_e8", torch.bfloat16), ("swiglu_e64_zipf", torch.bfloat16)])
def test_backward_against_oracle(name, grad_dtype):
    cfg, z_beta, post = CASES[name]
    plan, g, ref, _ = _run(cfg, z_beta, post, grad_dtype=grad_dtype)
    assert g["dw1"].dtype == grad_dtype
    errs = {}
    for key in ("dx", "dW", "db", "dw1", "dw2", "dgate", "dl"):
        got = g[key].float().cpu().numpy().astype(np.float64)
        if key in ("dx", "dgate", "dl"):
            got = got[:cfg.T]
        errs[key] = rel_fro(got, ref[key])
    print(f"[backward parity] {name}: " + ", ".join(f"{k} {v:.2e}" for k, v in errs.items()))
    for key, err in errs.items():
        assert err <= TOL, (key, err)


@pytest.mark.parametrize("name,G,M,aw,zw", [("swiglu_e64_zipf", 16, 3, 0.5, 2.0), ("swiglu_e128_top8", 8, 4, 1.0, 1.0),
                                           ("gelu_e32_norenorm", 8, 2, 2.0, 0.0)])
def test_backward_with_group_routing_and_loss_weights(name, G, M, aw, zw):
    """Group-limited routing in the forward, other aux / z-loss weights."""
    cfg, z_beta, post = CASES[name]
    plan, g, ref, _ = _run(cfg, z_beta or 1e-3, post, aux_weight=aw, z_weight=zw, n_group=G, topk_group=M)
    for key in ("dx", "dW", "db", "dw1", "dw2", "dgate", "dl"):
        got = g[key].float().cpu().numpy().astype(np.float64)
        if key in ("dx", "dgate", "dl"):
            got = got[:cfg.T]
        assert rel_fro(got, ref[key]) <= TOL, key


def test_backward_is_bitwise_reproducible():
    cfg, z_beta, post = CASES["swiglu_e64_zipf"]
    p1, g1, _, case = _run(cfg, z_beta, post)
    snap = {k: v.clone() for k, v in g1.items()}
    g2 = p1.backward(case["x"], case["W"], case["w1"], case["w2"], _dy(cfg).cuda())
    moe.check()
    for k in ("dx", "dW", "db", "dw1", "dw2"):
        assert torch.equal(snap[k], g2[k]), k


def test_transpose_and_pack_are_exact():
    g = torch.Generator(device="cuda").manual_seed(5)
    w = torch.randn(3, 192, 320, device="cuda", generator=g).to(torch.bfloat16)
    wt = moe.transpose_experts(w)
    assert torch.equal(wt, w.transpose(1, 2).contiguous())
    # ragged segments incl. an empty one and one longer than 64
    kept = torch.tensor([70, 0, 5, 64, 1], dtype=torch.int32, device="cuda")
    offsets = torch.zeros(6, dtype=torch.int32, device="cuda")
    offsets[1:] = torch.cumsum(kept, 0)
    R = int(offsets[-1])
    src = torch.randn(R, 128, device="cuda", generator=g).to(torch.bfloat16)
    ld = moe.wgrad_cols(R, 5)
    out = torch.full((128, ld), 7.0, dtype=torch.bfloat16, device="cuda")
    moe.pack_segments_t(src, offsets, kept, R, ld, out=out)
    moe.check()
    col = 0
    for e in range(5):
        n = int(kept[e])
        kp = (n + 63) // 64 * 64
        o = int(offsets[e])
        assert torch.equal(out[:, col:col + n], src[o:o + n].T)
        assert torch.all(out[:, col + n:col + kp] == 0)
        col += kp


def test_expert_wgrad_against_torch_per_expert():
    """dw[e] = at[:, seg] bt[:, seg]^T against torch fp32 matmul, M not a
    multiple of 128 and N not of 256; an empty expert gets zeros."""
    g = torch.Generator(device="cuda").manual_seed(6)
    kept = torch.tensor([100, 0, 300, 64], dtype=torch.int32, device="cuda")
    E, M, N = 4, 192, 320
    ld = moe.wgrad_cols(int(kept.sum()), E)
    at = torch.zeros(M, ld, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(N, ld, dtype=torch.bfloat16, device="cuda")
    col = 0
    for e in range(E):
        n = int(kept[e])
        at[:, col:col + n] = torch.randn(M, n, device="cuda", generator=g).to(torch.bfloat16)
        bt[:, col:col + n] = torch.randn(N, n, device="cuda", generator=g).to(torch.bfloat16)
        col += (n + 63) // 64 * 64
    dw = moe.expert_wgrad(at, bt, kept)
    dwb = moe.expert_wgrad(at, bt, kept, dtype=torch.bfloat16)
    moe.check()
    col = 0
    for e in range(E):
        n = int(kept[e])
        ref = at[:, col:col + n].float() @ bt[:, col:col + n].float().T
        assert torch.allclose(dw[e], ref, rtol=1e-4, atol=1e-3), e
        assert torch.equal(dwb[e], dw[e].to(torch.bfloat16)), e          # one rounding of the same sums
        col += (n + 63) // 64 * 64


def test_expert_wgrad_rows_against_torch_and_packed():
    """dw[e] = a[seg]^T b[seg] read straight from row-major a [rows, M], b [rows, N]:
    against torch fp32 and bit for bit against the packed-transpose path (the
    same products in the same order).  The segments leave gaps and a tail that
    hold NaN, so a partial 64-row block that read past its segment would show;
    M % 128 == 64, N % 256 == 64, an empty expert, segments of 1, 64 and 65 rows."""
    g = torch.Generator(device="cuda").manual_seed(16)
    kept_l = [100, 0, 300, 64, 1, 65]
    gaps = [3, 7, 0, 5, 2, 1]
    E, M, N = len(kept_l), 192, 320
    offs, pos = [], 0
    for n, gp in zip(kept_l, gaps):
        pos += gp
        offs.append(pos)
        pos += n
    R = pos + 37   # NaN rows past the last segment
    a = torch.full((R, M), float("nan"), dtype=torch.bfloat16, device="cuda")
    b = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    for o, n in zip(offs, kept_l):
        a[o:o + n] = torch.randn(n, M, device="cuda", generator=g).to(torch.bfloat16)
        b[o:o + n] = torch.randn(n, N, device="cuda", generator=g).to(torch.bfloat16)
    offsets = torch.tensor(offs + [pos], dtype=torch.int32, device="cuda")
    kept = torch.tensor(kept_l, dtype=torch.int32, device="cuda")
    dw = moe.expert_wgrad_rows(a, b, offsets, kept, R)
    dwb = moe.expert_wgrad_rows(a, b, offsets, kept, R, dtype=torch.bfloat16)
    # the packed path on the same segments (gap-free copies)
    cont = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    cont[1:] = torch.cumsum(kept, 0)
    A = int(cont[-1])
    ac = torch.cat([a[o:o + n] for o, n in zip(offs, kept_l)])
    bc = torch.cat([b[o:o + n] for o, n in zip(offs, kept_l)])
    ld = moe.wgrad_cols(A, E)
    dwp = moe.expert_wgrad(moe.pack_segments_t(ac, cont, kept, A, ld), moe.pack_segments_t(bc, cont, kept, A, ld),
                           kept)
    moe.check()
    assert bool(torch.isfinite(dw).all())
    for e, (o, n) in enumerate(zip(offs, kept_l)):
        ref = a[o:o + n].float().T @ b[o:o + n].float()
        assert torch.allclose(dw[e], ref, rtol=1e-4, atol=1e-3), e
        assert torch.equal(dwb[e], dw[e].to(torch.bfloat16)), e
    assert torch.equal(dw, dwp)


def _router_grad_inputs(T, E, k, d, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    R = T * k + 7
    dx_perm = torch.randn(R, d, device="cuda", generator=g).to(torch.bfloat16)
    slot_row = torch.randperm(R, device="cuda", generator=g)[:T * k].view(T, k).to(torch.int32)
    drop = torch.rand(T, k, device="cuda", generator=g) < 0.2
    slot_row[drop] = -1
    dl = torch.randn(T, E, device="cuda", generator=g) * 1e-2
    W = torch.randn(E, d, device="cuda", generator=g) * 0.05
    x = torch.randn(T, d, device="cuda", generator=g).to(torch.bfloat16)
    return dx_perm, slot_row.contiguous(), dl, W, x


def _router_grad_refs(dx_perm, slot_row, dl, W, x):
    """fp64 torch: dx = sum of the kept dx_perm rows + dl W, dW = dl^T x, db = sum_t dl."""
    T, k = slot_row.shape
    rows = dx_perm.double()
    gath = torch.where((slot_row >= 0)[..., None], rows[slot_row.clamp(min=0).long()], torch.zeros((), dtype=torch.float64,
                                                                                             device="cuda"))
    dx = gath.sum(1) + dl.double() @ W.double()
    return dx, dl.double().T @ x.double(), dl.double().sum(0)


@pytest.mark.parametrize("T,E,k,d", [(1000, 8, 2, 256), (777, 128, 8, 128), (300, 256, 16, 64), (4097, 64, 2, 512),
                                     (5, 1, 1, 64), (129, 3, 2, 128)])
def test_router_grads_on_tensor_cores(T, E, k, d):
    """moe_router_grads (bf16 hi/lo parts on the tensor cores) against fp64:
    dx within one bf16 rounding, dW and db to fp32 accuracy; the CUDA-core
    pair moe_grad_x + moe_router_wgrad against the same references; both
    bitwise reproducible.  The shapes cover E = 8 (padded to 64), E = 256
    with top-16, d = 64 (one partial N tile), ragged token splits, a single
    expert with five tokens and three experts over 129 tokens."""
    dx_perm, slot_row, dl, W, x = _router_grad_inputs(T, E, k, d, T + E)
    dx, dW, db = moe.router_grads(dx_perm, slot_row, dl, W, x)
    dx2, dW2, db2 = moe.router_grads(dx_perm, slot_row, dl, W, x)
    dx_c = moe.grad_x(dx_perm, slot_row, dl, W)
    dW_c, db_c = moe.router_wgrad(dl, x)
    moe.check()
    rdx, rdW, rdb = _router_grad_refs(dx_perm, slot_row, dl, W, x)
    for got in (dx, dx_c):
        err = (got.double() - rdx).abs()
        assert bool((err <= rdx.abs() * 2.0 ** -8 + 1e-5).all()), float(err.max())
    for got in (dW, dW_c):
        assert float((got.double() - rdW).norm() / rdW.norm()) < 1e-5
    for got in (db, db_c):
        assert float((got.double() - rdb).norm() / rdb.norm()) < 1e-6
    assert torch.equal(dx, dx2) and torch.equal(dW, dW2) and torch.equal(db, db2)


def test_router_grads_no_tokens():
    E, d = 8, 128
    dW = torch.full((E, d), 3.0, device="cuda")
    db = torch.full((E,), 3.0, device="cuda")
    x = torch.empty((0, d), dtype=torch.bfloat16, device="cuda")
    moe.router_grads(torch.empty((1, d), dtype=torch.bfloat16, device="cuda"),
                     torch.empty((0, 2), dtype=torch.int32, device="cuda"), torch.empty((0, E), device="cuda"),
                     torch.zeros(E, d, device="cuda"), x, dW=dW, db=db)
    moe.check()
    assert bool((dW == 0).all()) and bool((db == 0).all())


def test_weight_gradient_tile_orders_agree():
    """M-fastest and N-fastest tile orders give the same bits (the order only
    changes which blocks run together)."""
    cfg = CASES["swiglu_e8"][0]
    case = make_case(cfg)
    plan = moe.MoEPlan(cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.act, torch.bfloat16, case["cap"], "cuda", cfg.alpha,
                       cfg.renorm, train=True)
    plan.run(case["x"], case["W"], case["b"], case["w1"], case["w2"])
    dy = _dy(cfg).cuda()
    out = {}
    try:
        for order in (1, 2):
            moe.set_wgrad_order(order)
            g = plan.backward(case["x"], case["W"], case["w1"], case["w2"], dy)
            out[order] = (g["dw1"].clone(), g["dw2"].clone())
    finally:
        moe.set_wgrad_order(0)
    moe.check()
    assert torch.equal(out[1][0], out[2][0]) and torch.equal(out[1][1], out[2][1])


def test_expert_wgrad_rows_no_rows_gives_zeros():
    kept = torch.zeros(3, dtype=torch.int32, device="cuda")
    offsets = torch.zeros(4, dtype=torch.int32, device="cuda")
    a = torch.full((1, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    b = torch.full((1, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    for rows_max in (0, 1):   # no buffer rows at all / rows but empty segments
        dw = torch.full((3, 64, 128), 5.0, device="cuda")
        moe.expert_wgrad_rows(a, b, offsets, kept, rows_max, dw=dw)
        moe.check()
        assert bool((dw == 0).all()), rows_max


@pytest.mark.parametrize("name", ["swiglu_e8", "gelu_e16_hot"])
def test_kept_pre_activation_equals_recompute(name):
    """The z that the training forward keeps (moe_expert_up_z) is bit for bit
    the identity-epilogue GEMM of w1 on x_perm, and h is unchanged by keeping it."""
    cfg = CASES[name][0]
    case = make_case(cfg)
    plan = moe.MoEPlan(cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.act, torch.bfloat16, case["cap"], case["x"].device,
                       cfg.alpha, cfg.renorm, train=True)
    plan.run(case["x"], case["W"], case["b"], case["w1"], case["w2"])
    D = plan.disp
    R = plan.rows_max
    A = int(D.offsets[-1])
    N1 = case["w1"].shape[1]
    z2 = moe.expert_up(D.x_perm, D.offsets, D.kept, case["w1"], N1, "identity", R)
    h2 = moe.expert_up(D.x_perm, D.offsets, D.kept, case["w1"], cfg.F, cfg.act, R)
    moe.check()
    assert torch.equal(plan.z[:A], z2[:A])
    assert torch.equal(plan.h[:A], h2[:A])


@pytest.mark.parametrize("kept_list", [[150, 0, 7, 300], [1000, 777, 0, 1300]])
def test_expert_dgrad_mn_major_against_torch(kept_list):
    """out[r] = a[r] . w[e] with w [E, K, N] read MN-major, against torch fp32
    per expert: ragged segments, an empty expert, N not a multiple of 256;
    the second segment list has >= 3 row tiles per expert on average, so its
    output blocks go by TMA stores, and they match the per-thread stores bit
    for bit."""
    g = torch.Generator(device="cuda").manual_seed(7)
    E, K, N = 4, 192, 320
    kept = torch.tensor(kept_list, dtype=torch.int32, device="cuda")
    offsets = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    offsets[1:] = torch.cumsum(kept, 0)
    R = int(offsets[-1])
    a = torch.randn(R, K, device="cuda", generator=g).to(torch.bfloat16)
    w = (torch.randn(E, K, N, device="cuda", generator=g) / 8).to(torch.bfloat16)
    out = moe.expert_dgrad(a, offsets, kept, w, R)
    moe.set_gemm_tma_store(False)
    try:
        out2 = moe.expert_dgrad(a, offsets, kept, w, R)
    finally:
        moe.set_gemm_tma_store(True)
    moe.check()
    assert torch.equal(out, out2)
    for e in range(E):
        o, n = int(offsets[e]), int(kept[e])
        ref = a[o:o + n].float() @ w[e].float()
        assert torch.allclose(out[o:o + n].float(), ref, rtol=1e-2, atol=2e-2), e


def test_backward_capacity_zero_and_empty_batch():
    """cap = 0: every slot dropped, so the expert weights get zero gradients
    and dx is the router's part alone (against the oracle); T = 0: the call
    runs and every weight gradient is zero."""
    cfg = C("cap0", 300, 128, 8, 2, 128, "swiglu", 1.0, "bf16")
    case = make_case(cfg)
    plan = moe.MoEPlan(cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.act, torch.bfloat16, 0, case["x"].device, cfg.alpha,
                       cfg.renorm, train=True)
    plan.run(case["x"], case["W"], case["b"], case["w1"], case["w2"])
    dy = _dy(cfg)
    g = plan.backward(case["x"], case["W"], case["w1"], case["w2"], dy.cuda())
    moe.check()
    assert not g["dw1"].any() and not g["dw2"].any()
    ref = OB.backward(case["x_h"], case["W_h"], case["b_h"], case["w1"].cpu(), case["w2"].cpu(), dy, k=cfg.k, cap=0,
                      act=cfg.act, renorm=cfg.renorm, alpha=cfg.alpha)
    for key in ("dx", "dW", "db", "dl"):
        got = g[key].float().cpu().numpy().astype(np.float64)
        if key in ("dx", "dl"):
            got = got[:cfg.T]
        assert rel_fro(got, ref[key]) <= TOL, key

    x0 = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    plan0 = moe.MoEPlan(0, 128, 8, 2, 128, "swiglu", torch.bfloat16, 0, "cuda", train=True)
    plan0.run(x0, case["W"], case["b"], case["w1"], case["w2"])
    g0 = plan0.backward(x0, case["W"], case["w1"], case["w2"], x0)
    moe.check()
    assert not g0["dw1"].any() and not g0["dw2"].any() and not g0["dW"].any() and not g0["db"].any()


@pytest.mark.slow
def test_backward_full_size_e8_swiglu():
    """The 8-expert bench layer at full size (T=4096, d=4096, F=14336, 2.8 GB of
    weights): every gradient against the fp64 oracle (weight gradients
    stored in fp32 on the host side)."""
    cfg = synth.workload("e8_swiglu")
    case = make_case(cfg)
    plan = moe.MoEPlan(cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.act, torch.bfloat16, case["cap"], case["x"].device,
                       cfg.alpha, cfg.renorm, train=True)
    plan.run(case["x"], case["W"], case["b"], case["w1"], case["w2"])
    dy = _dy(cfg)
    g = plan.backward(case["x"], case["W"], case["w1"], case["w2"], dy.cuda())
    moe.check()
    ref = OB.backward(case["x_h"], case["W_h"], case["b_h"], case["w1"].cpu(), case["w2"].cpu(), dy, k=cfg.k,
                      cap=case["cap"], act=cfg.act, renorm=cfg.renorm, alpha=cfg.alpha, wgrad_dtype=np.float32)
    def rel_fro_chunked(a, b):
        num = den = 0.0
        for i in range(a.shape[0]):          # one expert (or row) at a time keeps host memory bounded
            ai, bi = a[i].astype(np.float64), b[i].astype(np.float64)
            num += float(np.sum((ai - bi) ** 2))
            den += float(np.sum(bi * bi))
        return math.sqrt(num / den) if den > 0 else math.sqrt(num)

    errs = {}
    for key in ("dx", "dW", "db", "dw1", "dw2", "dgate", "dl"):
        got = g[key].float().cpu().numpy()
        if key in ("dx", "dgate", "dl"):
            got = got[:cfg.T]
        errs[key] = rel_fro_chunked(got[None] if got.ndim == 1 else got, ref[key][None] if ref[key].ndim == 1
                                    else ref[key])
    print("[backward parity] e8_swiglu full size: " + ", ".join(f"{k} {v:.2e}" for k, v in errs.items()))
    for key, err in errs.items():
        assert err <= TOL, (key, err)


@pytest.mark.parametrize("act", ["swiglu", "gelu"])
def test_act_bwd_and_fused_dgrad_act(act):
    """moe_act_bwd against the torch fp32 formula; moe_expert_dgrad_act (the da
    GEMM with the activation backward in its epilogue) against
    moe_act_bwd(z, moe_expert_dgrad(...)) -- the same values up to the bf16
    rounding of da that the fused path skips."""
    g = torch.Generator(device="cuda").manual_seed(9)
    E, d, F = 3, 256, 320
    N1 = 2 * F if act == "swiglu" else F
    kept = torch.tensor([130, 0, 70], dtype=torch.int32, device="cuda")
    offsets = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    offsets[1:] = torch.cumsum(kept, 0)
    R = int(offsets[-1])
    do = torch.randn(R, d, device="cuda", generator=g).to(torch.bfloat16)
    w2 = (torch.randn(E, d, F, device="cuda", generator=g) / 16).to(torch.bfloat16)
    z = torch.randn(R, N1, device="cuda", generator=g).to(torch.bfloat16)
    da = moe.expert_dgrad(do, offsets, kept, w2, R)
    dz = moe.act_bwd(z, da, offsets, F, act, R)
    dz_fused = moe.expert_dgrad_act(do, offsets, kept, w2, z, act, R)
    moe.check()
    zf, daf = z.float(), da.float()
    if act == "swiglu":
        zg, zu = zf[:, :F], zf[:, F:]
        s = torch.sigmoid(zg)
        ref = torch.cat([daf * zu * s * (1 + zg * (1 - s)), daf * zg * s], dim=1)
    else:
        cdf = 0.5 * (1 + torch.erf(zf / 2 ** 0.5))
        ref = daf * (cdf + zf * torch.exp(-0.5 * zf * zf) / (2 * torch.pi) ** 0.5)
    assert torch.allclose(dz.float(), ref, rtol=1e-2, atol=1e-2)
    err = (dz_fused.float() - dz.float()).norm() / dz.float().norm()
    assert err < 1e-2, err


def test_training_step_as_one_cuda_graph():
    """Forward + backward captured once and replayed: bit-identical to eager."""
    cfg, z_beta, post = CASES["swiglu_e64_zipf"]
    p1, g1, _, case = _run(cfg, z_beta, post)
    snap = {k: g1[k].clone() for k in ("dx", "dW", "db", "dw1", "dw2")}
    y = p1.y.clone()
    dy = _dy(cfg).cuda()
    graph = p1.capture(case["x"], case["W"], case["b"], case["w1"], case["w2"], dy=dy)
    for k in snap:
        p1._bwd[k].zero_()
    graph.replay()
    torch.cuda.synchronize()
    moe.check()
    assert torch.equal(p1.y, y)
    for k, v in snap.items():
        assert torch.equal(p1._bwd[k], v), k
