"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs.  Sizes span several tiles with ragged tails in M
(expert segments), N and K; bars are in moe_cases."""
import numpy as np
import pytest
import torch

import oracle
import top_routing_expert_02_b300 as moe
from top_routing_expert_02_b300 import synth

from moe_cases import (Y_TOL, check_expert_rows_on_device, compare_dispatch, compare_output, compare_routing,
                       make_case, rel_fro, run_gpu, run_oracle)

pytestmark = pytest.mark.gpu

C = synth.MoEConfig

SMALL = {
    # ragged M tiles (cap 313 = 128+128+57), 4 K blocks, 3 SwiGLU N tiles
    "swiglu_e8": C("swiglu_e8", 2000, 256, 8, 2, 384, "swiglu", 1.25, "bf16"),
    # GELU with a half N tile (F=320), 3 K blocks, two hot experts over capacity
    "gelu_e16_hot": C("gelu_e16_hot", 1500, 192, 16, 2, 320, "gelu", 1.0, "bf16", bias="hot2"),
    # 64 experts, Zipf skew: many empty or tiny segments; SwiGLU half N tile
    "swiglu_e64_zipf": C("swiglu_e64_zipf", 3000, 128, 64, 2, 192, "swiglu", 1.25, "bf16", bias="zipf"),
    # 128 experts, top-8, dropless
    "swiglu_e128_top8": C("swiglu_e128_top8", 300, 256, 128, 8, 128, "swiglu", 0.0, "bf16"),
    # router without renormalisation, E=32 (one expert per lane)
    "gelu_e32_norenorm": C("gelu_e32_norenorm", 900, 128, 32, 4, 256, "gelu", 1.5, "bf16", renorm=False),
    # fp32 x with E=200 (8 experts per lane), through the fp32 FFN
    "f32_e200": C("f32_e200", 400, 128, 200, 3, 128, "swiglu", 2.0, "f32"),
    # bf16 x with E=200: above the tensor-core router's 128 experts -> CUDA-core router
    "bf16_e200": C("bf16_e200", 257, 128, 200, 2, 128, "gelu", 0.0, "bf16"),
    # bf16, E=160, top-16: above the tensor-core router's 128 experts -> CUDA-core router
    "bf16_e160_top16": C("bf16_e160_top16", 300, 192, 160, 16, 128, "swiglu", 0.0, "bf16", renorm=False),
    # fewer tokens than one 128-row tile, and fewer kept rows than one GEMM tile
    "small_T": C("small_T", 50, 128, 8, 2, 128, "swiglu", 1.25, "bf16"),
    # the largest expert count and top-k: 256 experts (CUDA-core router), top-16
    "bf16_e256_top16": C("bf16_e256_top16", 600, 128, 256, 16, 64, "swiglu", 0.0, "bf16"),
    # the smallest shapes: d = F = 64 (one K block, one half N tile), two experts, top-1, one token
    "min_d64_f64": C("min_d64_f64", 1, 64, 2, 1, 64, "gelu", 0.0, "bf16"),
    # fp32 layer with GELU and drops, two K blocks
    "f32_gelu_e4": C("f32_gelu_e4", 333, 128, 4, 2, 192, "gelu", 1.0, "f32"),
    # more GEMM tiles than two per SM (up: 128 M-tiles x 6 N-tiles, down: 128 x 2), so the
    # persistent blocks run several tiles each, through both TMEM accumulators; every token checked
    "many_tiles": C("many_tiles", 8192, 512, 8, 2, 768, "swiglu", 0.0, "bf16"),
}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "these tests need a CUDA device"
    moe.lib()
    yield


def test_tiny_fp32_layer_full():
    case = make_case(synth.workload("tiny_fp32"))
    plan = run_gpu(case)
    ref = run_oracle(case)
    compare_routing(plan, ref, "f32")
    compare_dispatch(plan, ref, case["x_h"])
    assert ref["n_dropped"] > 0
    compare_output(plan, ref, "f32")


@pytest.mark.parametrize("name", list(SMALL))
def test_small_layers_full(name):
    cfg = SMALL[name]
    case = make_case(cfg)
    plan = run_gpu(case)
    check_expert_rows_on_device(plan, case["x"], case["w1"], case["w2"], cfg.act, tol=Y_TOL[cfg.dtype])
    ref = run_oracle(case)
    compare_routing(plan, ref, cfg.dtype)
    compare_dispatch(plan, ref, case["x_h"])
    compare_output(plan, ref, cfg.dtype)


def test_expert_up_and_down_against_torch():
    """The two grouped GEMMs alone, against CPU torch fp32 per expert."""
    cfg = SMALL["swiglu_e8"]
    case = make_case(cfg)
    plan = run_gpu(case)
    D = plan.disp
    kept, offs = D.kept.cpu().numpy(), D.offsets.cpu().numpy()
    xp = D.x_perm.float().cpu()
    h = plan.h.float().cpu()
    yp = plan.y_perm.float().cpu()
    rg = D.row_gate.cpu()
    w1, w2 = case["w1"].float().cpu(), case["w2"].float().cpu()
    F = cfg.F
    for e in range(cfg.E):
        r0, r1 = offs[e], offs[e] + kept[e]
        z = xp[r0:r1] @ w1[e].T
        href = torch.nn.functional.silu(z[:, :F]) * z[:, F:]
        assert rel_fro(h[r0:r1].numpy(), href.numpy()) < 1e-2
        yref = rg[r0:r1, None] * (h[r0:r1] @ w2[e].T)
        assert rel_fro(yp[r0:r1].numpy(), yref.numpy()) < 1e-2


@pytest.mark.parametrize("bn", [128, 192, 256])
@pytest.mark.parametrize("name", ["swiglu_e8", "gelu_e16_hot"])
def test_every_gemm_tile_width(name, bn):
    """Each output-tile width of the tensor-core GEMMs, forced, on layers with
    ragged M, N and K tails."""
    cfg = SMALL[name]
    case = make_case(cfg)
    moe.set_gemm_tile_n(bn)
    try:
        plan = run_gpu(case)
    finally:
        moe.set_gemm_tile_n(0)
    ref = run_oracle(case)
    compare_routing(plan, ref, cfg.dtype)
    compare_dispatch(plan, ref)
    compare_output(plan, ref, cfg.dtype)


@pytest.mark.parametrize("name", ["swiglu_e8", "gelu_e16_hot", "swiglu_e128_top8", "many_tiles"])
def test_gemm_tile_order_changes_no_bit(name):
    """N-fastest tiles inside each expert (the blocks running together share a
    row tile instead of a weight tile) give the same bits as the default
    M-fastest order, and the oracle's layer."""
    cfg = SMALL[name]
    case = make_case(cfg)
    base = run_gpu(case)
    moe.set_gemm_order(2)
    try:
        plan = run_gpu(case)
    finally:
        moe.set_gemm_order(0)
    moe.check()
    A = int(base.disp.offsets[-1].item())
    assert torch.equal(plan.h[:A], base.h[:A])
    assert torch.equal(plan.y_perm[:A], base.y_perm[:A])
    assert torch.equal(plan.y, base.y)
    compare_output(plan, run_oracle(case), cfg.dtype)


@pytest.mark.parametrize("name", ["swiglu_e8", "swiglu_e128_top8"])
def test_launch_overlap_off_changes_no_bit(name):
    """Plain stream order instead of programmatic dependent launches between
    the library's kernels gives the same bits (the overlap only moves launch
    and set-up work)."""
    cfg = SMALL[name]
    case = make_case(cfg)
    base = run_gpu(case)
    y0, h0 = base.y.clone(), base.h.clone()
    moe.set_launch_overlap(False)
    try:
        plan = run_gpu(case)
    finally:
        moe.set_launch_overlap(True)
    moe.check()
    A = int(plan.disp.offsets[-1].item())
    assert torch.equal(plan.h[:A], h0[:A])
    assert torch.equal(plan.y, y0)


@pytest.mark.parametrize("name", ["swiglu_e8", "gelu_e16_hot", "swiglu_e64_zipf", "swiglu_e128_top8", "many_tiles",
                                  "gelu_e8_tail"])
def test_forward_gemm_tma_store_changes_no_bit(name):
    """The forward GEMMs' output blocks written by TMA stores (the default)
    and by per-thread stores give the same h, y_perm and y bits (SwiGLU and
    GELU up projections, gate-scaled down projection), and the oracle's
    layer: ragged last M tiles (per-thread rows), several tiles per block,
    and (gelu_e8_tail) half-width last-wave units with a ragged N tile.  The
    TMA stores apply from 3 row tiles per expert on average (swiglu_e8,
    many_tiles, gelu_e8_tail); the other cases check that the weight-bound
    launches keep the per-thread stores."""
    cfg = C("gelu_e8_tail", 5500, 448, 8, 2, 384, "gelu", 4.0, "bf16") if name == "gelu_e8_tail" else SMALL[name]
    case = make_case(cfg)
    base = run_gpu(case)
    moe.set_gemm_tma_store(False)
    try:
        plan = run_gpu(case)
    finally:
        moe.set_gemm_tma_store(True)
    moe.check()
    A = int(base.disp.offsets[-1].item())
    assert torch.equal(plan.h[:A], base.h[:A])
    assert torch.equal(plan.y_perm[:A], base.y_perm[:A])
    assert torch.equal(plan.y, base.y)
    compare_output(base, run_oracle(case), cfg.dtype)


def _halves_apply(plan, n_out, sms):
    """Whether a forward GEMM of n_out columns (256-column tiles) runs its last
    wave as half-width units: its tiles end in a wave that uses at most half
    of the blocks (the launch's grid is min(SMs, the host's tile bound))."""
    kept = plan.disp.kept.cpu().numpy().astype(np.int64)
    n_tiles = -(-n_out // 256)
    tiles = int(sum(-(-int(c) // 128) for c in kept)) * n_tiles
    grid = min(sms, (-(-plan.rows_max // 128) + len(kept)) * n_tiles)
    tail = tiles % grid
    return 0 < tail and 2 * tail <= grid


@pytest.mark.parametrize("name", ["gelu_e8_tail", "gelu_e16_hot"])
def test_gemm_half_width_last_wave_changes_no_bit(name):
    """A last wave of R <= SMs/2 tiles run as 2R half-width units (GELU up
    and gate-scaled down GEMMs) gives the same bits as whole tiles, and the
    oracle's layer.  gelu_e8_tail is sized so that both GEMMs take that path
    on 148 SMs (~1375 rows = 11 M tiles per expert, 2 N tiles: ~176 tiles,
    a last wave of ~28), with a ragged last N tile in both (F = 384: the
    second half of the second up tile is past F; d = 448: the second half of
    the second down tile holds 64 columns)."""
    cfg = C("gelu_e8_tail", 5500, 448, 8, 2, 384, "gelu", 4.0, "bf16") if name == "gelu_e8_tail" else SMALL[name]
    case = make_case(cfg)
    base = run_gpu(case)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if name == "gelu_e8_tail" and sms >= 128:
        assert _halves_apply(base, cfg.F, sms) and _halves_apply(base, cfg.d, sms)
    moe.set_gemm_tail_halves(False)
    try:
        plan = run_gpu(case)
    finally:
        moe.set_gemm_tail_halves(True)
    moe.check()
    A = int(base.disp.offsets[-1].item())
    assert torch.equal(plan.h[:A], base.h[:A])
    assert torch.equal(plan.y_perm[:A], base.y_perm[:A])
    assert torch.equal(plan.y, base.y)
    compare_output(base, run_oracle(case), cfg.dtype)


@pytest.mark.parametrize("name", ["swiglu_e8", "gelu_e16_hot", "swiglu_e64_zipf", "swiglu_e128_top8", "small_T",
                                  "gelu_e32_norenorm"])
def test_cta_pair_gemm_kernel(name):
    """The CTA-pair (2-SM) grouped GEMMs, forced, against the oracle.  A short
    wait limit turns any pipeline stall into a reported timeout."""
    cfg = SMALL[name]
    case = make_case(cfg)
    moe.set_gemm_kernel(2)
    moe.set_wait_limit(400_000_000)
    try:
        plan = run_gpu(case)
    finally:
        moe.set_gemm_kernel(0)
        moe.set_wait_limit(0)
    ref = run_oracle(case)
    compare_routing(plan, ref, cfg.dtype)
    compare_dispatch(plan, ref)
    compare_output(plan, ref, cfg.dtype)


@pytest.mark.parametrize("name", ["swiglu_e8", "gelu_e16_hot", "swiglu_e64_zipf", "swiglu_e128_top8", "small_T",
                                  "gelu_e32_norenorm", "bf16_e160_top16"])
def test_gathered_up_projection(name):
    """MoEPlan(gather=True): no permuted copy of x; the up GEMM reads x rows
    through row_token with TMA four-row gathers.  Against the oracle, and
    bitwise against the materialised-x_perm path (same operands, same
    accumulation order)."""
    cfg = SMALL[name]
    case = make_case(cfg)
    moe.set_wait_limit(400_000_000)
    try:
        plan = moe.MoEPlan(cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.act, torch.bfloat16, case["cap"],
                           case["x"].device, cfg.alpha, cfg.renorm, gather=True)
        run_gpu(case, plan)
    finally:
        moe.set_wait_limit(0)
    assert plan.disp.x_perm is None
    ref = run_oracle(case)
    compare_routing(plan, ref, cfg.dtype)
    compare_dispatch(plan, ref)
    compare_output(plan, ref, cfg.dtype)
    base = run_gpu(case)
    A = int(plan.disp.offsets[-1].item())
    assert torch.equal(plan.h[:A], base.h[:A])
    assert torch.equal(plan.y, base.y)


def test_identity_experts_return_x_bf16():
    """w1 = w2 = I, act = identity, renormalised gates, dropless: y = x up to
    the bf16 roundings of y_perm and y."""
    T, d, E, k = 700, 128, 8, 2
    cfg = C("ident", T, d, E, k, d, "identity", 0.0, "bf16")
    ri = synth.make_routing_inputs(cfg)
    case = make_case(cfg, routing=ri)
    eye = torch.eye(d, dtype=torch.bfloat16, device="cuda").expand(E, d, d).contiguous()
    case["w1"], case["w2"] = eye, eye
    plan = run_gpu(case)
    y = plan.y.float().cpu().numpy()
    x = case["x_h"].float().numpy()
    assert rel_fro(y, x) < 8e-3
    assert int(plan.disp.n_dropped.item()) == 0


@pytest.mark.parametrize("T,k,E,cap", [(8192, 2, 64, 160), (8193, 2, 64, 160), (2048, 8, 128, 100),
                                       (4097, 8, 128, 300), (1, 1, 8, 1), (33, 16, 256, 2),
                                       (32768, 2, 8, 9000), (9001, 8, 128, 700), (70001, 1, 16, 5000),
                                       (32768, 2, 16, 3000), (65537, 1, 16, 3000)])
def test_dispatch_both_rank_paths_against_oracle(T, k, E, cap):
    """The histogram + rank kernels with chunks of 256 assignments (T*k <=
    65536) and of 1024 (larger T*k) against the oracle's queue simulation: counts, kept,
    n_dropped, offsets (exclusive scan of kept) and every slot's row, bit for
    bit, on skewed expert choices (distinct experts per token)."""
    g = torch.Generator().manual_seed(T * 31 + k)
    w = torch.arange(E, 0, -1, dtype=torch.float64) ** 1.5          # skewed: low experts are hot
    idx = torch.multinomial(w.expand(T, E), k, replacement=False, generator=g).to(torch.int32)
    gate = torch.rand(T, k, generator=g)
    x = torch.randn(T, 64, generator=g).to(torch.bfloat16)
    D = moe.dispatch(idx.cuda(), gate.cuda(), x.cuda(), E, cap)
    moe.check()
    counts, kept, pos, nd = oracle.dispatch(idx.numpy(), E, cap)
    assert np.array_equal(D.counts.cpu().numpy(), counts)
    assert np.array_equal(D.kept.cpu().numpy(), kept)
    assert int(D.n_dropped.cpu()) == nd
    off = np.concatenate([[0], np.cumsum(kept)]).astype(np.int32)
    assert np.array_equal(D.offsets.cpu().numpy(), off)
    want = np.where(pos >= 0, off[idx.numpy()] + pos, -1)
    sr = D.slot_row.cpu().numpy()
    assert np.array_equal(sr, want)
    rows = sr[sr >= 0]
    tok = np.nonzero(sr >= 0)[0]
    assert np.array_equal(D.row_token.cpu().numpy()[rows], tok)
    assert np.array_equal(D.row_gate.cpu().numpy()[rows], gate.numpy()[sr >= 0])
    assert torch.equal(D.x_perm[torch.as_tensor(rows, dtype=torch.long).cuda()].cpu(), x[torch.as_tensor(tok)])


@pytest.mark.parametrize("d", [2112, 192])
def test_dispatch_rows_of_partial_chunks(d):
    """The row scatter moves rows in 2 KB chunks staged by bulk copies; rows of
    2112 bf16 (4224 bytes: chunks of 2048, 2048 and 128 bytes) and 192 bf16
    (384 bytes, one partial chunk) land bit for bit, every kept slot row."""
    T, k, E, cap = 3000, 2, 16, 300
    g = torch.Generator().manual_seed(d)
    w = torch.arange(E, 0, -1, dtype=torch.float64)
    idx = torch.multinomial(w.expand(T, E), k, replacement=False, generator=g).to(torch.int32)
    gate = torch.rand(T, k, generator=g)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    D = moe.dispatch(idx.cuda(), gate.cuda(), x.cuda(), E, cap)
    moe.check()
    sr = D.slot_row.cpu().numpy()
    rows = sr[sr >= 0]
    tok = np.nonzero(sr >= 0)[0]
    assert len(rows) > 0 and int(D.n_dropped.item()) > 0
    assert torch.equal(D.x_perm[torch.as_tensor(rows, dtype=torch.long).cuda()].cpu(), x[torch.as_tensor(tok)])


def test_combine_aux_equals_the_two_calls():
    """moe_combine_aux: the same y and the same loss bits as moe_combine then moe_aux_loss."""
    cfg = SMALL["swiglu_e8"]
    case = make_case(cfg)
    plan = moe.MoEPlan(cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.act, torch.bfloat16, case["cap"], "cuda", cfg.alpha,
                       cfg.renorm)
    plan.run(case["x"], case["W"], case["b"], case["w1"], case["w2"])
    D = plan.disp
    y1 = moe.combine(plan.y_perm, D.slot_row)
    l1 = moe.aux_loss(D.counts, plan.prob_sum, cfg.T, cfg.alpha)
    y2, l2 = moe.combine_aux(plan.y_perm, D.slot_row, D.counts, plan.prob_sum, cfg.alpha)
    moe.check()
    assert torch.equal(y1, y2) and torch.equal(l1, l2)
    assert torch.equal(plan.y, y2) and torch.equal(plan.loss, l2)


def test_capacity_zero_drops_everything():
    cfg = C("cap0", 256, 128, 8, 2, 128, "swiglu", 0.001, "bf16")
    case = make_case(cfg)
    assert case["cap"] == 0
    plan = run_gpu(case)
    assert int(plan.disp.n_dropped.item()) == cfg.T * cfg.k
    assert (plan.disp.kept.cpu() == 0).all() and (plan.disp.slot_row.cpu() == -1).all()
    assert torch.count_nonzero(plan.y).item() == 0
    ref = run_oracle(case, tokens=[0])
    assert abs(plan.loss.item() - ref["loss"]) <= 2e-4 * ref["loss"]


SMALL_E_ROUTER = {
    # E = 1 (every token to the one expert), the smallest d
    "r_e1": C("r_e1", 257, 256, 1, 1, 128, "gelu", 1.0, "bf16"),
    # E = 3, d = 768 (three warps), two hot experts over capacity
    "r_e3_k2_hot": C("r_e3_k2_hot", 1001, 768, 3, 2, 128, "swiglu", 1.25, "bf16", bias="hot2"),
    # E = 5, k = 4, no renormalisation, an odd token count
    "r_e5_k4": C("r_e5_k4", 333, 256, 5, 4, 128, "gelu", 2.0, "bf16", renorm=False),
    # E = k = 8 at the largest d (512 threads per block), dropless
    "r_e8_k8_d4096": C("r_e8_k8_d4096", 600, 4096, 8, 8, 128, "swiglu", 0.0, "bf16"),
    # one token
    "r_e8_T1": C("r_e8_T1", 1, 512, 8, 2, 128, "gelu", 1.0, "bf16"),
    # more than one wave of 64-token blocks, a ragged odd last block
    "r_e7_two_waves": C("r_e7_two_waves", 148 * 64 + 37, 256, 7, 2, 128, "gelu", 1.25, "bf16"),
}


@pytest.mark.parametrize("name", list(SMALL_E_ROUTER))
def test_small_e_router_against_oracle_and_tensor_core_router(name):
    """The CUDA-core router for E <= 8 and the tensor-core router (the
    default) on the same inputs: both against the oracle's routing, dispatch
    and layer; their top-k indices are identical (near-ties are conditioned
    away)."""
    cfg = SMALL_E_ROUTER[name]
    case = make_case(cfg)
    ref = run_oracle(case)
    plans = []
    for kind in (2, 1):
        moe.set_router_kernel(kind)
        try:
            plan = run_gpu(case)
        finally:
            moe.set_router_kernel(0)
        compare_routing(plan, ref, cfg.dtype)
        compare_dispatch(plan, ref)
        compare_output(plan, ref, cfg.dtype)
        plans.append(plan.topk_idx.clone())
    assert torch.equal(plans[0], plans[1])


def test_single_expert_dense_layer():
    cfg = C("dense", 300, 128, 1, 1, 256, "gelu", 0.0, "bf16")
    case = make_case(cfg)
    plan = run_gpu(case)
    ref = run_oracle(case)
    compare_routing(plan, ref, "bf16")
    compare_dispatch(plan, ref)
    compare_output(plan, ref, "bf16")


@pytest.mark.parametrize("xdtype", ["f32", "bf16"])
def test_exact_ties_go_to_lower_index(xdtype):
    """One-hot x rows make every logit an exact table entry; the table repeats
    values on purpose, so GPU and oracle must both break ties by index."""
    T, d, E, k = 96, 64, 16, 4
    rng = np.random.default_rng(5)
    table = (rng.integers(-6, 7, size=(E, d)) / 8.0).astype(np.float32)
    table[5] = table[3]
    table[11] = table[2]
    x = np.zeros((T, d), dtype=np.float32)
    x[np.arange(T), np.arange(T) % d] = 1.0
    cfg = C("ties", T, d, E, k, 128, "swiglu", 0.0, xdtype)
    xt = torch.from_numpy(x)
    ri = synth.RoutingInputs(x=xt.to(torch.bfloat16) if xdtype == "bf16" else xt, W=torch.from_numpy(table), b=None)
    case = make_case(cfg, condition=False, routing=ri)
    idx, gate, ps = moe.route(case["x"], case["W"], None, k)
    ref_idx, ref_gate, ref_ps = oracle.route(oracle.router_logits(ri.x, ri.W), k)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    # one-hot x: every logit is an exact table entry on both paths
    np.testing.assert_allclose(gate.cpu().numpy(), ref_gate, rtol=1e-5)
    np.testing.assert_allclose(ps.cpu().numpy(), ref_ps, rtol=1e-5)


def test_run_to_run_bitwise_determinism():
    cfg = SMALL["swiglu_e64_zipf"]
    case = make_case(cfg)
    p1 = run_gpu(case)
    snap = [t.clone() for t in (p1.topk_idx, p1.topk_gate, p1.prob_sum, p1.disp.slot_row, p1.y, p1.loss)]
    p2 = run_gpu(case, plan=p1)
    for a, b in zip(snap, (p2.topk_idx, p2.topk_gate, p2.prob_sum, p2.disp.slot_row, p2.y, p2.loss)):
        assert torch.equal(a, b)


def test_cuda_graph_replay_matches_eager():
    """The five calls captured once into a CUDA graph and replayed on new data
    in the same input tensors give the same bits as eager runs."""
    cfg = SMALL["swiglu_e8"]
    case = make_case(cfg)
    eager = run_gpu(case)
    ref = [t.clone() for t in (eager.topk_idx, eager.topk_gate, eager.prob_sum, eager.disp.slot_row, eager.y,
                               eager.loss)]
    plan = moe.MoEPlan(cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.act, torch.bfloat16, case["cap"], "cuda",
                       cfg.alpha, cfg.renorm)
    x = torch.zeros_like(case["x"])
    graph = plan.capture(x, case["W"], case["b"], case["w1"], case["w2"])
    x.copy_(case["x"])
    graph.replay()
    moe.check()
    got = (plan.topk_idx, plan.topk_gate, plan.prob_sum, plan.disp.slot_row, plan.y, plan.loss)
    for a, b in zip(ref, got):
        assert torch.equal(a, b)


def test_empty_batch():
    x = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    W = torch.randn(8, 128, device="cuda")
    idx, gate, ps = moe.route(x, W, None, 2)
    torch.cuda.synchronize()
    assert idx.shape == (0, 2) and torch.count_nonzero(ps).item() == 0
    D = moe.dispatch(idx, gate, x, 8, 4)
    torch.cuda.synchronize()
    assert (D.counts.cpu() == 0).all() and (D.offsets.cpu() == 0).all() and D.n_dropped.item() == 0
    moe.check()


def test_bad_expert_id_is_reported_not_trapped():
    T, k, E, d = 64, 2, 8, 128
    idx = torch.zeros(T, k, dtype=torch.int32, device="cuda")
    idx[3, 1] = 99
    gate = torch.full((T, k), 0.5, device="cuda")
    x = torch.zeros(T, d, dtype=torch.bfloat16, device="cuda")
    D = moe.dispatch(idx, gate, x, E, T)
    with pytest.raises(moe.MoEError) as ei:
        moe.check()
    assert ei.value.code == 1
    assert D.slot_row[3, 1].item() == -1
    moe.check()   # status was cleared


def test_wait_time_limit_path_reports_timeout():
    """A barrier nothing completes, under a ~1 ms limit: the kernel records a
    timeout and returns; the context stays usable."""
    moe.set_wait_limit(2_000_000)
    try:
        moe.selftest_wait_timeout()
        with pytest.raises(moe.MoEError) as ei:
            moe.check()
        assert ei.value.code == 5
    finally:
        moe.set_wait_limit(0)
    moe.check()
    test_tiny_fp32_layer_full()
