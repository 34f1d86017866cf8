"""Guard canaries: every output buffer of the forward and the backward is a
view into a larger allocation whose tail holds a known bit pattern; after the
calls the tails must be untouched (no kernel writes past its output), and the
rows the contract leaves alone (permuted rows past the kept count) too."""
import pytest
import torch

import top_routing_expert_02_b300 as moe
from top_routing_expert_02_b300 import synth

from moe_cases import make_case

pytestmark = pytest.mark.gpu

PAD = 257   # extra elements after every output


def guarded(shape, dtype, fill):
    n = 1
    for s in shape:
        n *= s
    big = torch.full((n + PAD,), fill, dtype=dtype, device="cuda")
    return big, big[:n].view(*shape)


def untouched(big, n, fill):
    return bool((big[n:] == fill).all())


@pytest.mark.parametrize("name", ["swiglu_e8", "gelu_e16_hot"])
def test_forward_outputs_stay_in_bounds(name):
    # cf 2.0: some experts overflow and some do not, so fewer rows are kept than allocated
    cfg = {"swiglu_e8": synth.MoEConfig("c8", 1000, 256, 8, 2, 384, "swiglu", 2.0, "bf16"),
           "gelu_e16_hot": synth.MoEConfig("c16", 900, 192, 16, 2, 320, "gelu", 1.0, "bf16", bias="hot2")}[name]
    case = make_case(cfg)
    x, W, b, w1, w2 = case["x"], case["W"], case["b"], case["w1"], case["w2"]
    T, d, E, k, F = cfg.T, cfg.d, cfg.E, cfg.k, cfg.F
    R = moe.perm_rows_max(T, k, E, case["cap"])
    i32, f32, bf = torch.int32, torch.float32, torch.bfloat16
    bufs = {}

    def g(key, shape, dtype, fill):
        bufs[key] = guarded(shape, dtype, fill) + (fill,)
        return bufs[key][1]

    idx = g("idx", (T, k), i32, -777)
    gate = g("gate", (T, k), f32, 7.5)
    ps = g("ps", (E,), f32, 7.5)
    moe.route(x, W, b, k, topk_idx=idx, topk_gate=gate, prob_sum=ps)
    D = moe.Dispatched(g("counts", (E,), i32, -777), g("kept", (E,), i32, -777), g("offsets", (E + 1,), i32, -777),
                       g("slot", (T, k), i32, -777), g("row_token", (R,), i32, -777), g("row_gate", (R,), f32, 7.5),
                       g("x_perm", (R, d), bf, 3.0), g("nd", (1,), i32, -777), R)
    moe.dispatch(idx, gate, x, E, case["cap"], out=D)
    h = g("h", (R, F), bf, 3.0)
    yp = g("y_perm", (R, d), bf, 3.0)
    moe.expert_up(D.x_perm, D.offsets, D.kept, w1, F, cfg.act, R, h=h)
    moe.expert_down(h, D.offsets, D.kept, w2, D.row_gate, R, y_perm=yp)
    y = g("y", (T, d), bf, 3.0)
    moe.combine(yp, D.slot_row, y=y)
    loss = g("loss", (1,), f32, 7.5)
    moe.aux_loss(D.counts, ps, T, cfg.alpha, loss=loss)
    moe.check()
    for key, (big, view, fill) in bufs.items():
        assert untouched(big, view.numel(), fill), key
    A = int(D.offsets[-1])
    if name == "swiglu_e8":
        assert A < R
    for key in ("x_perm", "h", "y_perm"):
        assert bool((bufs[key][1][A:] == 3.0).all()), key          # rows past the kept count are left alone


def test_backward_outputs_stay_in_bounds():
    cfg = synth.MoEConfig("cb", 700, 256, 8, 2, 384, "swiglu", 1.25, "bf16")
    case = make_case(cfg)
    plan = moe.MoEPlan(cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.act, torch.bfloat16, case["cap"], "cuda", train=True)
    plan.run(case["x"], case["W"], case["b"], case["w1"], case["w2"])
    B = plan._bwd_buffers(torch.device("cuda"))
    # replace every backward output with a guarded view of the same shape
    bufs = {}
    for key in ("do_perm", "dgate", "dz", "dx_perm", "dw1", "dw2", "dl", "dx", "dW", "db"):
        t = B[key]
        fill = 3.0 if t.dtype == torch.bfloat16 else 7.5
        big, view = guarded(tuple(t.shape), t.dtype, fill)
        B[key] = view
        bufs[key] = (big, view, fill)
    dy = torch.randn(cfg.T, cfg.d, device="cuda").to(torch.bfloat16)
    plan.backward(case["x"], case["W"], case["w1"], case["w2"], dy)
    moe.check()
    for key, (big, view, fill) in bufs.items():
        assert untouched(big, view.numel(), fill), key
