"""Pins of the CPU backward oracle (oracle/backward.py).

Three independent roads to the same gradients: torch autograd through an
fp64 forward written here from the method's definition (routing fixed, as it
is piecewise constant); central finite differences of the C forward oracle
with perturbations exactly representable in fp32; and closed forms (identity
experts pass dy straight through; a uniform router's aux-loss gradient)."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import oracle
from oracle import backward as B


def _grid(g, shape, scale, step=2.0 ** -12):
    """Random normals rounded to a 2^-12 grid: +-2^-16 perturbations of them are exact in fp32."""
    return (torch.round(torch.randn(*shape, generator=g, dtype=torch.float64) * scale / step) * step).float()


def _case(seed, T=24, d=16, E=8, k=2, F=8, act="swiglu", n_group=1, topk_group=1, bias=True):
    g = torch.Generator().manual_seed(seed)
    N1 = 2 * F if act == "swiglu" else F
    for _ in range(50):
        x = _grid(g, (T, d), 1.0)
        W = _grid(g, (E, d), 0.5)
        b = _grid(g, (E,), 0.3) if bias else None
        L = oracle.router_logits(x, W, b)
        if (oracle.decision_gaps(L, k, n_group, topk_group) > 1e-3).all():
            break
    else:
        raise RuntimeError("no tie-free draw")
    w1 = _grid(g, (E, N1, d), 1.0 / math.sqrt(d))
    w2 = _grid(g, (E, d, F), 1.0 / math.sqrt(F))
    dy = _grid(g, (T, d), 1.0)
    return x, W, b, w1, w2, dy


def torch_loss(x, W, b, w1, w2, dy, idx, pos, act, renorm, alpha, aux_weight, z_beta, z_weight, f):
    """L = <dy, y> + aux_weight L_aux + z_weight L_z, written slot by slot."""
    T, d = x.shape
    E = W.shape[0]
    F = w2.shape[2]
    l = x @ W.T + (b if b is not None else 0.0)
    p = torch.softmax(l, dim=1)
    sel = p.gather(1, torch.from_numpy(idx).long())
    gate = sel / sel.sum(1, keepdim=True) if renorm else sel
    rows = []
    for t in range(T):
        yt = torch.zeros(d, dtype=x.dtype)
        for j in range(idx.shape[1]):
            if pos[t, j] < 0:
                continue
            e = int(idx[t, j])
            z = w1[e] @ x[t]
            a = Fn.gelu(z) if act == "gelu" else (Fn.silu(z[:F]) * z[F:] if act == "swiglu" else z)
            yt = yt + gate[t, j] * (w2[e] @ a)
        rows.append(yt)
    y = torch.stack(rows)
    aux = alpha * E * torch.sum(torch.from_numpy(f) * p.mean(0))
    zl = z_beta * torch.mean(torch.logsumexp(l, dim=1) ** 2)
    return torch.sum(dy * y) + aux_weight * aux + z_weight * zl


CFGS = [
    dict(act="swiglu", renorm=True, cap=4, z_beta=0.0, post=False, grp=(1, 1)),
    dict(act="gelu", renorm=False, cap=3, z_beta=0.05, post=False, grp=(1, 1)),
    dict(act="identity", renorm=True, cap=100, z_beta=0.02, post=True, grp=(1, 1)),
    dict(act="swiglu", renorm=True, cap=5, z_beta=0.01, post=True, grp=(4, 2)),
    dict(act="gelu", renorm=True, cap=2, z_beta=0.0, post=False, grp=(2, 1)),
]


@pytest.mark.parametrize("i", range(len(CFGS)))
def test_backward_matches_autograd(i):
    c = CFGS[i]
    G, M = c["grp"]
    x, W, b, w1, w2, dy = _case(10 + i, act=c["act"], n_group=G, topk_group=M)
    alpha, aw, zw = 0.01, 0.7, 1.3
    r = B.backward(x, W, b, w1, w2, dy, k=2, cap=c["cap"], act=c["act"], renorm=c["renorm"], alpha=alpha,
                   aux_weight=aw, z_beta=c["z_beta"], z_weight=zw, aux_post_drop=c["post"], n_group=G,
                   topk_group=M)
    assert (r["pos"] < 0).any() or c["cap"] >= 24          # drops are exercised where the capacity bites
    f = (r["kept"] if c["post"] else r["counts"]).astype(np.float64) / x.shape[0]
    leaves = [t.double().requires_grad_() for t in (x, W, b, w1, w2)]
    loss = torch_loss(*leaves, dy.double(), r["idx"], r["pos"], c["act"], c["renorm"], alpha, aw, c["z_beta"], zw,
                      f)
    loss.backward()
    for name, leaf in zip(("dx", "dW", "db", "dw1", "dw2"), leaves):
        np.testing.assert_allclose(r[name], leaf.grad.numpy(), rtol=1e-10, atol=1e-12, err_msg=name)


def _c_loss(x, W, b, w1, w2, dy, k, cap, act, renorm, alpha, aw, z_beta, zw, post, G, M):
    """L from the C forward oracle, in fp64."""
    out = oracle.forward(x, W, b, w1, w2, k=k, cap=cap, act=act, renorm=renorm, alpha=alpha, n_group=G,
                         topk_group=M, z_beta=z_beta, aux_post_drop=post)
    return float(np.sum(dy.double().numpy() * out["y"])) + aw * out["loss"] + zw * out["z_loss"]


@pytest.mark.parametrize("i", [0, 1, 3])
def test_backward_matches_finite_differences_of_the_c_forward(i):
    """Central differences with h = 2^-16 on parameters held on a 2^-12 grid, so
    both perturbed values are exact in fp32 and the C oracle sees them as they
    are; every routing decision clears a 1e-3 margin, so none flips."""
    c = CFGS[i]
    G, M = c["grp"]
    x, W, b, w1, w2, dy = _case(10 + i, act=c["act"], n_group=G, topk_group=M)
    args = dict(k=2, cap=c["cap"], act=c["act"], renorm=c["renorm"], alpha=0.01, aw=0.7, z_beta=c["z_beta"],
                zw=1.3, post=c["post"], G=G, M=M)
    r = B.backward(x, W, b, w1, w2, dy, k=2, cap=c["cap"], act=c["act"], renorm=c["renorm"], alpha=0.01,
                   aux_weight=0.7, z_beta=c["z_beta"], z_weight=1.3, aux_post_drop=c["post"], n_group=G,
                   topk_group=M)
    h = 2.0 ** -16
    rng = np.random.default_rng(i)
    params = dict(x=x, W=W, b=b, w1=w1, w2=w2)
    grads = dict(x="dx", W="dW", b="db", w1="dw1", w2="dw2")
    for name, t in params.items():
        flat = t.view(-1)
        for pos in rng.choice(flat.numel(), size=6, replace=False):
            old = float(flat[pos])
            vals = []
            for s in (+1, -1):
                flat[pos] = old + s * h
                assert float(flat[pos]) == old + s * h          # exact in fp32
                vals.append(_c_loss(x, W, b, w1, w2, dy, args["k"], args["cap"], args["act"], args["renorm"],
                                    args["alpha"], args["aw"], args["z_beta"], args["zw"], args["post"], G, M))
            flat[pos] = old
            fd = (vals[0] - vals[1]) / (2 * h)
            an = r[grads[name]].reshape(-1)[pos]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, pos, fd, an)


def test_identity_experts_pass_dy_through():
    """w1 = w2 = I, identity activation, renormalised gates, no drops, no
    aux or z terms: y = x, so dx = dy and the router gets no gradient."""
    T, d, E, k = 20, 8, 4, 2
    g = torch.Generator().manual_seed(3)
    x = torch.randn(T, d, generator=g)
    W = torch.randn(E, d, generator=g)
    eye = torch.eye(d).expand(E, d, d).contiguous()
    dy = torch.randn(T, d, generator=g)
    r = B.backward(x, W, None, eye, eye, dy, k=k, cap=T, act="identity", aux_weight=0.0)
    np.testing.assert_allclose(r["dx"], dy.double().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["dW"], 0.0, atol=1e-12)
    np.testing.assert_allclose(r["db"], 0.0, atol=1e-12)


def test_aux_loss_gradient_of_a_uniform_router():
    """W = 0, b = 0 (p = 1/E), dy = 0: dl[t,e] = (c_e - mean c) / E with
    c_e = alpha E f_e / T, and dW = dl^T x."""
    T, d, E, k, alpha = 30, 6, 8, 2, 0.01
    g = torch.Generator().manual_seed(4)
    x = torch.randn(T, d, generator=g)
    W = torch.zeros(E, d)
    w1 = torch.randn(E, 4, d, generator=g)
    w2 = torch.randn(E, d, 4, generator=g)
    r = B.backward(x, W, torch.zeros(E), w1, w2, torch.zeros(T, d), k=k, cap=T, act="gelu", alpha=alpha)
    c = alpha * E * (r["counts"] / T) / T
    np.testing.assert_allclose(r["dl"], np.tile((c - c.mean()) / E, (T, 1)), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(r["dW"], r["dl"].T @ x.double().numpy(), rtol=1e-12, atol=1e-15)
