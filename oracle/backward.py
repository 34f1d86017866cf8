"""CPU oracle of the MoE-layer backward -- TEST INFRASTRUCTURE ONLY.

The gradient of the forward that ``moe_oracle.c`` defines, by the chain rule,
step by step in reverse order of the forward, in float64 numpy.  Only the
tests, the package smoke check and the benchmark's CPU legs use it; the CUDA
library never does.

Sources.  The expert-parallelism tutorial "专家并行：混合专家模型的分布式训练方案"
(§2.1: gate, dispatch, expert compute, combine; §5.1: the auxiliary loss is
added to the training objective and its gradient pushes the router towards
even use of the experts) and the deployment guide "细粒度专家并行部署实践与优化指南"
(步骤三 item 3: expert compute and the reverse exchange that returns the
gradients) state that the layer is trained through these steps; the pages
give no formula for the backward, so it is the derivative of the forward:

  y[t]      = sum over kept slots j of g[t,j] * o[t,j],  o = w2[e] act(w1[e] x[t])
  L         = <dy, y> + aux_weight * L_aux + z_weight * L_z
  L_aux     = alpha * E * sum_e f_e * (1/T) sum_t p[t,e]     (f_e = counts or kept / T, a constant)
  L_z       = z_beta * (1/T) * sum_t lse[t]^2                (router z-loss, ST-MoE eq. 5)

The top-k choice, the capacity cut and f_e are piecewise constant in the
inputs, so they carry no gradient (the routing is taken from the forward
oracle).  A dropped slot contributes nothing to y, so its gate gets a zero
gradient; with renormalisation the gate g_j = p_j / S divides by the sum S
over all k chosen experts, dropped ones included (the forward's reading).

Step by step (per kept slot r of expert e, token t, gate g):
  dgate_r = <dy[t], o_r>
  do_r    = g * dy[t]
  dw2[e] += do_r a_r^T;   da_r = w2[e]^T do_r
  dz_r    = act'(z_r) da_r   (GELU: Phi(z) + z phi(z); SwiGLU: gate part
            da * up * silu'(gate), up part da * silu(gate))
  dw1[e] += dz_r x[t]^T;  dx[t] += w1[e]^T dz_r
then for every token:
  dp[e_j] = (dgate_j - sum_i dgate_i g_i) / S   (renorm)  or  dgate_j
  dp[e]  += aux_weight * alpha * E * f_e / T
  dl      = p * (dp - <p, dp>) + z_weight * (2 z_beta / T) * lse * p
  dW     += dl^T x;   db += sum_t dl;   dx[t] += W^T dl[t]
"""
from __future__ import annotations

import math

import numpy as np
import scipy.special

from . import _host, dispatch, logsumexp, route, route_grouped, router_logits


def _f64(a) -> np.ndarray:
    """Exact float64 copy of a torch tensor or array (bf16 values widened)."""
    h, dt = _host(a)
    if dt == 1:   # bf16 bits -> float32 -> float64
        u = h.view(np.uint16).astype(np.uint32) << 16
        return u.view(np.float32).astype(np.float64)
    return h.astype(np.float64)


def act_forward(z: np.ndarray, act: str) -> np.ndarray:
    if act == "gelu":
        return z * 0.5 * (1.0 + _erf(z / math.sqrt(2.0)))
    if act == "swiglu":
        F = z.shape[1] // 2
        gate, up = z[:, :F], z[:, F:]
        return gate / (1.0 + np.exp(-gate)) * up
    return z.copy()


def act_backward(z: np.ndarray, da: np.ndarray, act: str) -> np.ndarray:
    """dz from the pre-activation z and the gradient da of the activation output."""
    if act == "gelu":
        cdf = 0.5 * (1.0 + _erf(z / math.sqrt(2.0)))
        pdf = np.exp(-0.5 * z * z) / math.sqrt(2.0 * math.pi)
        return da * (cdf + z * pdf)
    if act == "swiglu":
        F = z.shape[1] // 2
        gate, up = z[:, :F], z[:, F:]
        s = 1.0 / (1.0 + np.exp(-gate))
        silu = gate * s
        dsilu = s * (1.0 + gate * (1.0 - s))
        return np.concatenate([da * up * dsilu, da * silu], axis=1)
    return da.copy()


_erf = scipy.special.erf   # float64 erf (library routine)


def backward(x, W, b, w1, w2, dy, *, k: int, cap: int, act: str, renorm: bool = True, alpha: float = 0.01,
             aux_weight: float = 1.0, z_beta: float = 0.0, z_weight: float = 1.0, aux_post_drop: bool = False,
             n_group: int = 1, topk_group: int = 1, wgrad_dtype=np.float64) -> dict:
    """Gradients of L (module docstring) with respect to x, the router W and b,
    w1 and w2, plus the intermediates dgate [T,k] and dl [T,E].  Everything is
    computed in float64; ``wgrad_dtype`` only sets how dw1 and dw2 are stored
    (float32 keeps full-size layers within host memory).  The expert weights
    are widened one expert at a time."""
    X, Wr, DY = _f64(x), _f64(W), _f64(dy)
    L = router_logits(x, W, b)
    T, E = L.shape
    if n_group > 1:
        idx, gate, _, P = route_grouped(L, k, n_group, topk_group, renorm, want_prob=True)
    else:
        idx, gate, _, P = route(L, k, renorm, want_prob=True)
    counts, kept, pos, _ = dispatch(idx, E, cap)
    d = X.shape[1]

    # expert part, one expert at a time over its kept slots
    dgate = np.zeros((T, k))
    dX = np.zeros((T, d))
    dW1 = np.zeros(tuple(w1.shape), dtype=wgrad_dtype)
    dW2 = np.zeros(tuple(w2.shape), dtype=wgrad_dtype)
    for e in range(E):
        ts, js = np.nonzero((idx == e) & (pos >= 0))
        if ts.size == 0:
            continue
        W1e, W2e = _f64(w1[e]), _f64(w2[e])
        Xe = X[ts]
        Z = Xe @ W1e.T
        A = act_forward(Z, act)
        O = A @ W2e.T
        g = gate[ts, js]
        dgate[ts, js] = np.sum(DY[ts] * O, axis=1)
        dO = g[:, None] * DY[ts]
        dW2[e] = dO.T @ A
        dA = dO @ W2e
        dZ = act_backward(Z, dA, act)
        dW1[e] = dZ.T @ Xe
        np.add.at(dX, ts, dZ @ W1e)

    # gates -> full softmax probabilities
    dP = np.zeros((T, E))
    for t in range(T):
        sel = idx[t]
        if renorm:
            S = P[t, sel].sum()
            dP[t, sel] += (dgate[t] - np.dot(dgate[t], gate[t])) / S
        else:
            dP[t, sel] += dgate[t]
    f = (kept if aux_post_drop else counts).astype(np.float64) / T
    dP += aux_weight * alpha * E * f[None, :] / T

    # softmax and z-loss -> logits
    dL = P * (dP - np.sum(P * dP, axis=1, keepdims=True))
    lse = logsumexp(L)
    dL += z_weight * (2.0 * z_beta / T) * lse[:, None] * P

    # the linear router
    dWr = dL.T @ X
    db = dL.sum(axis=0)
    dX += dL @ Wr
    return dict(dx=dX, dW=dWr, db=db, dw1=dW1, dw2=dW2, dgate=dgate, dl=dL, idx=idx, gate=gate, pos=pos,
                counts=counts, kept=kept, prob=P, lse=lse)
