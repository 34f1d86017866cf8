"""CPU oracle of the MoE-layer forward -- TEST INFRASTRUCTURE ONLY.

Thin ctypes wrapper around ``moe_oracle.c`` (fp64, plain loops).  Only the
tests, the package smoke check and the benchmark's CPU-baseline leg may import
this package; the product path never does.  It shares no code with the CUDA
library.  See ``moe_oracle.c`` for the method statement and page citations.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")

F32, BF16 = 0, 1
ACTS = {"gelu": 0, "swiglu": 1, "identity": 2}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FP contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = load(build())
    return _lib


def load(path: str):
    """A ctypes handle on an oracle library built from this source (the tests
    also load deliberately broken copies to check that the pins catch them)."""
    L = ctypes.CDLL(path)
    P, I64, I32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
    L.orc_capacity.restype = I64
    L.orc_capacity.argtypes = [I64, I32, D]
    L.orc_router_logits.argtypes = [P, I32, P, P, I64, I32, I32, P]
    L.orc_route.argtypes = [P, I64, I32, I32, I32, P, P, P, P]
    L.orc_dispatch.argtypes = [P, I64, I32, I32, I64, P, P, P, P]
    L.orc_expert_ffn_row.argtypes = [P, I32, P, P, I32, I32, I32, I32, I32, P, P]
    L.orc_combine.argtypes = [P, I32, P, I64, P, P, P, I32, P, P, I32, I32, I32, I32, P]
    L.orc_aux_loss.restype = D
    L.orc_aux_loss.argtypes = [P, P, I64, I32, D]
    L.orc_num_threads.restype = I32
    L.orc_route_grouped.argtypes = [P, I64, I32, I32, I32, I32, I32, P, P, P, P]
    L.orc_logsumexp.argtypes = [P, I64, I32, P]
    L.orc_z_loss.restype = D
    L.orc_z_loss.argtypes = [P, I64, D]
    return L


def _host(a):
    """(contiguous host array keeping memory alive, dtype code)."""
    if isinstance(a, torch.Tensor):
        a = a.detach().to("cpu").contiguous()
        if a.dtype == torch.bfloat16:
            return a.view(torch.int16).numpy(), BF16
        if a.dtype == torch.float32:
            return a.numpy(), F32
        raise TypeError(f"unsupported tensor dtype {a.dtype}")
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError(f"unsupported array dtype {a.dtype}")


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return lib().orc_num_threads()


def capacity(T: int, E: int, cf: float) -> int:
    return int(lib().orc_capacity(T, E, float(cf)))


def router_logits(x, W, b=None) -> np.ndarray:
    xa, xdt = _host(x)
    Wa = np.ascontiguousarray(W.detach().cpu().numpy() if isinstance(W, torch.Tensor) else W,
                              dtype=np.float32)
    ba = None
    if b is not None:
        ba = np.ascontiguousarray(b.detach().cpu().numpy() if isinstance(b, torch.Tensor) else b,
                                  dtype=np.float32)
    T, d = xa.shape
    E = Wa.shape[0]
    L = np.empty((T, E), dtype=np.float64)
    lib().orc_router_logits(_ptr(xa), xdt, _ptr(Wa), _ptr(ba), T, d, E, _ptr(L))
    return L


def route(L: np.ndarray, k: int, renorm: bool = True, want_prob: bool = False):
    """(idx [T,k] int32, gate [T,k] f64, prob_sum [E] f64[, prob [T,E]])."""
    L = np.ascontiguousarray(L, dtype=np.float64)
    T, E = L.shape
    idx = np.empty((T, k), dtype=np.int32)
    gate = np.empty((T, k), dtype=np.float64)
    ps = np.empty(E, dtype=np.float64)
    prob = np.empty((T, E), dtype=np.float64) if want_prob else None
    lib().orc_route(_ptr(L), T, E, k, int(bool(renorm)), _ptr(idx), _ptr(gate), _ptr(prob), _ptr(ps))
    return (idx, gate, ps, prob) if want_prob else (idx, gate, ps)


def route_grouped(L: np.ndarray, k: int, n_group: int, topk_group: int, renorm: bool = True,
                  want_prob: bool = False):
    """Group-limited routing: top-k among the experts of the topk_group best
    of n_group contiguous expert groups (group score = its largest logit)."""
    L = np.ascontiguousarray(L, dtype=np.float64)
    T, E = L.shape
    if n_group < 1 or E % n_group or not 1 <= topk_group <= n_group or k > topk_group * (E // n_group):
        raise ValueError("need E % n_group == 0, 1 <= topk_group <= n_group, k <= topk_group * E / n_group")
    idx = np.empty((T, k), dtype=np.int32)
    gate = np.empty((T, k), dtype=np.float64)
    ps = np.empty(E, dtype=np.float64)
    prob = np.empty((T, E), dtype=np.float64) if want_prob else None
    lib().orc_route_grouped(_ptr(L), T, E, k, int(bool(renorm)), int(n_group), int(topk_group), _ptr(idx),
                            _ptr(gate), _ptr(prob), _ptr(ps))
    return (idx, gate, ps, prob) if want_prob else (idx, gate, ps)


def logsumexp(L: np.ndarray) -> np.ndarray:
    """lse [T] = log sum_e exp(L[t, e])."""
    L = np.ascontiguousarray(L, dtype=np.float64)
    T, E = L.shape
    out = np.empty(T, dtype=np.float64)
    lib().orc_logsumexp(_ptr(L), T, E, _ptr(out))
    return out


def z_loss(lse: np.ndarray, beta: float) -> float:
    """Router z-loss beta * mean_t lse[t]^2."""
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    return float(lib().orc_z_loss(_ptr(lse), lse.size, float(beta)))


def decision_gaps(L: np.ndarray, k: int, n_group: int = 1, topk_group: int = 1) -> np.ndarray:
    """Smallest logit gap, per token, among the comparisons that decide the
    routing: the top k+1 logits (ungrouped), or, with groups, the best
    topk_group+1 group scores and the top k+1 logits inside the kept groups.
    Input conditioning uses it to keep every choice far from a tie."""
    L = np.asarray(L, dtype=np.float64)
    T, E = L.shape

    def top_gaps(v, m):
        top = -np.sort(-v, axis=1)[:, :m]
        return (top[:, :-1] - top[:, 1:]).min(axis=1) if top.shape[1] > 1 else np.full(v.shape[0], np.inf)

    if n_group <= 1:
        return top_gaps(L, min(k + 1, E))
    gsz = E // n_group
    score = L.reshape(T, n_group, gsz).max(axis=2)
    gap = top_gaps(score, min(topk_group + 1, n_group))
    ranked = np.argsort(-score, axis=1, kind="stable")[:, :topk_group]
    keep = np.zeros((T, n_group), dtype=bool)
    np.put_along_axis(keep, ranked, True, axis=1)
    Lm = np.where(np.repeat(keep, gsz, axis=1), L, -np.inf)
    m = min(k + 1, topk_group * gsz)
    inner = top_gaps(Lm, m)
    return np.minimum(gap, inner)


def dispatch(idx: np.ndarray, E: int, cap: int):
    """(counts [E], kept [E], pos [T,k] (-1 = dropped), n_dropped)."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    counts = np.empty(E, dtype=np.int32)
    kept = np.empty(E, dtype=np.int32)
    pos = np.empty((T, k), dtype=np.int32)
    nd = ctypes.c_int64(0)
    lib().orc_dispatch(_ptr(idx), T, k, E, int(cap), _ptr(counts), _ptr(kept), _ptr(pos),
                       ctypes.byref(nd))
    return counts, kept, pos, int(nd.value)


def expert_ffn_row(v, w1, w2, e: int, act: str):
    """(a [F], out [d]) of expert e applied to one row v."""
    va, vdt = _host(v)
    w1a, wdt = _host(w1)
    w2a, wdt2 = _host(w2)
    assert wdt == wdt2
    d = va.shape[-1]
    F = w2a.shape[-1]
    a = np.empty(F, dtype=np.float64)
    out = np.empty(d, dtype=np.float64)
    lib().orc_expert_ffn_row(_ptr(va), vdt, _ptr(w1a), _ptr(w2a), wdt, int(e), d, F, ACTS[act],
                             _ptr(a), _ptr(out))
    return a, out


def combine(x, tokens: Sequence[int], idx, gate, pos, w1, w2, act: str) -> np.ndarray:
    """y rows [len(tokens), d] of the layer output for the listed tokens."""
    xa, xdt = _host(x)
    w1a, wdt = _host(w1)
    w2a, _ = _host(w2)
    T, d = xa.shape
    F = w2a.shape[-1]
    toks = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    gate = np.ascontiguousarray(gate, dtype=np.float64)
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    k = idx.shape[1]
    y = np.empty((toks.size, d), dtype=np.float64)
    lib().orc_combine(_ptr(xa), xdt, _ptr(toks), toks.size, _ptr(idx), _ptr(gate), _ptr(pos), k,
                      _ptr(w1a), _ptr(w2a), wdt, d, F, ACTS[act], _ptr(y))
    return y


def aux_loss(counts, prob_sum, T: int, alpha: float) -> float:
    counts = np.ascontiguousarray(counts, dtype=np.int32)
    ps = np.ascontiguousarray(prob_sum, dtype=np.float64)
    return float(lib().orc_aux_loss(_ptr(counts), _ptr(ps), int(T), counts.size, float(alpha)))


def forward(x, W, b, w1, w2, *, k: int, cap: int, act: str, renorm: bool = True,
            alpha: float = 0.01, tokens: Optional[Sequence[int]] = None, n_group: int = 1,
            topk_group: int = 1, z_beta: float = 0.0, aux_post_drop: bool = False) -> dict:
    """The whole layer: routing and dispatch for every token, y for ``tokens``
    (all tokens when None), the aux loss (f_i before drops, or after them with
    ``aux_post_drop``), the per-token log-sum-exp of the logits and the router
    z-loss with coefficient ``z_beta``."""
    L = router_logits(x, W, b)
    T, E = L.shape
    if n_group > 1:
        idx, gate, ps = route_grouped(L, k, n_group, topk_group, renorm)
    else:
        idx, gate, ps = route(L, k, renorm)
    counts, kept, pos, nd = dispatch(idx, E, cap)
    toks = np.arange(T, dtype=np.int32) if tokens is None else np.asarray(tokens, dtype=np.int32)
    y = combine(x, toks, idx, gate, pos, w1, w2, act)
    lse = logsumexp(L)
    return dict(logits=L, idx=idx, gate=gate, prob_sum=ps, counts=counts, kept=kept, pos=pos,
                n_dropped=nd, tokens=toks, y=y, loss=aux_loss(kept if aux_post_drop else counts, ps, T, alpha),
                lse=lse, z_loss=z_loss(lse, z_beta))
