"""Seeded synthetic inputs for the MoE-layer forward.

This module only draws random numbers and lays them out; it computes nothing
of the layer itself (no logits, no softmax, no top-k, no dispatch, no FFN).
Both the CUDA path and the CPU oracle consume exactly the bytes it returns.

Recipe (one seed per workload, default 0):

* ``numpy.random.SeedSequence(seed).spawn(6)`` gives six independent streams,
  used in the order [x, router W, router bias, w1, w2, resample].
* ``x``  : PCG64 standard normal, float32, rounded once to bf16
  (round-to-nearest-even) for bf16 workloads.
* ``W``  : PCG64 normal with standard deviation ``router_std`` (fp32, [E, d]).
* ``b``  : no bias, or the workload's fixed skew (two hot experts, or a Zipf
  profile); drawn from nothing random.
* ``w1`` : [E, N1, d] with N1 = 2F for SwiGLU (rows 0..F-1 gate, F..2F-1 up)
  and N1 = F otherwise; ``w2`` : [E, d, F].  Both are normal with standard
  deviation 1/sqrt(fan_in), drawn with a ``torch.Generator`` on the device that
  will hold them (seeded from the w1 / w2 streams), expert by expert, then
  rounded to the workload dtype.  Copies handed to the oracle are the same
  bytes, copied to the host.
* ``resample``: fresh x rows for tokens whose router logits sit closer than a
  margin (see :func:`condition_near_ties`).  The logits themselves come from a
  caller-supplied function; this module only sorts and compares them.

"N(0, s)" in the workload descriptions means standard deviation s.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Callable, Optional

import numpy as np
import torch

__all__ = [
    "MoEConfig", "WORKLOADS", "workload", "RoutingInputs", "make_routing_inputs",
    "make_expert_weights", "condition_near_ties", "bias_vector",
]

# Offset of the two "hot" experts' router bias in the E=16 GELU workload.  It
# was chosen by bisection (step 0.01) so that each hot expert receives about
# three times the mean number of (token, choice) assignments, T*k/E; the
# calibration script next to the golden fixtures reproduces it.
HOT2_BIAS = 1.33


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    """One MoE-layer forward workload (all sizes are plain integers)."""
    name: str
    T: int                 # tokens
    d: int                 # model width
    E: int                 # experts
    k: int                 # experts chosen per token
    F: int                 # expert FFN width (d_ff)
    act: str               # "gelu" | "swiglu" | "identity"
    cf: float              # capacity factor; <= 0 means dropless (capacity T)
    dtype: str             # "f32" | "bf16"  (x, w1, w2, h, y_perm, y)
    router_std: float = 0.02
    bias: str = "none"     # "none" | "hot2" | "zipf"
    alpha: float = 0.01    # aux-loss weight
    renorm: bool = True    # divide the k gates by their sum
    seed: int = 0

    @property
    def N1(self) -> int:
        return 2 * self.F if self.act == "swiglu" else self.F

    @property
    def dropless(self) -> bool:
        return self.cf <= 0

    def replace(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)

    def describe(self) -> str:
        cap = "dropless" if self.dropless else f"cf={self.cf:g}"
        return (f"{self.dtype} MoE forward T={self.T} d={self.d} E={self.E} top-{self.k} "
                f"F={self.F} {self.act} {cap} bias={self.bias}")


def _mk(name, T, d, E, k, F, act, cf, dtype, **kw):
    return MoEConfig(name=name, T=T, d=d, E=E, k=k, F=F, act=act, cf=cf, dtype=dtype, **kw)


WORKLOADS = {
    # tiny fp32 layer; the oracle runs it in well under a second
    "tiny_fp32": _mk("tiny_fp32", 64, 128, 8, 2, 256, "gelu", 1.25, "f32"),
    # d=4096, 8 experts, top-2, SwiGLU d_ff=14336, uniform-ish routing
    "e8_swiglu": _mk("e8_swiglu", 4096, 4096, 8, 2, 14336, "swiglu", 1.25, "bf16"),
    # the 4096->16384->4096 GELU expert; two hot experts overflow capacity
    "e16_gelu_hot2": _mk("e16_gelu_hot2", 8192, 4096, 16, 2, 16384, "gelu", 1.0, "bf16",
                         bias="hot2"),
    # fine-grained: 64 small SwiGLU experts, Zipf(1.1)-skewed router bias
    "e64_zipf": _mk("e64_zipf", 16384, 2048, 64, 2, 1408, "swiglu", 1.25, "bf16",
                    bias="zipf"),
}
# small profiling case of the e8 SwiGLU layer (d_ff 2048): weights 400 MB, still
# larger than L2, short kernels, so a full ncu capture stays small
WORKLOADS["prof_e8_swiglu_F2048"] = _mk("prof_e8_swiglu_F2048", 4096, 4096, 8, 2, 2048, "swiglu", 1.25, "bf16")
# router profiling cases: x above L2 (134 / 268 MB), small experts
WORKLOADS["prof_route_e8_T32768"] = _mk("prof_route_e8_T32768", 32768, 4096, 8, 2, 128, "swiglu", 1.25, "bf16")
WORKLOADS["prof_route_e128_T16384"] = _mk("prof_route_e128_T16384", 16384, 4096, 128, 8, 128, "swiglu", 1.25,
                                          "bf16")
# profiling cases of the many-expert layer: the e128 per-token shape with tiny
# experts (route, dispatch and combine bytes per token as at full size, a few
# GB on the device), and 32 experts at 2048 rows each (the per-expert GEMM
# shape of T=32768, top-8 over 128 experts)
WORKLOADS["prof_e128_T16384_F128"] = _mk("prof_e128_T16384_F128", 16384, 4096, 128, 8, 128, "swiglu", 0.0, "bf16")
WORKLOADS["prof_e32_top8_T8192"] = _mk("prof_e32_top8_T8192", 8192, 4096, 32, 8, 1536, "swiglu", 0.0, "bf16")
for _T in (512, 2048, 8192, 32768):
    WORKLOADS[f"e128_top8_T{_T}"] = _mk(f"e128_top8_T{_T}", _T, 4096, 128, 8, 1536,
                                        "swiglu", 0.0, "bf16")


def workload(name: str) -> MoEConfig:
    return WORKLOADS[name]


def bias_vector(cfg: MoEConfig) -> Optional[np.ndarray]:
    """The router bias of a workload, fp32 [E], or None."""
    if cfg.bias == "none":
        return None
    b = np.zeros(cfg.E, dtype=np.float64)
    if cfg.bias == "hot2":
        b[:2] = HOT2_BIAS
    elif cfg.bias == "zipf":
        # exp(b_e) proportional to (e+1)^-1.1: a Zipf(1.1) profile, expert 0 hottest
        b = -1.1 * np.log(np.arange(cfg.E, dtype=np.float64) + 1.0)
    else:
        raise ValueError(f"unknown bias kind {cfg.bias!r}")
    return b.astype(np.float32)


def _streams(seed: int):
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(6)]


def _torch_seed(seed: int, which: int) -> int:
    ss = np.random.SeedSequence(seed).spawn(6)[which]
    return int(ss.generate_state(1, dtype=np.uint64)[0] & np.uint64((1 << 63) - 1))


def _to_dtype(a32: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a32, dtype=np.float32))
    return t.to(torch.bfloat16) if dtype == "bf16" else t


@dataclasses.dataclass
class RoutingInputs:
    x: torch.Tensor                  # [T, d] host tensor, f32 or bf16
    W: torch.Tensor                  # [E, d] host fp32
    b: Optional[torch.Tensor]        # [E] host fp32 or None
    redrawn: int = 0                 # rows replaced by condition_near_ties
    _resample: Optional[np.random.Generator] = None


def make_routing_inputs(cfg: MoEConfig) -> RoutingInputs:
    """x, router W and router b of a workload, on the host."""
    rs = _streams(cfg.seed)
    x = _to_dtype(rs[0].standard_normal((cfg.T, cfg.d), dtype=np.float32), cfg.dtype)
    W = torch.from_numpy(rs[1].standard_normal((cfg.E, cfg.d), dtype=np.float32)
                         * np.float32(cfg.router_std))
    bv = bias_vector(cfg)
    b = None if bv is None else torch.from_numpy(bv)
    return RoutingInputs(x=x, W=W, b=b, redrawn=0, _resample=rs[5])


def make_expert_weights(cfg: MoEConfig, device="cpu"):
    """(w1 [E, N1, d], w2 [E, d, F]) in the workload dtype, on ``device``."""
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    out = []
    for which, shape, fan_in in ((3, (cfg.N1, cfg.d), cfg.d), (4, (cfg.d, cfg.F), cfg.F)):
        g = torch.Generator(device=device)
        g.manual_seed(_torch_seed(cfg.seed, which))
        w = torch.empty((cfg.E,) + shape, dtype=tdt, device=device)
        std = 1.0 / math.sqrt(fan_in)
        for e in range(cfg.E):
            w[e].copy_(torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std)
        out.append(w)
    return out[0], out[1]


def condition_near_ties(cfg: MoEConfig, ri: RoutingInputs,
                        logits_fn: Callable[[torch.Tensor, torch.Tensor, Optional[torch.Tensor]], np.ndarray],
                        margin: float = 1e-3, max_passes: int = 100,
                        gaps_fn: Optional[Callable[[np.ndarray], np.ndarray]] = None) -> RoutingInputs:
    """Redraw x rows whose top-(k+1) router logits are closer than ``margin``.

    ``logits_fn(x_rows, W, b)`` returns the float64 logits [rows, E] of the
    given rows; the caller supplies it.  ``gaps_fn(logits)``, when given,
    replaces the top-(k+1) test: it returns each row's smallest gap among the
    comparisons that decide its routing (a routing variant knows which those
    are).  Rows are redrawn in ascending token order from the resample
    stream, and only redrawn rows are re-checked, so the result depends on
    the seed alone.  With the margin in place every top-k choice and every
    k-rank is decided by more than 1e-3, far above the rounding error of an
    fp32 logit.
    """
    m = min(cfg.k + 1, cfg.E)
    rows = np.arange(cfg.T)
    for _ in range(max_passes):
        if rows.size == 0:
            return ri
        L = np.asarray(logits_fn(ri.x[torch.from_numpy(rows)], ri.W, ri.b), dtype=np.float64)
        if gaps_fn is not None:
            bad = rows[np.asarray(gaps_fn(L)) < margin]
        else:
            top = -np.sort(-L, axis=1)[:, :m]
            bad = rows[((top[:, :-1] - top[:, 1:]) < margin).any(axis=1)] if m > 1 else rows[:0]
        for t in bad:
            fresh = ri._resample.standard_normal((1, cfg.d), dtype=np.float32)
            ri.x[int(t)] = _to_dtype(fresh, cfg.dtype)[0]
        ri.redrawn += int(bad.size)
        rows = bad
    raise RuntimeError("near-tie redraw did not converge")
