"""B300-native MoE-layer forward (router, capacity dispatch, expert FFN,
combine, aux loss) for sm_103a.

This module is the Python binding of ``libmoe_b300.so``: it only marshals
torch tensors (device pointers, sizes, the current CUDA stream) into the C ABI
declared in ``include/moe_b300.h`` and turns status codes into exceptions.
Every step of the layer runs in the library's CUDA kernels; there is no
fallback.  PyTorch provides device memory and streams.

Entry points (same names as the C ABI, without the ``moe_`` prefix):
``route``, ``dispatch``, ``expert_up``, ``expert_up_gathered``, ``expert_down``, ``expert_ffn``,
``combine``, ``aux_loss``, plus ``capacity``, ``perm_rows_max``,
``workspace_bytes``, ``check``.  :class:`MoEPlan` holds preallocated buffers
for one layer shape and enqueues the five calls; :func:`moe_forward` is the
one-shot form.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

__all__ = [
    "MoEError", "lib", "capacity", "perm_rows_max", "workspace_bytes", "route", "z_loss", "dispatch", "expert_up",
    "expert_up_gathered", "expert_up_z", "expert_down", "expert_dgrad", "expert_dgrad_act", "permute_rows", "transpose_experts", "combine_bwd", "act_bwd", "wgrad_cols",
    "pack_segments_t", "expert_wgrad", "expert_wgrad_rows", "route_bwd", "grad_x", "router_wgrad", "router_grads", "expert_ffn", "combine", "combine_aux", "aux_loss", "check", "dispatch_noalloc", "set_wait_limit", "set_gemm_tile_n", "set_wgrad_order", "set_gemm_kernel", "selftest_wait_timeout",
    "MoEPlan", "moe_forward", "ACT", "CALL",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe_b300.so")

ACT = {"gelu": 0, "swiglu": 1, "identity": 2}
CALL = {"route": 0, "dispatch": 1, "ffn": 2, "router_wgrad": 3, "router_grads": 4}
_DT = {torch.float32: 0, torch.bfloat16: 1}
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT"}


class MoEError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({_lib.moe_status_string(code).decode()})")


_lib = None

_P, _I64, _I32, _D, _F, _SZ, _U64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double,
                                     ctypes.c_float, ctypes.c_size_t, ctypes.c_uint64)
_SIGS = {
    "moe_capacity": (_I64, [_I64, _I32, _D]),
    "moe_perm_rows_max": (_I64, [_I64, _I32, _I32, _I64]),
    "moe_workspace_bytes": (_SZ, [_I32, _I64, _I32, _I32, _I32, _I32, _I32, _I32]),
    "moe_status_string": (ctypes.c_char_p, [_I32]),
    "moe_abi_version": (_I32, []),
    "moe_route": (_I32, [_P, _I32, _P, _P, _I64, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _SZ, _P]),
    "moe_dispatch": (_I32, [_P, _P, _I64, _I32, _I32, _I64, _P, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P,
                            _P, _SZ, _P]),
    "moe_expert_up": (_I32, [_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _I64, _P, _P]),
    "moe_expert_dgrad_act": (_I32, [_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _P, _I64, _P, _P]),
    "moe_permute_rows": (_I32, [_P, _P, _I64, _I32, _I32, _P, _P]),
    "moe_expert_dgrad": (_I32, [_P, _P, _P, _I32, _I32, _I32, _I32, _P, _I64, _P, _P]),
    "moe_expert_up_z": (_I32, [_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _I64, _P, _P, _P]),
    "moe_expert_up_gathered": (_I32, [_P, _I64, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _I64, _P, _P]),
    "moe_expert_down": (_I32, [_P, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _I64, _P, _P]),
    "moe_expert_ffn": (_I32, [_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _I64, _P, _P, _P, _SZ,
                              _P]),
    "moe_combine": (_I32, [_P, _P, _I64, _I32, _I32, _I32, _P, _P]),
    "moe_aux_loss": (_I32, [_P, _P, _I64, _I32, _F, _P, _P]),
    "moe_combine_aux": (_I32, [_P, _P, _I64, _I32, _I32, _I32, _P, _P, _P, _I32, _F, _P, _P]),
    "moe_dispatch_noalloc": (_I32, [_P, _P, _I64, _I32, _I32, _I64, _P, _I32, _I32, _P, _P, _P, _P, _P, _P,
                                    _P, _P, _P]),
    "moe_route_ex": (_I32, [_P, _I32, _P, _P, _I64, _I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P,
                            _SZ, _P]),
    "moe_transpose_experts": (_I32, [_P, _I32, _I32, _I32, _I32, _P, _P]),
    "moe_combine_bwd": (_I32, [_P, _P, _P, _P, _I64, _I32, _I32, _I32, _P, _P, _P]),
    "moe_act_bwd": (_I32, [_P, _P, _P, _I32, _I32, _I32, _I32, _I64, _P, _P]),
    "moe_wgrad_cols": (_I64, [_I64, _I32]),
    "moe_pack_segments_t": (_I32, [_P, _P, _P, _I32, _I32, _I64, _I64, _I32, _P, _P]),
    "moe_expert_wgrad": (_I32, [_P, _P, _P, _I32, _I32, _I32, _I64, _I32, _P, _I32, _P]),
    "moe_expert_wgrad_rows": (_I32, [_P, _P, _P, _P, _I32, _I32, _I32, _I64, _I32, _P, _I32, _P]),
    "moe_route_bwd": (_I32, [_P, _P, _P, _P, _I64, _I32, _I32, _I32, _F, _F, _P, _P]),
    "moe_grad_x": (_I32, [_P, _P, _P, _P, _I64, _I32, _I32, _I32, _I32, _P, _P]),
    "moe_router_wgrad": (_I32, [_P, _P, _I32, _I64, _I32, _I32, _P, _P, _P, _SZ, _P]),
    "moe_router_grads": (_I32, [_P, _P, _P, _P, _P, _I64, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _SZ, _P]),
    "moe_z_loss": (_I32, [_P, _I64, _F, _P, _P]),
    "moe_check": (_I32, [_P]),
    "moe_set_wait_limit": (None, [_U64]),
    "moe_set_gemm_tile_n": (_I32, [_I32]),
    "moe_set_gemm_order": (_I32, [_I32]),
    "moe_set_gemm_tail_halves": (_I32, [_I32]),
    "moe_set_launch_overlap": (_I32, [_I32]),
    "moe_set_gemm_tma_store": (_I32, [_I32]),
    "moe_set_router_kernel": (_I32, [_I32]),
    "moe_set_wgrad_order": (_I32, [_I32]),
    "moe_set_gemm_kernel": (_I32, [_I32]),
    "moe_selftest_wait_timeout": (_I32, [_P]),
}


def lib():
    """The loaded CUDA library (built in-tree first if missing or stale)."""
    global _lib
    if _lib is None:
        from . import build as _build
        if _build.needs_build():
            _build.build_library()
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"CUDA library {LIB_PATH} is missing; run python -m top_routing_expert_02_b300.build")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the MoE library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dt(t: torch.Tensor) -> int:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}; use float32 or bfloat16") from None


# MOE_NVTX=1 wraps every call below in an NVTX range named after it (for
# nsight timelines); otherwise the functions are left as they are.
_NVTX = os.environ.get("MOE_NVTX", "") == "1"


def _traced(fn):
    if not _NVTX:
        return fn
    import functools

    @functools.wraps(fn)
    def wrapper(*args, **kwargs):
        torch.cuda.nvtx.range_push("moe_" + fn.__name__)
        try:
            return fn(*args, **kwargs)
        finally:
            torch.cuda.nvtx.range_pop()
    return wrapper


def _ok(fn: str, code: int):
    if code != 0:
        raise MoEError(fn, code)


def _empty_ws(nbytes: int, device):
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ host ---

def capacity(T: int, E: int, cf: float) -> int:
    return int(lib().moe_capacity(T, E, float(cf)))


def perm_rows_max(T: int, k: int, E: int, cap: int) -> int:
    return int(lib().moe_perm_rows_max(T, k, E, cap))


def workspace_bytes(call: str, T: int, d: int, E: int, k: int, F: int, act: str = "swiglu",
                    dtype: torch.dtype = torch.bfloat16) -> int:
    return int(lib().moe_workspace_bytes(CALL[call], T, d, E, k, F, ACT[act], _DT[dtype]))


def check(stream=None):
    """Synchronise the stream and raise if a kernel recorded a device error."""
    _ok("moe_check", lib().moe_check(_stream(stream)))


def set_wait_limit(cycles: int):
    lib().moe_set_wait_limit(int(cycles))


def set_gemm_tile_n(bn: int):
    """Force the bf16 expert GEMM tile width (128, 192, 256) or 0 for automatic."""
    _ok("moe_set_gemm_tile_n", lib().moe_set_gemm_tile_n(int(bn)))


def set_gemm_order(order: int):
    """Forward / data-gradient GEMM tile order: 0 automatic, 1 M-fastest, 2 N-fastest (results unchanged)."""
    _ok("moe_set_gemm_order", lib().moe_set_gemm_order(int(order)))


def set_gemm_tail_halves(on: bool):
    """Let a short last wave of the forward GEMMs run as half-width units (default on; results unchanged)."""
    _ok("moe_set_gemm_tail_halves", lib().moe_set_gemm_tail_halves(int(bool(on))))


def set_launch_overlap(on: bool):
    """Programmatic dependent launch between the library's kernels (default on; results unchanged)."""
    _ok("moe_set_launch_overlap", lib().moe_set_launch_overlap(int(bool(on))))


def set_router_kernel(kind: int):
    """bf16 router kernel: 0 automatic (tensor cores), 1 tensor cores, 2 CUDA cores for E <= 8 (where each applies)."""
    _ok("moe_set_router_kernel", lib().moe_set_router_kernel(int(kind)))


def set_gemm_tma_store(on: bool):
    """Forward GEMM output blocks by TMA stores (default on) or per-thread stores (results unchanged)."""
    _ok("moe_set_gemm_tma_store", lib().moe_set_gemm_tma_store(int(bool(on))))


def set_wgrad_order(order: int):
    """Weight-gradient tile order: 0 automatic, 1 M-fastest, 2 N-fastest (results unchanged)."""
    _ok("moe_set_wgrad_order", lib().moe_set_wgrad_order(int(order)))


def set_gemm_kernel(kind: int):
    """Force the bf16 expert GEMM kernel: 1 one-SM tiles, 2 CTA-pair tiles, 0 automatic."""
    _ok("moe_set_gemm_kernel", lib().moe_set_gemm_kernel(int(kind)))


def selftest_wait_timeout(stream=None):
    _ok("moe_selftest_wait_timeout", lib().moe_selftest_wait_timeout(_stream(stream)))


# --------------------------------------------------------------- compute ---

@_traced
def route(x, w_router, b_router, k: int, renorm: bool = True, *, topk_idx=None, topk_gate=None, prob_sum=None,
          ws=None, stream=None, n_group: int = 1, topk_group: int = 1, lse=None, logits=None):
    """Router (moe_route): returns (topk_idx [T,k] int32, topk_gate [T,k] f32, prob_sum [E] f32).

    ``n_group`` > 1 selects group-limited routing (moe_route_ex): top-k among
    the experts of the ``topk_group`` best of ``n_group`` contiguous groups.
    ``lse`` ([T] f32) receives each token's log-sum-exp of the logits and
    ``logits`` ([T, E] f32) the logits themselves (for the backward)."""
    T, d = x.shape
    E = w_router.shape[0]
    dev = x.device
    topk_idx = torch.empty((T, k), dtype=torch.int32, device=dev) if topk_idx is None else topk_idx
    topk_gate = torch.empty((T, k), dtype=torch.float32, device=dev) if topk_gate is None else topk_gate
    prob_sum = torch.empty(E, dtype=torch.float32, device=dev) if prob_sum is None else prob_sum
    need = workspace_bytes("route", T, d, E, k, 64)
    ws = _empty_ws(need, dev) if ws is None else ws
    if n_group == 1 and lse is None and logits is None:
        _ok("moe_route", lib().moe_route(_ptr(x), _dt(x), _ptr(w_router), _ptr(b_router), T, d, E, k, int(renorm),
                                         _ptr(topk_idx), _ptr(topk_gate), _ptr(prob_sum), _ptr(ws), ws.numel(),
                                         _stream(stream)))
    else:
        _ok("moe_route_ex", lib().moe_route_ex(
            _ptr(x), _dt(x), _ptr(w_router), _ptr(b_router), T, d, E, k, int(renorm), int(n_group), int(topk_group),
            _ptr(topk_idx), _ptr(topk_gate), _ptr(prob_sum), _ptr(lse), _ptr(logits), _ptr(ws), ws.numel(),
            _stream(stream)))
    return topk_idx, topk_gate, prob_sum


@dataclass
class Dispatched:
    counts: torch.Tensor
    kept: torch.Tensor
    offsets: torch.Tensor
    slot_row: torch.Tensor
    row_token: torch.Tensor
    row_gate: torch.Tensor
    x_perm: torch.Tensor
    n_dropped: torch.Tensor
    rows_max: int


@_traced
def dispatch(topk_idx, topk_gate, x, E: int, cap: int, *, out: Optional[Dispatched] = None, ws=None,
             stream=None, copy_rows: bool = True) -> Dispatched:
    """Capacity dispatch + row permutation (moe_dispatch).  With
    ``copy_rows=False`` (or ``out.x_perm`` None) no permuted copy of x is
    written: :func:`expert_up_gathered` reads x through ``row_token``."""
    T, k = topk_idx.shape
    d = x.shape[1]
    dev = x.device
    R = perm_rows_max(T, k, E, cap)
    if out is None:
        i32 = dict(dtype=torch.int32, device=dev)
        xp = torch.empty((max(R, 1), d), dtype=x.dtype, device=dev) if copy_rows else None
        out = Dispatched(torch.empty(E, **i32), torch.empty(E, **i32), torch.empty(E + 1, **i32),
                         torch.empty((T, k), **i32), torch.empty(max(R, 1), **i32),
                         torch.empty(max(R, 1), dtype=torch.float32, device=dev), xp, torch.empty(1, **i32), R)
    need = workspace_bytes("dispatch", T, d, E, k, 64)
    ws = _empty_ws(need, dev) if ws is None else ws
    _ok("moe_dispatch", lib().moe_dispatch(_ptr(topk_idx), _ptr(topk_gate), T, k, E, cap, _ptr(x), _dt(x), d,
                                           _ptr(out.counts), _ptr(out.kept), _ptr(out.offsets), _ptr(out.slot_row),
                                           _ptr(out.row_token), _ptr(out.row_gate), _ptr(out.x_perm),
                                           _ptr(out.n_dropped), _ptr(ws), ws.numel(), _stream(stream)))
    return out


@_traced
def dispatch_noalloc(topk_idx, topk_gate, x, E: int, cap: int, *, out: Optional[Dispatched] = None,
                     stream=None) -> Dispatched:
    """moe_dispatch_noalloc: dispatch with the library's built-in scratch
    instead of a workspace (for callers that cannot allocate device memory
    where they run the layer).  Outputs are allocated here only when ``out``
    is None; pass ``out`` to allocate nothing."""
    T, k = topk_idx.shape
    d = x.shape[1]
    dev = x.device
    R = perm_rows_max(T, k, E, cap)
    if out is None:
        i32 = dict(dtype=torch.int32, device=dev)
        out = Dispatched(torch.empty(E, **i32), torch.empty(E, **i32), torch.empty(E + 1, **i32),
                         torch.empty((T, k), **i32), torch.empty(max(R, 1), **i32),
                         torch.empty(max(R, 1), dtype=torch.float32, device=dev),
                         torch.empty((max(R, 1), d), dtype=x.dtype, device=dev), torch.empty(1, **i32), R)
    _ok("moe_dispatch_noalloc", lib().moe_dispatch_noalloc(
        _ptr(topk_idx), _ptr(topk_gate), T, k, E, cap, _ptr(x), _dt(x), d, _ptr(out.counts), _ptr(out.kept),
        _ptr(out.offsets), _ptr(out.slot_row), _ptr(out.row_token), _ptr(out.row_gate), _ptr(out.x_perm),
        _ptr(out.n_dropped), _stream(stream)))
    return out


@_traced
def expert_up(x_perm, offsets, kept, w1, F: int, act: str, rows_max: int, *, h=None, stream=None):
    E, _, d = w1.shape
    h = torch.empty((max(rows_max, 1), F), dtype=x_perm.dtype, device=x_perm.device) if h is None else h
    _ok("moe_expert_up", lib().moe_expert_up(_ptr(x_perm), _ptr(offsets), _ptr(kept), E, d, F, ACT[act],
                                             _dt(x_perm), _ptr(w1), rows_max, _ptr(h), _stream(stream)))
    return h


@_traced
def expert_up_z(x_perm, offsets, kept, w1, F: int, act: str, rows_max: int, *, h=None, z=None, stream=None):
    """moe_expert_up_z: h and the pre-activation z [rows, N1] (kept for the backward)."""
    E, N1, d = w1.shape
    h = torch.empty((max(rows_max, 1), F), dtype=x_perm.dtype, device=x_perm.device) if h is None else h
    z = torch.empty((max(rows_max, 1), N1), dtype=x_perm.dtype, device=x_perm.device) if z is None else z
    _ok("moe_expert_up_z", lib().moe_expert_up_z(_ptr(x_perm), _ptr(offsets), _ptr(kept), E, d, F, ACT[act],
                                                 _dt(x_perm), _ptr(w1), rows_max, _ptr(h), _ptr(z),
                                                 _stream(stream)))
    return h, z


@_traced
def expert_up_gathered(x, row_token, offsets, kept, w1, F: int, act: str, rows_max: int, *, h=None,
                       stream=None):
    """moe_expert_up with the A rows read from x at row_token (no x_perm)."""
    E, _, d = w1.shape
    T = x.shape[0]
    h = torch.empty((max(rows_max, 1), F), dtype=x.dtype, device=x.device) if h is None else h
    _ok("moe_expert_up_gathered", lib().moe_expert_up_gathered(
        _ptr(x), T, _ptr(row_token), _ptr(offsets), _ptr(kept), E, d, F, ACT[act], _dt(x), _ptr(w1), rows_max,
        _ptr(h), _stream(stream)))
    return h


@_traced
def expert_down(h, offsets, kept, w2, row_gate, rows_max: int, *, y_perm=None, stream=None):
    E, d, F = w2.shape
    y_perm = torch.empty((max(rows_max, 1), d), dtype=h.dtype, device=h.device) if y_perm is None else y_perm
    _ok("moe_expert_down", lib().moe_expert_down(_ptr(h), _ptr(offsets), _ptr(kept), E, d, F, _dt(h), _ptr(w2),
                                                 _ptr(row_gate), rows_max, _ptr(y_perm), _stream(stream)))
    return y_perm


@_traced
def expert_ffn(x_perm, offsets, kept, w1, w2, row_gate, act: str, rows_max: int, *, h=None, y_perm=None,
               stream=None):
    E, d, F = w2.shape
    dev = x_perm.device
    h = torch.empty((max(rows_max, 1), F), dtype=x_perm.dtype, device=dev) if h is None else h
    y_perm = torch.empty((max(rows_max, 1), d), dtype=x_perm.dtype, device=dev) if y_perm is None else y_perm
    _ok("moe_expert_ffn", lib().moe_expert_ffn(_ptr(x_perm), _ptr(offsets), _ptr(kept), E, d, F, ACT[act],
                                               _dt(x_perm), _ptr(w1), _ptr(w2), _ptr(row_gate), rows_max, _ptr(h),
                                               _ptr(y_perm), None, 0, _stream(stream)))
    return h, y_perm


@_traced
def combine(y_perm, slot_row, *, y=None, stream=None):
    T, k = slot_row.shape
    d = y_perm.shape[1]
    y = torch.empty((T, d), dtype=y_perm.dtype, device=y_perm.device) if y is None else y
    _ok("moe_combine", lib().moe_combine(_ptr(y_perm), _ptr(slot_row), T, k, d, _dt(y_perm), _ptr(y),
                                         _stream(stream)))
    return y


@_traced
def combine_aux(y_perm, slot_row, counts, prob_sum, alpha: float, *, y=None, loss=None, stream=None):
    """combine + aux loss in one launch (moe_combine_aux): returns (y, loss)."""
    T, k = slot_row.shape
    d = y_perm.shape[1]
    E = counts.shape[0]
    y = torch.empty((T, d), dtype=y_perm.dtype, device=y_perm.device) if y is None else y
    loss = torch.empty(1, dtype=torch.float32, device=y_perm.device) if loss is None else loss
    _ok("moe_combine_aux", lib().moe_combine_aux(_ptr(y_perm), _ptr(slot_row), T, k, d, _dt(y_perm), _ptr(y),
                                                 _ptr(counts), _ptr(prob_sum), E, float(alpha), _ptr(loss),
                                                 _stream(stream)))
    return y, loss


@_traced
def aux_loss(counts, prob_sum, T: int, alpha: float, *, loss=None, stream=None):
    E = counts.shape[0]
    loss = torch.empty(1, dtype=torch.float32, device=counts.device) if loss is None else loss
    _ok("moe_aux_loss", lib().moe_aux_loss(_ptr(counts), _ptr(prob_sum), T, E, float(alpha), _ptr(loss),
                                           _stream(stream)))
    return loss


@_traced
def z_loss(lse, beta: float, *, loss=None, stream=None):
    """Router z-loss beta * mean_t lse[t]^2 (moe_z_loss); lse from route(..., lse=)."""
    loss = torch.empty(1, dtype=torch.float32, device=lse.device) if loss is None else loss
    _ok("moe_z_loss", lib().moe_z_loss(_ptr(lse), lse.shape[0], float(beta), _ptr(loss), _stream(stream)))
    return loss


# --------------------------------------------------------------- backward ---

@_traced
def expert_dgrad_act(do_perm, offsets, kept, w2, z, act: str, rows_max: int, *, dz=None, stream=None):
    """dz = act'(z) * (do_perm . w2[e]) per kept row (moe_expert_dgrad_act)."""
    E, d, F = w2.shape
    dz = torch.empty_like(z) if dz is None else dz
    _ok("moe_expert_dgrad_act", lib().moe_expert_dgrad_act(_ptr(do_perm), _ptr(offsets), _ptr(kept), E, d, F,
                                                           ACT[act], _dt(do_perm), _ptr(w2), _ptr(z), rows_max,
                                                           _ptr(dz), _stream(stream)))
    return dz


@_traced
def permute_rows(src, index, *, out=None, stream=None):
    """out[i] = src[index[i]] (moe_permute_rows); index int32 on the device."""
    n = index.shape[0]
    d = src.shape[1]
    out = torch.empty((n, d), dtype=src.dtype, device=src.device) if out is None else out
    _ok("moe_permute_rows", lib().moe_permute_rows(_ptr(src), _ptr(index), n, d, _dt(src), _ptr(out),
                                                   _stream(stream)))
    return out


@_traced
def expert_dgrad(a, offsets, kept, w, rows_max: int, *, out=None, stream=None):
    """out [rows, N] = a[r] . w[e] per kept row r of expert e, w [E, K, N] as stored (moe_expert_dgrad)."""
    E, K, N = w.shape
    out = torch.empty((max(rows_max, 1), N), dtype=a.dtype, device=a.device) if out is None else out
    _ok("moe_expert_dgrad", lib().moe_expert_dgrad(_ptr(a), _ptr(offsets), _ptr(kept), E, K, N, _dt(a), _ptr(w),
                                                   rows_max, _ptr(out), _stream(stream)))
    return out


@_traced
def transpose_experts(w, *, out=None, stream=None):
    """w [E, R, C] -> [E, C, R] (moe_transpose_experts)."""
    E, R, C = w.shape
    out = torch.empty((E, C, R), dtype=w.dtype, device=w.device) if out is None else out
    _ok("moe_transpose_experts", lib().moe_transpose_experts(_ptr(w), E, R, C, _dt(w), _ptr(out), _stream(stream)))
    return out


@_traced
def combine_bwd(dy, slot_row, row_gate, y_perm, *, do_perm=None, dgate=None, stream=None):
    """(do_perm [rows, d], dgate [T, k] f32) (moe_combine_bwd)."""
    T, k = slot_row.shape
    d = dy.shape[1]
    do_perm = torch.empty_like(y_perm) if do_perm is None else do_perm
    dgate = torch.empty((T, k), dtype=torch.float32, device=dy.device) if dgate is None else dgate
    _ok("moe_combine_bwd", lib().moe_combine_bwd(_ptr(dy), _ptr(slot_row), _ptr(row_gate), _ptr(y_perm), T, k, d,
                                                 _dt(dy), _ptr(do_perm), _ptr(dgate), _stream(stream)))
    return do_perm, dgate


@_traced
def act_bwd(z, da, offsets, F: int, act: str, rows_max: int, *, dz=None, stream=None):
    """dz [rows, N1] from the pre-activation z and da (moe_act_bwd)."""
    E = offsets.shape[0] - 1
    dz = torch.empty_like(z) if dz is None else dz
    _ok("moe_act_bwd", lib().moe_act_bwd(_ptr(z), _ptr(da), _ptr(offsets), E, F, ACT[act], _dt(z), rows_max,
                                         _ptr(dz), _stream(stream)))
    return dz


def wgrad_cols(rows_max: int, E: int) -> int:
    return int(lib().moe_wgrad_cols(rows_max, E))


@_traced
def pack_segments_t(src, offsets, kept, rows_max: int, ld: int, *, out=None, stream=None):
    """src [rows, C] -> [C, ld], expert segments as zero-padded column blocks (moe_pack_segments_t)."""
    C = src.shape[1]
    E = kept.shape[0]
    out = torch.empty((C, ld), dtype=src.dtype, device=src.device) if out is None else out
    _ok("moe_pack_segments_t", lib().moe_pack_segments_t(_ptr(src), _ptr(offsets), _ptr(kept), E, C, rows_max, ld,
                                                         _dt(src), _ptr(out), _stream(stream)))
    return out


@_traced
def expert_wgrad(at, bt, kept, *, dw=None, dtype=torch.float32, stream=None):
    """dw [E, M, N] (fp32 or bf16) = per-expert at[:, seg] bt[:, seg]^T (moe_expert_wgrad)."""
    M, ld = at.shape
    N = bt.shape[0]
    E = kept.shape[0]
    dw = torch.empty((E, M, N), dtype=dtype, device=at.device) if dw is None else dw
    _ok("moe_expert_wgrad", lib().moe_expert_wgrad(_ptr(at), _ptr(bt), _ptr(kept), E, M, N, ld, _dt(at), _ptr(dw),
                                                   _dt(dw), _stream(stream)))
    return dw


@_traced
def expert_wgrad_rows(a, b, offsets, kept, rows_max: int, *, dw=None, dtype=torch.float32, stream=None):
    """dw [E, M, N] (fp32 or bf16) = per-expert a[seg]^T b[seg] over the row
    segments [offsets[e], offsets[e] + kept[e]) of a [rows, M], b [rows, N]
    (moe_expert_wgrad_rows)."""
    M, N = a.shape[1], b.shape[1]
    E = kept.shape[0]
    dw = torch.empty((E, M, N), dtype=dtype, device=a.device) if dw is None else dw
    _ok("moe_expert_wgrad_rows", lib().moe_expert_wgrad_rows(_ptr(a), _ptr(b), _ptr(offsets), _ptr(kept), E, M, N,
                                                             rows_max, _dt(a), _ptr(dw), _dt(dw), _stream(stream)))
    return dw


@_traced
def route_bwd(logits, topk_idx, dgate, counts, renorm: bool, aux_coef: float, z_coef: float, *, dl=None,
              stream=None):
    """dl [T, E] f32, the gradient at the router logits (moe_route_bwd)."""
    T, k = topk_idx.shape
    E = logits.shape[1]
    dl = torch.empty((T, E), dtype=torch.float32, device=logits.device) if dl is None else dl
    _ok("moe_route_bwd", lib().moe_route_bwd(_ptr(logits), _ptr(topk_idx), _ptr(dgate), _ptr(counts), T, E, k,
                                             int(renorm), float(aux_coef), float(z_coef), _ptr(dl),
                                             _stream(stream)))
    return dl


@_traced
def grad_x(dx_perm, slot_row, dl, w_router, *, dx=None, stream=None):
    """dx [T, d] (moe_grad_x)."""
    T, k = slot_row.shape
    E, d = w_router.shape
    dx = torch.empty((T, d), dtype=dx_perm.dtype, device=dx_perm.device) if dx is None else dx
    _ok("moe_grad_x", lib().moe_grad_x(_ptr(dx_perm), _ptr(slot_row), _ptr(dl), _ptr(w_router), T, k, E, d,
                                       _dt(dx_perm), _ptr(dx), _stream(stream)))
    return dx


@_traced
def router_wgrad(dl, x, *, dW=None, db=None, ws=None, stream=None):
    """(dW [E, d] f32, db [E] f32) (moe_router_wgrad)."""
    T, E = dl.shape
    d = x.shape[1]
    dW = torch.empty((E, d), dtype=torch.float32, device=x.device) if dW is None else dW
    db = torch.empty(E, dtype=torch.float32, device=x.device) if db is None else db
    need = workspace_bytes("router_wgrad", T, d, E, 1, 64)
    ws = _empty_ws(need, x.device) if ws is None else ws
    _ok("moe_router_wgrad", lib().moe_router_wgrad(_ptr(dl), _ptr(x), _dt(x), T, E, d, _ptr(dW), _ptr(db), _ptr(ws),
                                                   ws.numel(), _stream(stream)))
    return dW, db


@_traced
def router_grads(dx_perm, slot_row, dl, w_router, x, *, dx=None, dW=None, db=None, ws=None, stream=None):
    """(dx [T, d] bf16, dW [E, d] f32, db [E] f32) on the tensor cores (moe_router_grads)."""
    T, d = x.shape
    k = slot_row.shape[1]
    E = w_router.shape[0]
    dx = torch.empty((T, d), dtype=x.dtype, device=x.device) if dx is None else dx
    dW = torch.empty((E, d), dtype=torch.float32, device=x.device) if dW is None else dW
    db = torch.empty(E, dtype=torch.float32, device=x.device) if db is None else db
    ws = _empty_ws(workspace_bytes("router_grads", T, d, E, k, 64), x.device) if ws is None else ws
    _ok("moe_router_grads", lib().moe_router_grads(_ptr(dx_perm), _ptr(slot_row), _ptr(dl), _ptr(w_router), _ptr(x),
                                                   T, k, E, d, _dt(x), _ptr(dx), _ptr(dW), _ptr(db), _ptr(ws),
                                                   ws.numel(), _stream(stream)))
    return dx, dW, db


# ------------------------------------------------------------ whole layer ---

class MoEPlan:
    """Preallocated device buffers for one layer shape.

    ``run(x, w_router, b_router, w1, w2)`` enqueues route, dispatch, the
    expert FFN, combine and the aux loss on the current stream (no host
    synchronisation; safe to capture in a CUDA graph) and returns ``y``.
    Every intermediate stays readable as an attribute afterwards.

    ``gather=True`` (bf16 only) skips the permuted copy of x: the dispatch
    writes only the row maps and the up-projection gathers its rows from x
    (``disp.x_perm`` is then None).

    Routing variants: ``n_group``/``topk_group`` (group-limited top-k),
    ``z_beta`` (router z-loss into ``z_loss``, with the per-token
    log-sum-exp in ``lse``; None skips it) and ``aux_post_drop`` (f_i from
    the kept slots instead of every choice).

    ``train=True`` keeps the router logits and the pre-activation so that
    :meth:`backward` can run after :meth:`run` (bf16 layers, x_perm path);
    the expert weight gradients come out in ``grad_dtype`` (fp32 or bf16).
    """

    def __init__(self, T: int, d: int, E: int, k: int, F: int, act: str, dtype: torch.dtype, cap: int,
                 device="cuda", alpha: float = 0.01, renorm: bool = True, gather: bool = False, *,
                 n_group: int = 1, topk_group: int = 1, z_beta: Optional[float] = None,
                 aux_post_drop: bool = False, train: bool = False, grad_dtype: torch.dtype = torch.float32):
        self.T, self.d, self.E, self.k, self.F, self.act = T, d, E, k, F, act
        self.dtype, self.cap, self.alpha, self.renorm = dtype, int(cap), float(alpha), bool(renorm)
        self.n_group, self.topk_group = int(n_group), int(topk_group)
        self.z_beta = None if z_beta is None else float(z_beta)
        self.aux_post_drop = bool(aux_post_drop)
        if gather and dtype != torch.bfloat16:
            raise ValueError("the gathered up-projection is bf16 only")
        self.gather = bool(gather)
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        self.rows_max = R = perm_rows_max(T, k, E, cap)
        Rb = max(R, 1)
        self.topk_idx = torch.empty((T, k), **i32)
        self.topk_gate = torch.empty((T, k), **f32)
        self.prob_sum = torch.empty(E, **f32)
        self.disp = Dispatched(torch.empty(E, **i32), torch.empty(E, **i32), torch.empty(E + 1, **i32),
                               torch.empty((T, k), **i32), torch.empty(Rb, **i32), torch.empty(Rb, **f32),
                               None if self.gather else torch.empty((Rb, d), dtype=dtype, device=dev),
                               torch.empty(1, **i32), R)
        self.h = torch.empty((Rb, F), dtype=dtype, device=dev)
        self.y_perm = torch.empty((Rb, d), dtype=dtype, device=dev)
        self.y = torch.empty((T, d), dtype=dtype, device=dev)
        self.loss = torch.empty(1, **f32)
        self.train = bool(train)
        self.grad_dtype = grad_dtype
        if self.train and (dtype != torch.bfloat16 or self.gather):
            raise ValueError("the backward runs on bf16 layers with a materialised x_perm")
        self.logits = torch.empty((max(T, 1), E), **f32) if self.train else None
        N1 = 2 * F if act == "swiglu" else F
        self.z = torch.empty((max(self.rows_max, 1), N1), dtype=dtype, device=dev) if self.train else None
        self._bwd = None
        self.lse = torch.empty(max(T, 1), **f32) if self.z_beta is not None else None
        self.z_loss = torch.empty(1, **f32) if self.z_beta is not None else None
        self.ws_route = _empty_ws(workspace_bytes("route", T, d, E, k, F), dev)
        self.ws_dispatch = _empty_ws(workspace_bytes("dispatch", T, d, E, k, F), dev)

    def capture(self, x, w_router, b_router, w1, w2, dy=None, **backward_kw) -> "torch.cuda.CUDAGraph":
        """Record run() -- and, given ``dy`` (``train=True``), backward() after
        it -- on these exact tensors into a CUDA graph (one launch per replay).
        The inputs' addresses are baked in: refill the same tensors and call
        ``graph.replay()``.  One eager pass happens first so every one-time
        setup (kernel attributes, driver entry points, backward buffers) is
        done before capture."""
        def step():
            self.run(x, w_router, b_router, w1, w2)
            if dy is not None:
                self.backward(x, w_router, w1, w2, dy, **backward_kw)

        step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        return graph

    def run(self, x, w_router, b_router, w1, w2, stream=None) -> torch.Tensor:
        route(x, w_router, b_router, self.k, self.renorm, topk_idx=self.topk_idx, topk_gate=self.topk_gate,
              prob_sum=self.prob_sum, ws=self.ws_route, stream=stream, n_group=self.n_group,
              topk_group=self.topk_group, lse=self.lse, logits=self.logits)
        dispatch(self.topk_idx, self.topk_gate, x, self.E, self.cap, out=self.disp, ws=self.ws_dispatch,
                 stream=stream)
        D = self.disp
        if self.gather:
            expert_up_gathered(x, D.row_token, D.offsets, D.kept, w1, self.F, self.act, self.rows_max, h=self.h,
                               stream=stream)
            expert_down(self.h, D.offsets, D.kept, w2, D.row_gate, self.rows_max, y_perm=self.y_perm,
                        stream=stream)
        elif self.train:
            expert_up_z(D.x_perm, D.offsets, D.kept, w1, self.F, self.act, self.rows_max, h=self.h, z=self.z,
                        stream=stream)
            expert_down(self.h, D.offsets, D.kept, w2, D.row_gate, self.rows_max, y_perm=self.y_perm,
                        stream=stream)
        else:
            expert_ffn(D.x_perm, D.offsets, D.kept, w1, w2, D.row_gate, self.act, self.rows_max, h=self.h,
                       y_perm=self.y_perm, stream=stream)
        if self.T > 0:
            combine_aux(self.y_perm, D.slot_row, D.kept if self.aux_post_drop else D.counts, self.prob_sum,
                        self.alpha, y=self.y, loss=self.loss, stream=stream)
            if self.z_beta is not None:
                z_loss(self.lse, self.z_beta, loss=self.z_loss, stream=stream)
        return self.y


    def _bwd_buffers(self, dev):
        if self._bwd is None:
            T, d, E, k, F = self.T, self.d, self.E, self.k, self.F
            R = max(self.rows_max, 1)
            N1 = 2 * F if self.act == "swiglu" else F
            bf = dict(dtype=torch.bfloat16, device=dev)
            f32 = dict(dtype=torch.float32, device=dev)
            self._bwd = dict(
                do_perm=torch.empty((R, d), **bf), dgate=torch.empty((max(T, 1), k), **f32),
                dz=torch.empty((R, N1), **bf),
                dx_perm=torch.empty((R, d), **bf),
                dw1=torch.empty((E, N1, d), dtype=self.grad_dtype, device=dev),
                dw2=torch.empty((E, d, F), dtype=self.grad_dtype, device=dev),
                dl=torch.empty((max(T, 1), E), **f32), dx=torch.empty((max(T, 1), d), **bf),
                dW=torch.empty((E, d), **f32), db=torch.empty(E, **f32),
                ws=_empty_ws(workspace_bytes("router_grads", max(T, 1), d, E, k, F), dev))
        return self._bwd

    def backward(self, x, w_router, w1, w2, dy, *, aux_weight: float = 1.0, z_weight: float = 1.0, stream=None,
                 mark=None) -> dict:
        """Gradients of <dy, y> + aux_weight * loss + z_weight * z_loss after
        :meth:`run` on the same inputs (``train=True``).  Returns dx, dW, db,
        dw1, dw2 (weight gradients fp32) and the intermediates; all buffers
        belong to the plan.  ``mark(name)``, when given, is called after each
        phase (for timing)."""
        if not self.train:
            raise ValueError("construct the plan with train=True")
        mark = mark or (lambda name: None)
        B = self._bwd_buffers(x.device)
        D = self.disp
        R, F, E, d = self.rows_max, self.F, self.E, self.d
        combine_bwd(dy, D.slot_row, D.row_gate, self.y_perm, do_perm=B["do_perm"], dgate=B["dgate"], stream=stream)
        mark("combine_bwd")
        # data gradients on the weights as stored: dz = act'(z) * (do . w2[e]) in
        # one GEMM (z kept by the forward), dx_perm = dz . w1[e]
        if self.act == "identity":
            expert_dgrad(B["do_perm"], D.offsets, D.kept, w2, R, out=B["dz"], stream=stream)
        else:
            expert_dgrad_act(B["do_perm"], D.offsets, D.kept, w2, self.z, self.act, R, dz=B["dz"], stream=stream)
        expert_dgrad(B["dz"], D.offsets, D.kept, w1, R, out=B["dx_perm"], stream=stream)
        mark("data_grad_gemms")
        # weight gradients straight from the row-major activations
        expert_wgrad_rows(B["do_perm"], self.h, D.offsets, D.kept, R, dw=B["dw2"], stream=stream)
        mark("wgrad_dw2")
        expert_wgrad_rows(B["dz"], D.x_perm, D.offsets, D.kept, R, dw=B["dw1"], stream=stream)
        mark("wgrad_dw1")
        # router
        counts = D.kept if self.aux_post_drop else D.counts
        zc = z_weight * (self.z_beta or 0.0)
        route_bwd(self.logits, self.topk_idx, B["dgate"], counts, self.renorm, aux_weight * self.alpha * E, zc,
                  dl=B["dl"], stream=stream)
        router_grads(B["dx_perm"], D.slot_row, B["dl"], w_router, x, dx=B["dx"], dW=B["dW"], db=B["db"],
                     ws=B["ws"], stream=stream)
        mark("router_and_dx")
        return dict(dx=B["dx"], dW=B["dW"], db=B["db"], dw1=B["dw1"], dw2=B["dw2"], dgate=B["dgate"], dl=B["dl"],
                    do_perm=B["do_perm"], z=self.z, dz=B["dz"], dx_perm=B["dx_perm"])


def moe_forward(x, w_router, b_router, w1, w2, *, k: int, cf: float, act: str, renorm: bool = True,
                alpha: float = 0.01, gather: bool = False):
    """One MoE-layer forward; returns (y, loss, plan) with every intermediate on ``plan``."""
    T, d = x.shape
    E, N1, _ = w1.shape
    F = w2.shape[2]
    plan = MoEPlan(T, d, E, k, F, act, x.dtype, capacity(T, E, cf), x.device, alpha, renorm, gather)
    y = plan.run(x, w_router, b_router, w1, w2)
    return y, plan.loss, plan
