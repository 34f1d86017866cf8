"""C ABI checks that need no GPU: the library builds and loads, exports every
function include/moe_b300.h declares, its host-side functions are right, and
argument errors come back synchronously before any CUDA work is enqueued."""
import ctypes
import os
import re

import pytest

import top_routing_expert_02_b300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_b300.h")
GOLDEN = os.path.join(ROOT, "tests", "golden", "capacity.txt")

FAKE = ctypes.c_void_p(0x1000)   # never dereferenced: every call below fails validation first


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", text)))


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ("moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_aux_loss"):
        assert n in names


def test_library_exports_every_declared_function():
    L = moe.lib()
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing
    assert L.moe_abi_version() == 1


def declared_parameter_counts():
    """{name: number of parameters} of every function declared in the header."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"\b(moe_\w+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_declares_a_signature_for_every_function():
    src = open(os.path.join(ROOT, "top_routing_expert_02_b300", "__init__.py")).read()
    missing = [n for n in declared_functions() if f'"{n}"' not in src]
    assert not missing, missing


def test_binding_signatures_match_the_header_parameter_counts():
    """Each ctypes signature has as many arguments as the header declares."""
    counts = declared_parameter_counts()
    assert set(counts) == set(declared_functions())
    wrong = {n: (c, len(moe._SIGS[n][1])) for n, c in counts.items() if len(moe._SIGS[n][1]) != c}
    assert not wrong, wrong


def _golden_caps():
    rows = []
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            T, E, cf, cap = line.split()
            rows.append((int(T), int(E), float(cf), int(cap)))
    return rows


@pytest.mark.parametrize("T,E,cf,cap", _golden_caps())
def test_capacity_matches_golden_table(T, E, cf, cap):
    assert moe.capacity(T, E, cf) == cap


def test_perm_rows_and_workspace():
    assert moe.perm_rows_max(4096, 2, 8, 640) == 5120
    assert moe.perm_rows_max(512, 8, 128, 512) == 4096
    assert moe.perm_rows_max(0, 2, 8, 10) == 0
    assert moe.perm_rows_max(10, 2, 8, -1) == -1
    assert moe.workspace_bytes("ffn", 4096, 4096, 8, 2, 14336) == 0
    assert moe.workspace_bytes("route", 4096, 4096, 8, 2, 14336) > 0
    # per-chunk expert histograms: chunks of 256 assignments up to T*k = 65536, of 1024 above
    assert moe.workspace_bytes("dispatch", 4096, 4096, 8, 2, 14336) == 32 * 8 * 4
    assert moe.workspace_bytes("dispatch", 16384, 2048, 64, 2, 1408) == 128 * 64 * 4
    assert moe.workspace_bytes("dispatch", 32768, 4096, 128, 8, 1536) == 256 * 128 * 4
    assert moe.workspace_bytes("dispatch", 0, 4096, 8, 2, 14336) == 0
    assert moe.workspace_bytes("route", 0, 4096, 8, 2, 14336) == 0


def test_status_strings():
    L = moe.lib()
    for code in range(6):
        assert L.moe_status_string(code)
    assert L.moe_status_string(5) == b"device wait timed out"


def _route(L, **over):
    a = dict(x=FAKE, xdt=1, w=FAKE, b=None, T=16, d=128, E=8, k=2, renorm=1, idx=FAKE, gate=FAKE, ps=FAKE,
             ws=FAKE, ws_bytes=1 << 20)
    a.update(over)
    return L.moe_route(a["x"], a["xdt"], a["w"], a["b"], a["T"], a["d"], a["E"], a["k"], a["renorm"], a["idx"],
                       a["gate"], a["ps"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("over,code", [
    (dict(E=0), 1), (dict(E=257), 1), (dict(k=0), 1), (dict(k=9, E=8), 1), (dict(k=17, E=64), 1),
    (dict(T=-1), 1), (dict(xdt=7), 1), (dict(x=None), 1), (dict(ps=None), 1),
    (dict(d=100), 2), (dict(ws=None), 3), (dict(ws_bytes=4), 3),
])
def test_route_argument_errors(over, code):
    assert _route(moe.lib(), **over) == code


def test_dispatch_ffn_combine_aux_argument_errors():
    L = moe.lib()
    F_ = FAKE
    # dispatch: negative capacity, null outputs, bad d, small workspace
    args = [F_, F_, 16, 2, 8, 4, F_, 1, 128, F_, F_, F_, F_, F_, F_, F_, F_, F_, 1 << 20, None]
    bad = list(args); bad[5] = -1
    assert L.moe_dispatch(*bad) == 1
    bad = list(args); bad[9] = None
    assert L.moe_dispatch(*bad) == 1
    bad = list(args); bad[8] = 96
    assert L.moe_dispatch(*bad) == 2
    bad = list(args); bad[18] = 8                       # 32 assignments: one chunk histogram of 8 experts (32 bytes)
    assert L.moe_dispatch(*bad) == 3
    # ffn: F not a multiple of 64, bad act, null weights
    assert L.moe_expert_up(F_, F_, F_, 8, 128, 96, 0, 1, F_, 10, F_, None) == 2
    assert L.moe_expert_up(F_, F_, F_, 8, 128, 128, 9, 1, F_, 10, F_, None) == 1
    assert L.moe_expert_down(F_, F_, F_, 8, 128, 128, 1, None, F_, 10, F_, None) == 1
    assert L.moe_expert_ffn(F_, None, F_, 8, 128, 128, 0, 1, F_, F_, F_, 10, F_, F_, None, 0, None) == 1
    # combine / aux
    assert L.moe_combine(F_, F_, 16, 0, 128, 1, F_, None) == 1
    assert L.moe_combine(F_, F_, 16, 2, 120, 1, F_, None) == 2
    assert L.moe_aux_loss(F_, F_, 0, 8, ctypes.c_float(0.01), F_, None) == 1
    assert L.moe_aux_loss(F_, F_, 16, 8, ctypes.c_float(0.01), None, None) == 1


def test_gemm_tile_width_setter_validates():
    L = moe.lib()
    assert L.moe_set_gemm_tile_n(100) == 1
    assert L.moe_set_gemm_tile_n(192) == 0
    assert L.moe_set_gemm_tile_n(0) == 0
    assert L.moe_set_wgrad_order(3) == 1
    assert L.moe_set_wgrad_order(-1) == 1
    assert L.moe_set_wgrad_order(1) == 0
    assert L.moe_set_wgrad_order(0) == 0
    assert L.moe_set_gemm_order(3) == 1
    assert L.moe_set_gemm_order(0) == 0
    assert L.moe_set_gemm_tail_halves(2) == 1
    assert L.moe_set_gemm_tail_halves(1) == 0
    assert L.moe_set_launch_overlap(-1) == 1
    assert L.moe_set_launch_overlap(1) == 0
    assert L.moe_set_router_kernel(3) == 1
    assert L.moe_set_router_kernel(0) == 0
    assert L.moe_set_gemm_tma_store(2) == 1
    assert L.moe_set_gemm_tma_store(1) == 0


def test_binding_rejects_unsupported_dtype():
    import torch
    x = torch.zeros(4, 64, dtype=torch.float16)
    with pytest.raises(TypeError):
        moe.route(x, torch.zeros(8, 64), None, 2)


def test_route_ex_and_z_loss_argument_errors():
    L = moe.lib()

    def rex(E=8, k=2, G=4, M=2, T=16):
        return L.moe_route_ex(FAKE, 1, FAKE, None, T, 128, E, k, 1, G, M, FAKE, FAKE, FAKE, None, None, FAKE,
                              1 << 20, None)

    assert rex(G=3) == 1            # 3 does not divide 8
    assert rex(G=0) == 1
    assert rex(E=64, G=64, M=1, k=1) == 1   # more than 32 groups
    assert rex(M=0) == 1
    assert rex(M=5) == 1            # more groups kept than exist
    assert rex(G=4, M=1, k=3) == 1  # one group of 2 cannot hold 3 choices
    assert L.moe_z_loss(FAKE, 0, ctypes.c_float(1e-3), FAKE, None) == 1
    assert L.moe_z_loss(None, 16, ctypes.c_float(1e-3), FAKE, None) == 1
    assert L.moe_z_loss(FAKE, 16, ctypes.c_float(1e-3), None, None) == 1


def test_backward_argument_errors():
    L = moe.lib()
    f = ctypes.c_float
    assert L.moe_wgrad_cols(5120, 8) == 5632
    assert L.moe_wgrad_cols(-1, 8) == -1
    assert L.moe_transpose_experts(FAKE, 2, 100, 64, 1, FAKE, None) == 2       # R not a multiple of 64
    assert L.moe_transpose_experts(FAKE, 2, 128, 64, 0, FAKE, None) == 2       # fp32 not supported
    assert L.moe_transpose_experts(None, 2, 128, 64, 1, FAKE, None) == 1
    assert L.moe_combine_bwd(FAKE, FAKE, FAKE, FAKE, 16, 2, 96, 1, FAKE, FAKE, None) == 2   # d % 64
    assert L.moe_combine_bwd(FAKE, FAKE, FAKE, FAKE, 16, 0, 128, 1, FAKE, FAKE, None) == 1
    assert L.moe_act_bwd(FAKE, FAKE, FAKE, 8, 96, 1, 1, 10, FAKE, None) == 2       # F % 64
    assert L.moe_act_bwd(FAKE, FAKE, FAKE, 8, 128, 7, 1, 10, FAKE, None) == 1      # bad activation
    assert L.moe_pack_segments_t(FAKE, FAKE, FAKE, 8, 128, 5120, 5000, 1, FAKE, None) == 1   # ld too small
    assert L.moe_expert_wgrad(FAKE, FAKE, FAKE, 8, 100, 128, 5632, 1, FAKE, 0, None) == 2   # M % 64
    assert L.moe_expert_wgrad(FAKE, FAKE, FAKE, 8, 128, 128, 5632, 1, FAKE, 5, None) == 1   # bad output type
    assert L.moe_expert_wgrad_rows(FAKE, FAKE, FAKE, FAKE, 8, 100, 128, 640, 1, FAKE, 0, None) == 2   # M % 64
    assert L.moe_expert_wgrad_rows(FAKE, FAKE, FAKE, FAKE, 8, 128, 96, 640, 1, FAKE, 0, None) == 2    # N % 64
    assert L.moe_expert_wgrad_rows(FAKE, FAKE, None, FAKE, 8, 128, 128, 640, 1, FAKE, 0, None) == 1   # no offsets
    assert L.moe_expert_wgrad_rows(None, FAKE, FAKE, FAKE, 8, 128, 128, 640, 1, FAKE, 0, None) == 1   # rows, no a
    assert L.moe_expert_wgrad_rows(FAKE, FAKE, FAKE, FAKE, 8, 128, 128, -1, 1, FAKE, 0, None) == 1    # rows < 0
    assert L.moe_expert_wgrad_rows(FAKE, FAKE, FAKE, FAKE, 8, 128, 128, 640, 0, FAKE, 0, None) == 2   # fp32 inputs
    assert L.moe_route_bwd(FAKE, FAKE, FAKE, None, 16, 8, 2, 1, f(0.1), f(0.0), FAKE, None) == 1
    # moe_router_grads(dx_perm, slot_row, dl, W, x, T, k, E, d, dtype, dx, dW, db, ws, ws_bytes, stream)
    rg = lambda **o: L.moe_router_grads(o.get("dxp", FAKE), FAKE, FAKE, FAKE, o.get("x", FAKE), o.get("T", 64),
                                        o.get("k", 2), o.get("E", 8), o.get("d", 128), o.get("dt", 1), FAKE,
                                        o.get("dW", FAKE), FAKE, o.get("ws", FAKE), o.get("wsb", 1 << 30), None)
    assert rg(k=0) == 1 and rg(E=0) == 1 and rg(T=-1) == 1 and rg(dW=None) == 1 and rg(x=None) == 1
    assert rg(d=96) == 2                 # d % 64
    assert rg(dt=0) == 2                 # bf16 only
    assert rg(dxp=ctypes.c_void_p(0x1008)) == 2   # 16-byte alignment
    assert rg(wsb=16) == 3               # workspace too small
    assert L.moe_workspace_bytes(4, 4096, 4096, 8, 2, 64, 0, 1) > 4096 * 4096 * 4   # holds the fp32 dl . W
    # moe_combine_aux(y_perm, slot_row, T, k, d, dtype, y, counts, prob_sum, E, alpha, loss, stream)
    assert L.moe_combine_aux(FAKE, FAKE, 0, 2, 128, 1, FAKE, FAKE, FAKE, 8, f(0.01), FAKE, None) == 1   # T >= 1
    assert L.moe_combine_aux(FAKE, FAKE, 16, 2, 128, 1, FAKE, FAKE, FAKE, 8, f(0.01), None, None) == 1
    assert L.moe_combine_aux(FAKE, FAKE, 16, 2, 120, 1, FAKE, FAKE, FAKE, 8, f(0.01), FAKE, None) == 2  # d % 64
    assert L.moe_route_bwd(FAKE, FAKE, FAKE, FAKE, 16, 8, 9, 1, f(0.1), f(0.0), FAKE, None) == 1
    assert L.moe_grad_x(FAKE, FAKE, FAKE, None, 16, 2, 8, 128, 1, FAKE, None) == 1
    assert L.moe_router_wgrad(FAKE, FAKE, 1, 0, 8, 128, FAKE, None, FAKE, 1 << 20, None) == 1
    assert L.moe_router_wgrad(FAKE, FAKE, 1, 64, 8, 128, FAKE, None, FAKE, 8, None) == 3    # workspace


def test_d_must_be_a_multiple_of_64():
    """d = 72 (16-byte rows, but not whole 64-element K blocks of the tensor-core
    GEMMs and the router) is MOE_ERR_UNSUPPORTED on every call that takes d."""
    L = moe.lib()
    d = 72
    assert L.moe_route(FAKE, 1, FAKE, None, 16, d, 8, 2, 1, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == 2
    assert L.moe_dispatch(FAKE, FAKE, 16, 2, 8, 4, FAKE, 1, d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                          1 << 20, None) == 2
    assert L.moe_expert_up(FAKE, FAKE, FAKE, 8, d, 128, 0, 1, FAKE, 10, FAKE, None) == 2
    assert L.moe_expert_down(FAKE, FAKE, FAKE, 8, d, 128, 1, FAKE, FAKE, 10, FAKE, None) == 2
    assert L.moe_combine(FAKE, FAKE, 16, 2, d, 1, FAKE, None) == 2


def test_misaligned_buffers_are_refused_before_any_work():
    """Buffers moved with 16-byte vectors or TMA must be 16-byte aligned; a
    misaligned one is MOE_ERR_UNSUPPORTED, returned before anything runs."""
    L = moe.lib()
    MIS = ctypes.c_void_p(0x1008)
    f = ctypes.c_float
    assert L.moe_route(MIS, 1, FAKE, None, 16, 128, 8, 2, 1, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == 2
    assert L.moe_dispatch(FAKE, FAKE, 16, 2, 8, 4, MIS, 1, 128, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                          1 << 20, None) == 2
    assert L.moe_expert_up(MIS, FAKE, FAKE, 8, 128, 128, 0, 1, FAKE, 10, FAKE, None) == 2
    assert L.moe_expert_down(FAKE, FAKE, FAKE, 8, 128, 128, 1, FAKE, FAKE, 10, MIS, None) == 2
    assert L.moe_combine(MIS, FAKE, 16, 2, 128, 1, FAKE, None) == 2
    assert L.moe_combine_bwd(FAKE, FAKE, FAKE, FAKE, 16, 2, 128, 1, MIS, FAKE, None) == 2
    assert L.moe_expert_dgrad(FAKE, FAKE, FAKE, 8, 128, 128, 1, MIS, 10, FAKE, None) == 2
    assert L.moe_expert_wgrad(FAKE, MIS, FAKE, 8, 128, 128, 5632, 1, FAKE, 0, None) == 2
    assert L.moe_expert_wgrad_rows(FAKE, MIS, FAKE, FAKE, 8, 128, 128, 640, 1, FAKE, 0, None) == 2
    assert L.moe_pack_segments_t(MIS, FAKE, FAKE, 8, 128, 10, 576, 1, FAKE, None) == 2
    assert L.moe_grad_x(MIS, FAKE, FAKE, FAKE, 16, 2, 8, 128, 1, FAKE, None) == 2
