"""moe_dispatch_noalloc: the dispatch step for callers that cannot allocate
device memory where they run the layer (an engine plugin that must not call
cudaMalloc, a process whose memory belongs to its own pool, a loop that cannot
take an allocation's synchronisation).  Its scratch is the library's own
fixed 256 KiB device array instead of a caller workspace.

Checked through the C ABI against moe_dispatch on the same inputs, on two
calls in a row with different shapes (the shared array keeps the previous
call's contents, which must not matter).  Dispatch output is integer and
copy work, so the bar is bit-for-bit equality, as in the other dispatch tests.
"""
import ctypes

import pytest
import torch

import top_routing_expert_02_b300 as moe

pytestmark = pytest.mark.gpu


def _routing(T, E, k, d, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    # k distinct experts per token, with a skew so some experts overflow
    scores = torch.rand(T, E, generator=g, device="cuda") + torch.linspace(1.0, 0.0, E, device="cuda")
    idx = scores.topk(k, dim=1).indices.to(torch.int32).contiguous()
    gate = torch.rand(T, k, generator=g, device="cuda").contiguous()
    x = torch.randn(T, d, generator=g, device="cuda").to(torch.bfloat16).contiguous()
    return idx, gate, x


def _check_against_workspace_path(T, E, k, d, cap, seed):
    idx, gate, x = _routing(T, E, k, d, seed)
    ref = moe.dispatch(idx, gate, x, E, cap)
    got = moe.dispatch_noalloc(idx, gate, x, E, cap)
    moe.check()
    for name in ("counts", "kept", "offsets", "slot_row", "n_dropped"):
        assert torch.equal(getattr(got, name), getattr(ref, name)), name
    A = int(ref.offsets[E].item())
    assert A > 0
    assert torch.equal(got.row_token[:A], ref.row_token[:A])
    assert torch.equal(got.row_gate[:A], ref.row_gate[:A])
    assert torch.equal(got.x_perm[:A], ref.x_perm[:A])
    return int(ref.n_dropped.item())


def test_noalloc_dispatch_matches_workspace_dispatch_twice_in_a_row():
    # The dispatch keeps its per-chunk histograms in the scratch array.
    # first call: 71 chunks of 256 assignments, 64 experts, drops
    d1 = _check_against_workspace_path(T=9000, E=64, k=2, d=256, cap=150, seed=11)
    # second call: other shape and chunk size (79 chunks of 1024); leftover
    # histogram cells of the first call remain in the array
    d2 = _check_against_workspace_path(T=40000, E=8, k=2, d=128, cap=6000, seed=12)
    assert d1 > 0 and d2 > 0


def test_noalloc_dispatch_small_batch():
    # a few chunks of 256 assignments, same results as the workspace call
    assert _check_against_workspace_path(T=1000, E=8, k=2, d=128, cap=200, seed=13) > 0


def test_noalloc_dispatch_rejects_sizes_beyond_its_scratch():
    L = moe.lib()
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: the size check comes first
    # ceil(140000*2/1024) * 256 cells > 65536 -> MOE_ERR_WORKSPACE, nothing enqueued
    rc = L.moe_dispatch_noalloc(fake, fake, 140000, 2, 256, 1000, fake, 1, 128, fake, fake, fake, fake, fake, fake,
                                fake, fake, None)
    assert rc == 3
    moe.check()
