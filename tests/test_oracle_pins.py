"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test reaches the oracle's answer by a different road (brute force,
closed form, a library routine, an invariant), so that a plausible slip in the
oracle -- a dropped bias, a wrong sign, a swapped gate/up half, token-major
instead of rank-major slot order, counts after instead of before drops --
fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as Fn

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def one_hot_router(Lmat: np.ndarray, b=None):
    """x = I_T and W[e, t] = Lmat[t, e]: the router's logits are Lmat + b."""
    T, E = Lmat.shape
    x = torch.eye(T, dtype=torch.float32)
    W = torch.from_numpy(np.ascontiguousarray(Lmat.T, dtype=np.float32))
    bb = None if b is None else torch.from_numpy(np.asarray(b, dtype=np.float32))
    return x, W, bb


# ----------------------------------------------------------------- top-k ---

@pytest.mark.parametrize("E,k", [(2, 1), (3, 2), (4, 2), (5, 3), (6, 4), (8, 2), (8, 4), (7, 7)])
def test_topk_brute_force_with_exact_ties(E, k):
    """Enumerate every ordered k-tuple of distinct experts; the right one is
    the lexicographic maximum of ((logit, -index), ...).  Small integer
    logits make exact ties common; the bias is added by the router."""
    rng = np.random.default_rng(100 * E + k)
    T = 40
    Lm = rng.integers(-2, 3, size=(T, E)).astype(np.float64)
    b = rng.integers(-1, 2, size=E).astype(np.float64)
    x, W, bb = one_hot_router(Lm, b)
    L = oracle.router_logits(x, W, bb)
    assert np.array_equal(L, Lm + b)                   # bias is part of the linear layer
    idx, gate, ps = oracle.route(L, k, renorm=False)
    for t in range(T):
        lt = Lm[t] + b
        best = max(itertools.permutations(range(E), k),
                   key=lambda tup: tuple((lt[e], -e) for e in tup))
        assert tuple(idx[t]) == best, (t, lt, idx[t], best)
        p = scipy.special.softmax(lt)
        np.testing.assert_allclose(gate[t], p[list(best)], rtol=1e-13, atol=0)


def test_topk_tie_goes_to_lower_index():
    Lm = np.zeros((3, 6))
    Lm[0] = [1, 5, 5, 0, 5, 2]      # three-way tie at the top
    Lm[1] = [3, 3, 3, 3, 3, 3]      # all equal
    Lm[2] = [0, 0, 9, 0, 0, 9]
    x, W, _ = one_hot_router(Lm)
    idx, _, _ = oracle.route(oracle.router_logits(x, W), 3, renorm=True)
    assert idx.tolist() == [[1, 2, 4], [0, 1, 2], [2, 5, 0]]


def test_zero_router_picks_first_k_with_uniform_gates():
    T, d, E, k = 50, 16, 8, 3
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(1))
    W = torch.zeros(E, d)
    L = oracle.router_logits(x, W, torch.zeros(E))
    for renorm, g in ((False, 1.0 / E), (True, 1.0 / k)):
        idx, gate, ps = oracle.route(L, k, renorm=renorm)
        assert (idx == np.arange(k)).all()
        np.testing.assert_allclose(gate, g, rtol=1e-15)
        np.testing.assert_allclose(ps, T / E, rtol=1e-13)


def test_softmax_against_library_and_two_expert_sigmoid():
    rng = np.random.default_rng(7)
    T, E = 30, 5
    Lm = rng.normal(0, 3, size=(T, E))
    x, W, _ = one_hot_router(Lm)
    L = oracle.router_logits(x, W)
    idx, gate, ps, prob = oracle.route(L, 2, renorm=True, want_prob=True)
    np.testing.assert_allclose(prob, scipy.special.softmax(L, axis=1), rtol=1e-13, atol=1e-300)
    np.testing.assert_allclose(ps, scipy.special.softmax(L, axis=1).sum(0), rtol=1e-12)
    # renormalised pair of gates = logistic function of the logit gap
    gap = L[np.arange(T), idx[:, 0]] - L[np.arange(T), idx[:, 1]]
    np.testing.assert_allclose(gate[:, 0], scipy.special.expit(gap), rtol=1e-12)
    np.testing.assert_allclose(gate[:, 1], scipy.special.expit(-gap), rtol=1e-12)
    assert (gap > 0).all()


def test_prob_sum_is_T_and_gate_sums():
    rng = np.random.default_rng(8)
    T, d, E, k = 200, 32, 16, 4
    x = torch.from_numpy(rng.normal(size=(T, d)).astype(np.float32))
    W = torch.from_numpy(rng.normal(0, 0.3, size=(E, d)).astype(np.float32))
    L = oracle.router_logits(x, W)
    _, g_r, ps = oracle.route(L, k, renorm=True)
    _, g_n, _ = oracle.route(L, k, renorm=False)
    assert abs(ps.sum() - T) < 1e-10
    np.testing.assert_allclose(g_r.sum(1), 1.0, rtol=1e-14)
    assert (g_n.sum(1) <= 1.0 + 1e-15).all() and (g_n.sum(1) > 0).all()
    assert (np.diff(g_n, axis=1) <= 0).all()          # k-rank follows probability


# -------------------------------------------------------------- capacity ---

def _capacity_rows():
    rows = []
    with open(os.path.join(GOLDEN, "capacity.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                T, E, cf, cap = line.split()
                rows.append((int(T), int(E), float(cf), int(cap)))
    return rows


@pytest.mark.parametrize("T,E,cf,cap", _capacity_rows())
def test_capacity_table(T, E, cf, cap):
    assert oracle.capacity(T, E, cf) == cap


# -------------------------------------------------------------- dispatch ---

def _brute_positions(idx, cap):
    """pos of (t,j) = number of earlier assignments to the same expert in
    k-rank-then-token order; O(n^2) counting, no queue."""
    T, k = idx.shape
    pos = np.empty((T, k), dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            before = 0
            for j2 in range(k):
                for t2 in range(T):
                    if (j2, t2) < (j, t) and idx[t2, j2] == e:
                        before += 1
            pos[t, j] = before if before < cap else -1
    return pos


@pytest.mark.parametrize("T,E,k,cap", [(30, 4, 2, 9), (25, 5, 3, 4), (17, 3, 1, 5), (20, 4, 2, 0),
                                       (12, 6, 6, 2), (16, 8, 2, 40)])
def test_slot_order_brute_force(T, E, k, cap):
    rng = np.random.default_rng(T * 31 + E)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, kept, pos, nd = oracle.dispatch(idx, E, cap)
    assert np.array_equal(pos, _brute_positions(idx, cap))
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert np.array_equal(kept, np.minimum(counts, cap))
    assert nd == int(np.maximum(counts - cap, 0).sum())
    assert kept.sum() + nd == T * k
    assert nd == int((pos < 0).sum())


def test_zero_router_slot_order_first_choices_in_token_order():
    """All tokens tie, so every first choice is expert 0 and every second
    choice expert 1: expert 0 keeps exactly tokens 0..cap-1 (rank 0)."""
    T, d, E, k, cap = 40, 8, 4, 2, 13
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(3))
    idx, _, _ = oracle.route(oracle.router_logits(x, torch.zeros(E, d)), k)
    counts, kept, pos, nd = oracle.dispatch(idx, E, cap)
    assert counts.tolist() == [T, T, 0, 0] and kept.tolist() == [cap, cap, 0, 0]
    assert pos[:cap, 0].tolist() == list(range(cap)) and (pos[cap:, 0] == -1).all()
    assert pos[:cap, 1].tolist() == list(range(cap)) and (pos[cap:, 1] == -1).all()
    assert nd == 2 * (T - cap)


def test_rank_beats_token_order():
    """A later token's first choice outranks an earlier token's second choice."""
    idx = np.array([[1, 0], [0, 1]], dtype=np.int32)   # t0: 1 then 0; t1: 0 then 1
    _, _, pos, _ = oracle.dispatch(idx, 2, 1)
    assert pos.tolist() == [[0, -1], [0, -1]]


# ------------------------------------------------------------ expert FFN ---

def _rand(shape, std, seed):
    return torch.randn(shape, generator=torch.Generator().manual_seed(seed), dtype=torch.float64) * std


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_dense_ffn_special_case_matches_torch(act):
    """E = 1, k = 1, dropless, renorm: the layer is one dense FFN."""
    T, d, F = 24, 16, 40
    N1 = 2 * F if act == "swiglu" else F
    x = _rand((T, d), 1.0, 1).float()
    w1 = _rand((1, N1, d), d ** -0.5, 2).float()
    w2 = _rand((1, d, F), F ** -0.5, 3).float()
    out = oracle.forward(x, torch.zeros(1, d), None, w1, w2, k=1, cap=T, act=act)
    X, A, B = x.double(), w1[0].double(), w2[0].double()
    if act == "gelu":
        h = Fn.gelu(X @ A.T)
    else:
        h = Fn.silu(X @ A[:F].T) * (X @ A[F:].T)
    ref = (h @ B.T).numpy()
    np.testing.assert_allclose(out["y"], ref, rtol=1e-12, atol=1e-13)
    assert out["n_dropped"] == 0 and np.allclose(out["gate"], 1.0)


def test_dense_mixture_k_equals_E():
    """k = E, dropless, no renorm: y = sum_e p_e FFN_e(x), with p the softmax."""
    T, d, E, F = 20, 12, 4, 24
    x = _rand((T, d), 1.0, 4).float()
    W = _rand((E, d), 0.5, 5).float()
    b = _rand((E,), 0.5, 6).float()
    w1 = _rand((E, 2 * F, d), d ** -0.5, 7).float()
    w2 = _rand((E, d, F), F ** -0.5, 8).float()
    out = oracle.forward(x, W, b, w1, w2, k=E, cap=T, act="swiglu", renorm=False)
    X = x.double()
    p = torch.softmax(X @ W.double().T + b.double(), dim=1)
    g = torch.einsum("tc,enc->ten", X, w1.double())
    h = Fn.silu(g[..., :F]) * g[..., F:]
    fe = torch.einsum("ten,edn->ted", h, w2.double())
    ref = torch.einsum("te,ted->td", p, fe).numpy()
    np.testing.assert_allclose(out["y"], ref, rtol=1e-11, atol=1e-13)


def test_single_row_ffn_exposes_activation():
    d, F = 8, 16
    v = _rand((d,), 1.0, 9).float()
    w1 = _rand((3, F, d), 0.4, 10).float()
    w2 = _rand((3, d, F), 0.3, 11).float()
    a, out = oracle.expert_ffn_row(v, w1, w2, 2, "gelu")
    z = w1[2].double() @ v.double()
    np.testing.assert_allclose(a, Fn.gelu(z).numpy(), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(out, (w2[2].double() @ Fn.gelu(z)).numpy(), rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------- combine ---

def test_identity_experts_return_x():
    """Every expert is the identity map (w1 = w2 = I, no activation),
    gates renormalised, nothing dropped: the layer output is x itself."""
    T, d, E, k = 48, 16, 6, 3
    x = _rand((T, d), 1.0, 12).float()
    W = _rand((E, d), 0.5, 13).float()
    eye = torch.eye(d).expand(E, d, d).contiguous()
    out = oracle.forward(x, W, None, eye, eye, k=k, cap=T, act="identity")
    np.testing.assert_allclose(out["y"], x.double().numpy(), rtol=1e-13, atol=1e-14)


def test_identity_experts_with_drops_scale_by_kept_gates():
    """With drops the identity layer returns (sum of kept gates) * x; a token
    whose slots were all dropped gets a zero row (it takes the residual path)."""
    T, d, E, k, cap = 64, 8, 4, 2, 9
    x = _rand((T, d), 1.0, 14).float()
    W = _rand((E, d), 1.0, 15).float()
    eye = torch.eye(d).expand(E, d, d).contiguous()
    out = oracle.forward(x, W, None, eye, eye, k=k, cap=cap, act="identity")
    kept_gate = np.where(out["pos"] >= 0, out["gate"], 0.0).sum(1)
    np.testing.assert_allclose(out["y"], kept_gate[:, None] * x.double().numpy(), rtol=1e-13, atol=1e-14)
    assert out["n_dropped"] > 0 and (kept_gate == 0).any()


# -------------------------------------------------------------- aux loss ---

@pytest.mark.parametrize("cap", [None, 0, 3])
def test_aux_loss_uniform_router_is_alpha_k(cap):
    """W = 0, b = 0: P_i = 1/E, so L = alpha * E * sum_i f_i / E = alpha * k
    whatever f is; with cap = 0 every slot drops and L is unchanged, which
    pins f_i to the counts before drops."""
    T, d, E, k, alpha = 40, 8, 8, 2, 0.01
    x = _rand((T, d), 1.0, 16).float()
    L = oracle.router_logits(x, torch.zeros(E, d), torch.zeros(E))
    idx, _, ps = oracle.route(L, k)
    counts, _, _, nd = oracle.dispatch(idx, E, T if cap is None else cap)
    assert abs(oracle.aux_loss(counts, ps, T, alpha) - alpha * k) < 1e-15
    if cap == 0:
        assert nd == T * k


@pytest.mark.parametrize("E,k", [(4, 1), (8, 2), (16, 4), (5, 5)])
def test_aux_loss_circulant_router_is_alpha_k(E, k):
    """T = d = E, x = I, W[e, c] = v[(e - c) mod E] with distinct v: every
    expert appears once at every k-rank (f_i = k/E) and every expert's mean
    probability is 1/E, so L = alpha * k."""
    rng = np.random.default_rng(E)
    v = rng.permutation(E) * 0.7 + rng.uniform(0, 0.1, E)
    W = np.array([[v[(e - c) % E] for c in range(E)] for e in range(E)], dtype=np.float32)
    x = torch.eye(E)
    L = oracle.router_logits(x, torch.from_numpy(W))
    idx, _, ps = oracle.route(L, k)
    counts, _, _, _ = oracle.dispatch(idx, E, E)
    assert (counts == k).all()
    np.testing.assert_allclose(ps, 1.0, rtol=1e-12)
    alpha = 0.01
    assert abs(oracle.aux_loss(counts, ps, E, alpha) - alpha * k) < 1e-14


def test_aux_loss_one_hot_concentration():
    """All mass on expert 0 for every token (k = 1): f_0 = 1, P_0 -> 1, so
    L -> alpha * E, the maximum."""
    T, E = 10, 8
    Lm = np.full((T, E), -60.0)
    Lm[:, 0] = 60.0
    x, W, _ = one_hot_router(Lm)
    idx, _, ps = oracle.route(oracle.router_logits(x, W), 1)
    counts, _, _, _ = oracle.dispatch(idx, E, T)
    assert math.isclose(oracle.aux_loss(counts, ps, T, 0.5), 0.5 * E, rel_tol=1e-12)


# ------------------------------------------------ group-limited routing ---

@pytest.mark.parametrize("E,G,M,k", [(4, 2, 1, 2), (6, 3, 1, 2), (6, 3, 2, 3), (8, 4, 2, 2), (8, 2, 1, 4),
                                     (8, 4, 3, 5)])
def test_grouped_topk_brute_force_with_exact_ties(E, G, M, k):
    """Enumerate every M-subset of groups and every ordered k-tuple of the
    kept experts.  The kept subset is the one whose groups, listed best
    first by (score desc, index asc), compare lexicographically best; the
    chosen tuple is the lexicographic maximum of ((logit, -index), ...)
    over the kept experts.  Integer logits make ties between group scores
    and between experts common."""
    rng = np.random.default_rng(1000 * E + 10 * G + M)
    T = 30
    L = rng.integers(-2, 3, size=(T, E)).astype(np.float64)
    idx, gate, ps = oracle.route_grouped(L, k, G, M, renorm=False)
    gsz = E // G
    for t in range(T):
        lt = L[t]
        score = [max(lt[g * gsz:(g + 1) * gsz]) for g in range(G)]
        best_set = max(itertools.combinations(range(G), M),
                       key=lambda S: sorted(((score[g], -g) for g in S), reverse=True))
        allowed = [e for e in range(E) if e // gsz in best_set]
        best = max(itertools.permutations(allowed, k), key=lambda tup: tuple((lt[e], -e) for e in tup))
        assert tuple(idx[t]) == best, (t, lt, idx[t], best)
        np.testing.assert_allclose(gate[t], scipy.special.softmax(lt)[list(best)], rtol=1e-13, atol=0)
    np.testing.assert_allclose(ps, scipy.special.softmax(L, axis=1).sum(0), rtol=1e-12)


def test_grouped_routing_worked_example():
    """Hand-worked: 8 experts in 4 groups of 2.  Row 0 has its best expert (2)
    in group 1, whose other expert (3) is weak: one kept group gives (2, 3),
    two kept groups (1 and 0) give (2, 0), as plain top-2 does.  Row 1 has
    three groups tied at score 3: the lowest (0) wins, giving (1, 0); with
    two groups (0 and 1) the tie 1 vs 2 goes to the lower index."""
    L = np.array([[5, 4.9, 6, 0, 1, 1, 0, 0], [1, 3, 3, 2, 0, 0, 3, 1]], dtype=np.float64)
    assert oracle.route_grouped(L, 2, 4, 1)[0].tolist() == [[2, 3], [1, 0]]
    assert oracle.route_grouped(L, 2, 4, 2)[0].tolist() == [[2, 0], [1, 2]]
    assert oracle.route_grouped(L, 3, 4, 2)[0].tolist() == [[2, 0, 1], [1, 2, 3]]
    assert oracle.route_grouped(L, 2, 2, 1)[0].tolist() == [[2, 0], [1, 2]]   # groups {0..3}, {4..7}


@pytest.mark.parametrize("G,M", [(1, 1), (4, 4), (8, 8)])
def test_grouped_routing_reduces_to_plain_topk(G, M):
    """One group, or every group kept: the restriction is void."""
    rng = np.random.default_rng(7)
    L = rng.standard_normal((200, 16))
    for renorm in (True, False):
        a = oracle.route(L, 3, renorm)
        b = oracle.route_grouped(L, 3, G, M, renorm)
        assert np.array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])
        np.testing.assert_array_equal(a[2], b[2])


def test_grouped_routing_keeps_first_choice_and_stays_in_kept_groups():
    """With one kept group the overall best expert is always chosen first
    (its group has the top score), and every choice lies in its group."""
    rng = np.random.default_rng(8)
    L = rng.standard_normal((300, 32))
    idx, gate, _ = oracle.route_grouped(L, 4, 8, 1)
    assert np.array_equal(idx[:, 0], np.argmax(L, axis=1))
    assert np.all(idx // 4 == (idx[:, :1] // 4))
    np.testing.assert_allclose(gate.sum(1), 1.0, rtol=1e-14)


def test_grouped_routing_rejects_bad_shapes():
    L = np.zeros((2, 8))
    for args in [(2, 3, 1), (2, 4, 0), (2, 4, 5), (5, 4, 2)]:
        with pytest.raises(ValueError):
            oracle.route_grouped(L, *args)


# --------------------------------------------------------- router z-loss ---

def test_logsumexp_against_library_and_closed_forms():
    rng = np.random.default_rng(9)
    L = rng.standard_normal((50, 24)) * 3
    np.testing.assert_allclose(oracle.logsumexp(L), scipy.special.logsumexp(L, axis=1), rtol=1e-14)
    np.testing.assert_allclose(oracle.logsumexp(np.zeros((3, 8))), math.log(8), rtol=1e-15)
    # shift invariance, and no overflow for large logits
    np.testing.assert_allclose(oracle.logsumexp(L + 1000.0), oracle.logsumexp(L) + 1000.0, rtol=1e-14)
    # two experts: lse(0, ln 3) = ln 4
    np.testing.assert_allclose(oracle.logsumexp(np.array([[0.0, math.log(3.0)]])), math.log(4.0), rtol=1e-15)


def test_z_loss_closed_forms():
    """Zero router: every lse is ln E, so L_z = beta (ln E)^2.  In general
    L_z = beta * mean(lse^2), checked on lse values given directly."""
    E, T = 16, 64
    x = torch.randn(T, 32)
    L = oracle.router_logits(x, torch.zeros(E, 32), torch.zeros(E))
    lse = oracle.logsumexp(L)
    assert oracle.z_loss(lse, 1e-3) == pytest.approx(1e-3 * math.log(E) ** 2, rel=1e-14)
    v = np.array([1.0, -2.0, 3.0, 0.5])
    assert oracle.z_loss(v, 0.5) == pytest.approx(0.5 * (1 + 4 + 9 + 0.25) / 4, rel=1e-15)
    assert oracle.z_loss(v, 0.0) == 0.0


# ------------------------------------------------- post-drop f_i variant ---

@pytest.mark.parametrize("cap", [0, 3, 7, 10**6])
def test_post_drop_aux_loss_uniform_router(cap):
    """Zero router (P_i = 1/E): with f_i = kept_i / T the loss is
    alpha * (T k - n_dropped) / T; dropless it equals the pre-drop loss."""
    E, k, T, alpha = 8, 2, 40, 0.01
    rng = np.random.default_rng(cap)
    x = torch.randn(T, 16)
    L = oracle.router_logits(x, torch.zeros(E, 16), None)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)   # any routing
    _, _, ps = oracle.route(L, k)
    counts, kept, pos, nd = oracle.dispatch(idx, E, cap)
    post = oracle.aux_loss(kept, ps, T, alpha)
    assert post == pytest.approx(alpha * (T * k - nd) / T, rel=1e-13)
    if cap >= T:
        assert post == oracle.aux_loss(counts, ps, T, alpha)
