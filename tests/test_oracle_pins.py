"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test names what fixes the expected value: a worked example printed on
the pages (fixtures in tests/golden/), a closed form, a library routine on a
special case (torch CPU fp64 functional ops and autograd), finite differences,
or brute force on tiny inputs.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import moe_oracle as mo

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ep_worked_examples.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _ffn_torch(x, Wg, Wu, Wd):
    """Dense SwiGLU MLP through torch's own linear / silu (library routines, fp64)."""
    x, Wg, Wu, Wd = (torch.as_tensor(np.asarray(a, dtype=np.float64)) for a in (x, Wg, Wu, Wd))
    return F.linear(F.silu(F.linear(x, Wg)) * F.linear(x, Wu), Wd).numpy()


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ---------------------------------------------------------------- worked examples


def test_top1_round_trip_worked_example():
    """EP page, 'Top-1 round trip': A1->E0, A2->E2, B1->E1, B2->E2, combine weight 1."""
    g = _golden()["top1_round_trip"]
    T, E, d, n = len(g["tokens"]), g["num_experts"], 8, 5
    choice = np.array(g["choice"])
    # X carries a one-hot routing code in its first E columns; W_r reads exactly those.
    X = np.concatenate([np.eye(E)[choice] * 3.0, _rand((T, d - E), 1)], axis=1)
    W_r = np.zeros((d, E))
    W_r[:E, :E] = np.eye(E)
    Wg, Wu, Wd = _rand((E, n, d), 2, 0.4), _rand((E, n, d), 3, 0.4), _rand((E, d, n), 4, 0.4)
    O, cache = mo.moe_forward(X, W_r, None, Wg, Wu, Wd, K=1)
    r = cache["routing"]
    assert r.counts.tolist() == g["expected_counts"]
    assert r.offsets.tolist() == g["expected_offsets"]
    assert [g["tokens"][t] for t in r.sorted_tok] == g["expected_expert_order"]
    w = cache["w_full"][np.arange(T), choice]
    assert np.all(w == g["combine_weight"])
    # every token gets its own expert's output back in its original slot
    for t in range(T):
        ref = _ffn_torch(X[t:t + 1], Wg[choice[t]], Wu[choice[t]], Wd[choice[t]])[0]
        np.testing.assert_allclose(O[t], ref, rtol=1e-12, atol=1e-14)


def test_top2_weighted_sum_worked_example():
    """EP page, 'Top-2': y(A2) = 0.7 u0 + 0.3 u2 (weights kept apart from selection)."""
    g = _golden()["top2_weights"]
    e0, e2 = g["experts"]
    E, d, n = 4, 6, 3
    # logits with l0 - l2 = ln(7/3), the other experts far below: softmax over the top-2 = (0.7, 0.3)
    logits = np.array([[math.log(7.0 / 3.0), -40.0, 0.0, -41.0]])
    X = _rand((1, d), 5)
    W_r = np.linalg.lstsq(X, logits, rcond=None)[0]  # X @ W_r reproduces the logits
    Wg, Wu, Wd = _rand((E, n, d), 6), _rand((E, n, d), 7), _rand((E, d, n), 8)
    O, cache = mo.moe_forward(X, W_r, None, Wg, Wu, Wd, K=2)
    assert cache["routing"].topk_ids[0].tolist() == [e0, e2]
    w = cache["w_full"][0, [e0, e2]]
    np.testing.assert_allclose(w, g["weights"], rtol=1e-12)
    u0 = _ffn_torch(X, Wg[e0], Wu[e0], Wd[e0])[0]
    u2 = _ffn_torch(X, Wg[e2], Wu[e2], Wd[e2])[0]
    np.testing.assert_allclose(O[0], 0.7 * u0 + 0.3 * u2, rtol=1e-11, atol=1e-13)


def test_imbalance_worked_example():
    """EP page, 'load imbalance': E0<-A1, E1<-B1, E2<- the other six -> GPU0 2 tokens, GPU1 6."""
    g = _golden()["imbalance"]
    choice = np.array(g["choice"])[:, None]
    counts, offsets, perm, sorted_tok = mo.group_by_expert(choice, g["num_experts"])
    assert counts.tolist() == g["expected_counts"]
    per_gpu = [int(counts[np.array(g["gpu_of_expert"]) == k].sum()) for k in (0, 1)]
    assert per_gpu == g["expected_tokens_per_gpu"]
    assert offsets.tolist() == [0, 1, 2, 8, 8]


# ---------------------------------------------------------------- invariants of the discrete stage


@pytest.mark.parametrize("T,E,K", [(97, 8, 2), (256, 16, 4), (300, 64, 8)])
def test_grouping_invariants(T, E, K):
    L = _rand((T, E), T + E)
    r = mo.route_discrete(L, K)
    assert r.counts.sum() == T * K
    assert r.offsets[0] == 0 and r.offsets[-1] == T * K and np.all(np.diff(r.offsets) == r.counts)
    counts, offsets, perm, sorted_tok = mo.group_by_expert(r.topk_ids, E)
    # perm is a bijection of the T*K pairs
    assert np.array_equal(np.sort(perm), np.arange(T * K))
    inv = np.empty_like(perm)
    inv[perm] = np.arange(T * K)
    assert np.array_equal(perm[inv], np.arange(T * K))
    # expert slices are contiguous and stable (ascending token inside an expert)
    flat = r.topk_ids.reshape(-1)
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)
    # top-K really holds the K largest values, largest first
    srt = -np.sort(-L, axis=1)
    np.testing.assert_array_equal(np.take_along_axis(L, r.topk_ids, 1), srt[:, :K])
    # renormalised weights sum to one over the top-K set
    w = mo.combine_weights(L, r.topk_ids)
    np.testing.assert_allclose(np.take_along_axis(w, r.topk_ids, 1).sum(1), 1.0, rtol=1e-14)
    # the per-token return map lists every pair once, in ascending expert
    for t in range(0, T, 7):
        js = r.tok_pairs[r.tok_ptr[t]:r.tok_ptr[t + 1]]
        assert np.all(r.sorted_tok[js] == t)
        assert np.all(np.diff(r.sorted_exp[js]) > 0)


def test_topk_tie_rule_lower_expert_first():
    """Reading: equal logits are ordered by expert index."""
    L = np.array([[1.0, 3.0, 3.0, 0.0, 3.0], [2.0, 2.0, 2.0, 2.0, 2.0]], dtype=np.float32)
    ids = mo.topk_experts(L, 3)
    assert ids.tolist() == [[1, 2, 4], [0, 1, 2]]


def test_k1_weight_is_exactly_one():
    L = _rand((50, 7), 11)
    r = mo.route_discrete(L, 1)
    w = mo.combine_weights(L, r.topk_ids)
    assert np.all(w[np.arange(50), r.topk_ids[:, 0]] == 1.0)


# ---------------------------------------------------------------- special cases = library routines


def test_identity_expert_combine():
    """With every expert the identity, the combine returns X * sum(w) = X."""
    T, d, E, K = 40, 6, 5, 3
    X = _rand((T, d), 12)
    L = _rand((T, E), 13)
    r = mo.route_discrete(L, K)
    w = mo.combine_weights(L, r.topk_ids)
    O = mo.combine(X[r.sorted_tok], r, w, T)
    np.testing.assert_allclose(O, X, rtol=1e-13, atol=1e-14)


def test_single_expert_is_dense_swiglu_mlp():
    """E=1, K=1: the layer is a dense SwiGLU MLP (torch functional ops), weight exactly 1."""
    T, d, n = 33, 10, 7
    X = _rand((T, d), 14)
    W_r = _rand((d, 1), 15)
    Wg, Wu, Wd = _rand((1, n, d), 16, 0.3), _rand((1, n, d), 17, 0.3), _rand((1, d, n), 18, 0.3)
    O, _ = mo.moe_forward(X, W_r, None, Wg, Wu, Wd, K=1)
    np.testing.assert_allclose(O, _ffn_torch(X, Wg[0], Wu[0], Wd[0]), rtol=1e-12, atol=1e-13)


def test_all_experts_is_dense_softmax_mixture():
    """K=E: the layer is sum_e softmax(l)_e * FFN_e(x) (torch softmax / functional ops)."""
    T, d, n, E = 21, 9, 4, 5
    X = _rand((T, d), 19)
    W_r, b = _rand((d, E), 20), _rand((E,), 21)
    Wg, Wu, Wd = _rand((E, n, d), 22, 0.3), _rand((E, n, d), 23, 0.3), _rand((E, d, n), 24, 0.3)
    O, _ = mo.moe_forward(X, W_r, b, Wg, Wu, Wd, K=E)
    s = torch.softmax(torch.as_tensor(X @ W_r + b), dim=1).numpy()
    ref = sum(s[:, e:e + 1] * _ffn_torch(X, Wg[e], Wu[e], Wd[e]) for e in range(E))
    np.testing.assert_allclose(O, ref, rtol=1e-11, atol=1e-13)


# ---------------------------------------------------------------- backward vs autograd / finite differences


def _dense_loss_torch(X, W_r, b, Wg, Wu, Wd, dO, member, topk):
    """Dense formulation with fixed pair sets: O_t = sum_e [e in F(t)] w_te FFN_e(x_t),
    w_te = exp(l_te) / sum_{j in TopK(t)} exp(l_tj).  Differentiated by torch autograd."""
    Xt = torch.tensor(X, dtype=torch.float64, requires_grad=True)
    Wrt = torch.tensor(W_r, dtype=torch.float64, requires_grad=True)
    Wgt = torch.tensor(Wg, dtype=torch.float64, requires_grad=True)
    Wut = torch.tensor(Wu, dtype=torch.float64, requires_grad=True)
    Wdt = torch.tensor(Wd, dtype=torch.float64, requires_grad=True)
    logits = Xt @ Wrt + torch.as_tensor(b)
    logits.retain_grad()
    topk_mask = torch.zeros_like(logits, dtype=torch.bool)
    topk_mask[torch.arange(X.shape[0])[:, None], torch.as_tensor(topk)] = True
    m = logits.masked_fill(~topk_mask, -torch.inf).max(dim=1, keepdim=True).values
    z = torch.exp(logits - m)
    w = z / (z * topk_mask).sum(dim=1, keepdim=True)
    O = torch.zeros_like(Xt)
    for e in range(Wg.shape[0]):
        y = F.linear(F.silu(F.linear(Xt, Wgt[e])) * F.linear(Xt, Wut[e]), Wdt[e])
        O = O + (w[:, e] * torch.as_tensor(member[:, e], dtype=torch.float64))[:, None] * y
    loss = (O * torch.as_tensor(dO)).sum()
    loss.backward()
    return dict(dX=Xt.grad.numpy(), dW_r=Wrt.grad.numpy(), dWg=Wgt.grad.numpy(), dWu=Wut.grad.numpy(),
                dWd=Wdt.grad.numpy(), dlogits=logits.grad.numpy(), O=O.detach().numpy())


@pytest.mark.parametrize("m_tile", [0, 2])
def test_backward_matches_autograd(m_tile):
    T, d, E, n, K = 12, 8, 4, 5, 2
    X, W_r, b = _rand((T, d), 30), _rand((d, E), 31, 0.5), _rand((E,), 32, 0.5)
    Wg, Wu, Wd = _rand((E, n, d), 33, 0.4), _rand((E, n, d), 34, 0.4), _rand((E, d, n), 35, 0.4)
    dO = _rand((T, d), 36)
    O, cache = mo.moe_forward(X, W_r, b, Wg, Wu, Wd, K, m_tile=m_tile)
    r = cache["routing"]
    if m_tile:
        assert not np.array_equal(r.member.sum(1), np.full(T, K)), "rounding should change some tokens"
    g = mo.moe_backward(X, W_r, b, Wg, Wu, Wd, dO, cache)
    ref = _dense_loss_torch(X, W_r, b, Wg, Wu, Wd, dO, r.member, r.topk_ids)
    np.testing.assert_allclose(O, ref["O"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dX"], ref["dX"], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dW_r"], ref["dW_r"], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dlogits"], ref["dlogits"], rtol=1e-10, atol=1e-12)
    for e in range(E):
        np.testing.assert_allclose(g["dW_gate"][e], ref["dWg"][e], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(g["dW_up"][e], ref["dWu"][e], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(g["dW_down"][e], ref["dWd"][e], rtol=1e-10, atol=1e-12)
    # router-gradient rows sum to zero (the weights over TopK sum to one)
    np.testing.assert_allclose(g["dlogits"].sum(1), 0.0, atol=1e-12)


def test_backward_finite_differences():
    """Central differences in fp64 (h = 1e-6) on tiny inputs, away from routing ties."""
    T, d, E, n, K = 4, 8, 3, 4, 2
    X, W_r = _rand((T, d), 40), _rand((d, E), 41, 0.6)
    Wg, Wu, Wd = _rand((E, n, d), 42, 0.5), _rand((E, n, d), 43, 0.5), _rand((E, d, n), 44, 0.5)
    dO = _rand((T, d), 45)
    O, cache = mo.moe_forward(X, W_r, None, Wg, Wu, Wd, K)
    srt = -np.sort(-cache["logits"], axis=1)
    assert np.min(srt[:, K - 1] - srt[:, K]) > 1e-3, "inputs too close to a routing tie"
    g = mo.moe_backward(X, W_r, None, Wg, Wu, Wd, dO, cache)

    def loss(X_, W_r_, Wg_, Wu_, Wd_):
        O_, c_ = mo.moe_forward(X_, W_r_, None, Wg_, Wu_, Wd_, K)
        assert np.array_equal(c_["routing"].member, cache["routing"].member)
        return float(np.sum(O_ * dO))

    h = 1e-6
    args = [X, W_r, Wg, Wu, Wd]
    grads = [g["dX"], g["dW_r"], np.stack([g["dW_gate"][e] for e in range(E)]),
             np.stack([g["dW_up"][e] for e in range(E)]), np.stack([g["dW_down"][e] for e in range(E)])]
    rng = np.random.default_rng(46)
    for ai, (a, ga) in enumerate(zip(args, grads)):
        for _ in range(6):
            idx = tuple(rng.integers(0, s) for s in a.shape)
            ap, am = a.copy(), a.copy()
            ap[idx] += h
            am[idx] -= h
            pa = [ap if i == ai else args[i] for i in range(5)]
            ma = [am if i == ai else args[i] for i in range(5)]
            fd = (loss(*pa) - loss(*ma)) / (2 * h)
            assert abs(fd - ga[idx]) <= 1e-6 * max(1.0, abs(fd)), (ai, idx, fd, ga[idx])


def test_score_gradient_identity():
    """<dO, y> = <dO W_down, a> since y = a W_down^T: the identity the device's dS uses."""
    T, d, E, n, K = 30, 12, 5, 7, 2
    X, W_r = _rand((T, d), 50), _rand((d, E), 51)
    Wg, Wu, Wd = _rand((E, n, d), 52, 0.3), _rand((E, n, d), 53, 0.3), _rand((E, d, n), 54, 0.3)
    dO = _rand((T, d), 55)
    O, cache = mo.moe_forward(X, W_r, None, Wg, Wu, Wd, K)
    r = cache["routing"]
    for e in range(E):
        rows = r.rows_of(e)
        if len(rows) == 0:
            continue
        blk = mo.expert_block_backward(X[rows], dO[rows], np.ones(len(rows)), Wg[e], Wu[e], Wd[e])
        alt = np.sum((dO[rows] @ Wd[e]) * blk["a"], axis=1)
        np.testing.assert_allclose(blk["dw"], alt, rtol=1e-11, atol=1e-12)


def test_empty_expert_weight_gradient_is_zero():
    T, d, E, n, K = 16, 6, 4, 3, 1
    X = _rand((T, d), 60)
    W_r = np.zeros((d, E))
    W_r[:, 0] = 1.0
    W_r[:, 1] = -1.0  # expert 2 and 3 never win
    Wg, Wu, Wd = _rand((E, n, d), 61), _rand((E, n, d), 62), _rand((E, d, n), 63)
    O, cache = mo.moe_forward(X, W_r, None, Wg, Wu, Wd, K)
    assert cache["routing"].counts[2] == 0 and cache["routing"].counts[3] == 0
    g = mo.moe_backward(X, W_r, None, Wg, Wu, Wd, _rand((T, d), 64), cache)
    for e in (2, 3):
        assert not g["dW_gate"][e].any() and not g["dW_up"][e].any() and not g["dW_down"][e].any()


# ---------------------------------------------------------------- token rounding


def test_rounding_closed_values():
    """r = M * floor((c + M/2) / M): nearest multiple, exact halves round up (reading)."""
    T, E, M = 512, 6, 128
    counts_wanted = [63, 64, 191, 192, 0, 2]
    rows = []
    for e, c in enumerate(counts_wanted):
        rows += [e] * c
    topk = np.array(rows + [5] * (T - len(rows)))[:, None]
    s = _rand((T, E), 70)
    member, r = mo.token_rounding(s, topk, M)
    assert r[:4].tolist() == [0, 128, 128, 256]
    assert np.all(member.sum(0) == r)


def _brute_force_round(scores, topk, M):
    """Enumerate every token subset of the rounded size; keep the one whose members, listed by
    priority (score desc, token asc), are lexicographically best, subject to keeping all routed
    tokens (pad) or only routed tokens (drop)."""
    T, E = scores.shape
    routed = np.zeros((T, E), bool)
    routed[np.arange(T)[:, None], topk] = True
    member = np.zeros((T, E), bool)
    for e in range(E):
        c = int(routed[:, e].sum())
        r = min(M * ((c + M // 2) // M), M * (T // M))
        best, best_key = None, None
        for S in itertools.combinations(range(T), r):
            S = set(S)
            R = set(np.nonzero(routed[:, e])[0].tolist())
            if (r <= c and not S <= R) or (r > c and not R <= S):
                continue
            # rank of each token in the priority order, smaller = better
            key = sorted((-scores[t, e], t) for t in S)
            if best_key is None or key < best_key:
                best, best_key = S, key
        for t in best:
            member[t, e] = True
    return member


def test_token_rounding_brute_force():
    rng = np.random.default_rng(80)
    for trial in range(60):
        T = int(rng.integers(2, 9))
        E = int(rng.integers(1, 4))
        K = int(rng.integers(1, E + 1))
        M = 2
        s = rng.random((T, E))
        if trial % 3 == 0:
            s = np.round(s * 3) / 3  # force score ties
        topk = mo.topk_experts(s, K)
        member, r = mo.token_rounding(s, topk, M)
        assert np.array_equal(member, _brute_force_round(s, topk, M)), trial
        assert np.all(r % M == 0)


@pytest.mark.parametrize("T,E,K,M", [(1024, 16, 2, 64), (2048, 40, 4, 128)])
def test_token_rounding_invariants(T, E, K, M):
    L = _rand((T, E), T + E)
    s = mo.softmax(L)
    topk = mo.topk_experts(L, K)
    routed = np.zeros((T, E), bool)
    routed[np.arange(T)[:, None], topk] = True
    member, r = mo.token_rounding(s, topk, M)
    c = routed.sum(0)
    assert np.all(r % M == 0) and np.all(np.abs(r - c) <= M // 2) and np.all(member.sum(0) == r)
    for e in range(E):
        pad = member[:, e] & ~routed[:, e]
        unchosen = ~member[:, e] & ~routed[:, e]
        drop = routed[:, e] & ~member[:, e]
        kept = routed[:, e] & member[:, e]
        if pad.any() and unchosen.any():
            assert s[pad, e].min() >= s[unchosen, e].max()
        if drop.any() and kept.any():
            assert s[drop, e].max() <= s[kept, e].min()
    # every final pair is in the expert-major order, tokens ascending
    rt = mo.route_discrete(L, K, m_tile=M, scores=s)
    assert np.array_equal(rt.counts, r)
    for e in range(E):
        assert np.all(np.diff(rt.rows_of(e)) > 0)


# ---------------------------------------------------------------- capacity (drop/pad) dispatch


def test_capacity_closed_values():
    # C = ceil(cf * T * K / E)
    assert mo.expert_capacity(4096, 128, 8, 1.0) == 256
    assert mo.expert_capacity(4096, 128, 8, 1.25) == 320
    assert mo.expert_capacity(10, 3, 2, 1.0) == 7
    assert mo.expert_capacity(5, 4, 1, 0.5) == 1


def test_capacity_probs_worked_values():
    # expert 0 receives tokens 0, 1, 3, 4 with probabilities .9, .5, .5, .8; expert 1 token 2
    ids = np.array([[0], [0], [1], [0], [0]])
    keys = np.array([[0.9], [0.5], [0.7], [0.5], [0.8]])
    m = mo.capacity_drop(ids, keys, 2, 2, "probs")
    assert sorted(np.nonzero(m[:, 0])[0].tolist()) == [0, 4] and np.nonzero(m[:, 1])[0].tolist() == [2]
    m = mo.capacity_drop(ids, keys, 2, 3, "probs")  # the tie at .5 goes to the lower token
    assert sorted(np.nonzero(m[:, 0])[0].tolist()) == [0, 1, 4]
    m = mo.capacity_drop(ids, keys, 2, 2, "position")  # first two in token order
    assert sorted(np.nonzero(m[:, 0])[0].tolist()) == [0, 1]


@pytest.mark.parametrize("policy", ["position", "probs"])
def test_capacity_brute_force_and_invariants(policy):
    rng = np.random.default_rng(7)
    T, E, K = 60, 6, 3
    L = rng.standard_normal((T, E))
    topk = mo.topk_experts(L, K)
    keys = np.take_along_axis(mo.combine_weights(L, topk), topk, axis=1)
    for C in (1, 5, 30, T):
        m = mo.capacity_drop(topk, keys, E, C, policy)
        # streaming reference: visit pairs in priority order, keep while the expert has room
        pairs = [(t, int(topk[t, k]), keys[t, k]) for t in range(T) for k in range(K)]
        if policy == "probs":
            pairs.sort(key=lambda x: (-x[2], x[0]))
        ref = np.zeros((T, E), dtype=bool)
        room = np.full(E, C)
        for t, e, _ in pairs:
            if room[e] > 0:
                ref[t, e] = True
                room[e] -= 1
        np.testing.assert_array_equal(m, ref)
        c = np.bincount(topk.reshape(-1), minlength=E)
        np.testing.assert_array_equal(m.sum(0), np.minimum(c, C))
    # capacity above every count keeps the plain top-K routing
    r0 = mo.route_discrete(L, K)
    r1 = mo.route_discrete(L, K, capacity=T, policy=policy)
    for f in ("member", "counts", "offsets", "sorted_tok", "tok_ptr", "tok_pairs"):
        np.testing.assert_array_equal(getattr(r0, f), getattr(r1, f))


@pytest.mark.parametrize("policy", ["position", "probs"])
def test_capacity_backward_matches_autograd(policy):
    T, d, E, n, K = 12, 8, 4, 5, 2
    X, W_r, b = _rand((T, d), 50), _rand((d, E), 51, 0.5), _rand((E,), 52, 0.5)
    Wg, Wu, Wd = _rand((E, n, d), 53, 0.4), _rand((E, n, d), 54, 0.4), _rand((E, d, n), 55, 0.4)
    dO = _rand((T, d), 56)
    O, cache = mo.moe_forward(X, W_r, b, Wg, Wu, Wd, K, capacity=4, policy=policy)
    r = cache["routing"]
    assert r.member.sum() < T * K, "capacity 4 should drop pairs"
    g = mo.moe_backward(X, W_r, b, Wg, Wu, Wd, dO, cache)
    ref = _dense_loss_torch(X, W_r, b, Wg, Wu, Wd, dO, r.member, r.topk_ids)
    np.testing.assert_allclose(O, ref["O"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dX"], ref["dX"], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dW_r"], ref["dW_r"], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dlogits"], ref["dlogits"], rtol=1e-10, atol=1e-12)
    for e in range(E):
        np.testing.assert_allclose(g["dW_gate"][e], ref["dWg"][e], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(g["dW_down"][e], ref["dWd"][e], rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- FP8 (e4m3) gate/up variant


def test_e4m3_rounding_matches_torch():
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal(50000) * 100, rng.standard_normal(50000) * 1e-3,
                        rng.uniform(-463, 463, 20000)]).astype(np.float32)
    # exact ties between neighbours of the e4m3 grid at several binades
    grid = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ties = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, ties, -ties])
    # torch's conversion does not saturate (|x| >= 464 gives NaN); the satfinite clamp is pinned separately
    x = x[np.abs(x) < 464]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn)
    np.testing.assert_array_equal(mo.e4m3_round(x), ref.to(torch.float64).numpy())
    np.testing.assert_array_equal(mo.e4m3_encode(mo.e4m3_round(x)), ref.view(torch.uint8).numpy())
    codes = np.arange(0, 256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]  # no NaN patterns
    np.testing.assert_array_equal(mo.e4m3_decode(codes),
                                  torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy())


def test_e4m3_closed_values():
    v = np.array([448.0, 1.0, 2.0 ** -9, 1.0625, 1.1875, 2.0 ** -10, 460.0, -3.3])
    np.testing.assert_array_equal(mo.e4m3_round(v), [448.0, 1.0, 2.0 ** -9, 1.0, 1.25, 0.0, 448.0, -3.25])
    np.testing.assert_array_equal(mo.e4m3_encode(mo.e4m3_round(v[:3])), [0x7E, 0x38, 0x01])
    # satfinite: anything beyond the largest finite value clamps to +-448
    np.testing.assert_array_equal(mo.e4m3_round(np.array([1e6, -500.0, 464.0])), [448.0, -448.0, 448.0])


def test_quantize_rows_scale_and_error():
    rng = np.random.default_rng(12)
    M = rng.standard_normal((40, 96)).astype(np.float32)
    q, s = mo.quantize_rows_e4m3(M)
    D = mo.dequantize_rows_e4m3(q, s)
    # the largest element of every row lands on +-448 times the scale
    np.testing.assert_array_equal(np.max(np.abs(mo.e4m3_decode(q)), axis=1), 448.0)
    np.testing.assert_array_equal(s, (np.max(np.abs(M), axis=1) / np.float32(448)).astype(np.float32))
    # relative error of normal-range values at most half a unit of the 3-bit mantissa
    big = np.abs(M) >= (2.0 ** -6) * s[:, None]
    assert np.max(np.abs(D - M)[big] / np.abs(M)[big]) <= 2.0 ** -4 + 1e-7


def test_fp8_forward_reduces_to_bf16_on_representable_inputs():
    # rows whose largest magnitude is 448 * 2^-k get a power-of-two scale, and elements that are e4m3 values
    # times that scale quantize without error, so the e4m3 forward equals the plain forward: X rows reach
    # 3.5 (scale 2^-7, elements in {-3..3}), weight rows reach 0.875 (scale 2^-9, elements in {-0.5, 0, 0.5})
    rng = np.random.default_rng(13)
    T, d, E, n, K = 24, 16, 4, 8, 2
    X = rng.integers(-3, 4, (T, d)).astype(np.float64)
    X[:, 0] = 3.5
    W_r = rng.standard_normal((d, E)) * 0.3
    Wg = rng.integers(-1, 2, (E, n, d)).astype(np.float64) * 0.5
    Wu = rng.integers(-1, 2, (E, n, d)).astype(np.float64) * 0.5
    Wg[:, :, 0] = 0.875
    Wu[:, :, 0] = -0.875
    Wd = rng.standard_normal((E, d, n)) * 0.2
    O8, c8 = mo.moe_forward_fp8(X, W_r, None, Wg, Wu, Wd, K)
    O, c = mo.moe_forward(X, W_r, None, Wg, Wu, Wd, K)
    np.testing.assert_allclose(O8, O, rtol=1e-12, atol=1e-12)
    for e in range(E):
        lo, hi = c["routing"].offsets[e], c["routing"].offsets[e + 1]
        h, u, _, _ = mo.expert_ffn(X[c["routing"].rows_of(e)], Wg[e], Wu[e], Wd[e])
        np.testing.assert_allclose(c8["h"][lo:hi], h, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(c8["u"][lo:hi], u, rtol=1e-12, atol=1e-12)


def test_fp8_gate_up_within_quantization_bound():
    # |x_i - xq_i| <= max(2^-4 |x_i|, 2^-10 s) (half a step of the 3-bit mantissa, or of the subnormal
    # spacing 2^-9 s), likewise for the weights; h from the quantized operands stays within the
    # resulting bound of the exact h, element by element, and differs from it (the quantization is real)
    rng = np.random.default_rng(14)
    T, d, E, n, K = 32, 64, 4, 16, 2
    X = rng.standard_normal((T, d)).astype(np.float32)
    Wg = (rng.standard_normal((E, n, d)) * 0.05).astype(np.float32)
    Wu = (rng.standard_normal((E, n, d)) * 0.05).astype(np.float32)
    W_r = rng.standard_normal((d, E)) * 0.3
    Wd = rng.standard_normal((E, d, n)) * 0.05
    O8, c8 = mo.moe_forward_fp8(X, W_r, None, Wg, Wu, Wd, K)
    r = c8["routing"]
    xs = c8["xs"].astype(np.float64)
    dx = np.maximum(2.0 ** -4 * np.abs(X), 2.0 ** -10 * xs[:, None])
    for e in range(E):
        lo, hi = r.offsets[e], r.offsets[e + 1]
        rows = r.rows_of(e)
        for W, key, skey in ((Wg[e], "h", "gs"), (Wu[e], "u", "us")):
            ws = c8[skey][e * n:(e + 1) * n].astype(np.float64)
            dw = np.maximum(2.0 ** -4 * np.abs(W), 2.0 ** -10 * ws[:, None])
            exact = X[rows].astype(np.float64) @ W.astype(np.float64).T
            bound = np.abs(X[rows]) @ dw.T + dx[rows] @ np.abs(W).T + dx[rows] @ dw.T
            err = np.abs(c8[key][lo:hi] - exact)
            assert np.all(err <= bound * (1 + 1e-9) + 1e-300)
            assert np.max(err) > 0
    O, _ = mo.moe_forward(X, W_r, None, Wg, Wu, Wd, K)
    assert 0 < np.max(np.abs(O8 - O)) < 0.2 * np.max(np.abs(O))


def test_round_bf16_matches_torch_and_ties():
    rng = np.random.default_rng(15)
    # values with at most 24 significant bits, where torch's conversion (through fp32) is exact RNE
    x = rng.standard_normal(20000).astype(np.float32).astype(np.float64) * np.exp2(rng.integers(-20, 20, 20000))
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(mo.round_bf16(x), ref)
    # halfway cases round to the even neighbour
    np.testing.assert_array_equal(mo.round_bf16([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 3.0]),
                                  [1.0, 1 + 2.0 ** -6, -1.0, 3.0])


def test_fp8_down_within_quantization_bound():
    # with e4m3 down-projection operands, y differs from (bf16 A) W_down^T by at most the element-wise
    # quantization bound of A's rows and W_down's rows, and does differ
    rng = np.random.default_rng(16)
    T, d, E, n, K = 32, 64, 4, 32, 2
    X = rng.standard_normal((T, d)).astype(np.float32)
    Wg = (rng.standard_normal((E, n, d)) * 0.1).astype(np.float32)
    Wu = (rng.standard_normal((E, n, d)) * 0.1).astype(np.float32)
    Wd = (rng.standard_normal((E, d, n)) * 0.1).astype(np.float32)
    W_r = rng.standard_normal((d, E)) * 0.3
    O8, c8 = mo.moe_forward_fp8(X, W_r, None, Wg, Wu, Wd, K, fp8_down=True)
    O8g, c8g = mo.moe_forward_fp8(X, W_r, None, Wg, Wu, Wd, K)
    r = c8["routing"]
    np.testing.assert_array_equal(c8["h"], c8g["h"])  # the gate/up part is unchanged
    a = mo.round_bf16(c8["a"])
    da = np.maximum(2.0 ** -4 * np.abs(a), 2.0 ** -10 * c8["as_"].astype(np.float64)[:, None])
    for e in range(E):
        lo, hi = r.offsets[e], r.offsets[e + 1]
        W = Wd[e].astype(np.float64)
        dw = np.maximum(2.0 ** -4 * np.abs(W), 2.0 ** -10 * c8["ds"][e * d:(e + 1) * d].astype(np.float64)[:, None])
        exact = a[lo:hi] @ W.T
        bound = np.abs(a[lo:hi]) @ dw.T + da[lo:hi] @ np.abs(W).T + da[lo:hi] @ dw.T
        err = np.abs(c8["y_sorted"][lo:hi] - exact)
        assert np.all(err <= bound * (1 + 1e-9) + 1e-300)
        assert np.max(err) > 0
    assert 0 < np.max(np.abs(O8 - O8g)) < 0.2 * np.max(np.abs(O8g))


def test_fp8_dx_within_quantization_bound():
    # with e4m3 dX operands, each pair's dX contribution differs from (bf16 [dH|dU]) [W_gate; W_up] by at
    # most the element-wise quantization bound of the two rows, and does differ; the rest is unchanged
    rng = np.random.default_rng(17)
    T, d, E, n, K = 24, 64, 4, 32, 2
    X = rng.standard_normal((T, d)).astype(np.float32)
    Wg = (rng.standard_normal((E, n, d)) * 0.1).astype(np.float32)
    Wu = (rng.standard_normal((E, n, d)) * 0.1).astype(np.float32)
    Wd = (rng.standard_normal((E, d, n)) * 0.1).astype(np.float32)
    W_r = rng.standard_normal((d, E)) * 0.3
    dO = rng.standard_normal((T, d)).astype(np.float32)
    O, cache = mo.moe_forward(X, W_r, None, Wg, Wu, Wd, K)
    g16 = mo.moe_backward(X, W_r, None, Wg, Wu, Wd, dO, cache)
    g8 = mo.moe_backward(X, W_r, None, Wg, Wu, Wd, dO, cache, fp8_dx=True)
    for k in ("dW_r", "dlogits", "dw"):
        np.testing.assert_array_equal(g8[k], g16[k])
    r = cache["routing"]
    w = cache["w_full"]
    bound = np.zeros((T, d))
    for e in range(E):
        rows = r.rows_of(e)
        if len(rows) == 0:
            continue
        blk = mo.expert_block_backward(X[rows], dO[rows], w[rows, e], Wg[e], Wu[e], Wd[e])
        hu = mo.round_bf16(np.concatenate([blk["dh"], blk["du"]], axis=1))
        _, hs = mo.quantize_rows_e4m3(hu.astype(np.float32))
        B = np.concatenate([Wg[e], Wu[e]], axis=0).T.astype(np.float64)
        _, bs = mo.quantize_rows_e4m3(B.astype(np.float32))
        dh = np.maximum(2.0 ** -4 * np.abs(hu), 2.0 ** -10 * hs.astype(np.float64)[:, None])
        db = np.maximum(2.0 ** -4 * np.abs(B), 2.0 ** -10 * bs.astype(np.float64)[:, None])
        bound[rows] += np.abs(hu) @ db.T + dh @ np.abs(B).T + dh @ db.T
        # reference with the bf16 [dH|dU] rows and exact weights
        g16["dX"][rows] += hu @ B.T - blk["dx"]
    err = np.abs(g8["dX"] - g16["dX"])
    assert np.all(err <= bound * (1 + 1e-9) + 1e-12)
    assert np.max(err) > 0


def test_fp8_dact_within_quantization_bound():
    # with e4m3 dA' operands (dO per token, W_down^T per row): dA' within the element-wise quantization bound
    # of the exact dO W_down, dS = <dA', A> exactly, and the weight gradients of W_down unchanged
    rng = np.random.default_rng(18)
    T, d, E, n, K = 24, 64, 4, 32, 2
    X = rng.standard_normal((T, d)).astype(np.float32)
    Wg = (rng.standard_normal((E, n, d)) * 0.1).astype(np.float32)
    Wu = (rng.standard_normal((E, n, d)) * 0.1).astype(np.float32)
    Wd = (rng.standard_normal((E, d, n)) * 0.1).astype(np.float32)
    W_r = rng.standard_normal((d, E)) * 0.3
    dO = rng.standard_normal((T, d)).astype(np.float32)
    O, cache = mo.moe_forward(X, W_r, None, Wg, Wu, Wd, K)
    g16 = mo.moe_backward(X, W_r, None, Wg, Wu, Wd, dO, cache)
    g8 = mo.moe_backward(X, W_r, None, Wg, Wu, Wd, dO, cache, fp8_dact=True)
    r = cache["routing"]
    w = cache["w_full"]
    for e in range(E):
        rows = r.rows_of(e)
        if len(rows) == 0:
            continue
        np.testing.assert_allclose(g8["dW_down"][e], g16["dW_down"][e], rtol=1e-12, atol=1e-12)
        D = dO[rows].astype(np.float64)
        Bt = Wd[e].T.astype(np.float64)  # [n, d]
        _, os_ = mo.quantize_rows_e4m3(D.astype(np.float32))
        _, ws_ = mo.quantize_rows_e4m3(Bt.astype(np.float32))
        dd = np.maximum(2.0 ** -4 * np.abs(D), 2.0 ** -10 * os_.astype(np.float64)[:, None])
        db = np.maximum(2.0 ** -4 * np.abs(Bt), 2.0 ** -10 * ws_.astype(np.float64)[:, None])
        bound = np.abs(D) @ db.T + dd @ np.abs(Bt).T + dd @ db.T
        blk = mo.expert_block_backward(X[rows], dO[rows], w[rows, e], Wg[e], Wu[e], Wd[e])
        exact = D @ Bt.T
        oq, _ = mo.quantize_rows_e4m3(D.astype(np.float32))
        wq, _ = mo.quantize_rows_e4m3(Bt.astype(np.float32))
        dap = mo.dequantize_rows_e4m3(oq, os_) @ mo.dequantize_rows_e4m3(wq, ws_).T
        assert np.all(np.abs(dap - exact) <= bound * (1 + 1e-9) + 1e-12) and np.max(np.abs(dap - exact)) > 0
        np.testing.assert_allclose(g8["dw"][rows, e], np.sum(dap * blk["a"], axis=1), rtol=1e-12, atol=1e-12)
    assert 0 < np.max(np.abs(g8["dX"] - g16["dX"])) < 0.2 * np.max(np.abs(g16["dX"]))


# ---------------------------------------------------------------- block-scaled (1 x 32) e4m3


def test_mx_block_exponent_is_the_smallest_that_fits():
    # the definition, by brute force over every admissible exponent: the smallest e with amax <= 448 2^e
    rng = np.random.default_rng(21)
    amax = np.concatenate([np.exp2(rng.uniform(-140, 120, 3000)),
                           448.0 * np.exp2(np.arange(-30, 30)),                # exactly on a boundary
                           448.0 * np.exp2(np.arange(-30, 30)) * (1 + 2.0 ** -20),  # just above it
                           [2.0 ** -133, 2.0 ** -126, 1.0, 0.5, 3.0e38]])
    e = oracle.mx_block_exponents(amax)
    grid = np.arange(-127, 128)
    for a, got in zip(amax, e):
        fits = grid[a <= 448.0 * np.exp2(grid.astype(np.float64))]
        assert got == fits[0], (a, got, fits[0])
    np.testing.assert_array_equal(oracle.mx_block_exponents([0.0, 448.0, 449.0, 256.0, 1.75, 1.76]),
                                  [0, 0, 1, 0, -8, -7])


def test_mx_codes_match_torch_conversion():
    # codes are torch's float8_e4m3fn conversion of x 2^-e (an exact scaling), block by block
    rng = np.random.default_rng(22)
    M = (rng.standard_normal((64, 256)) * np.exp2(rng.integers(-20, 20, (64, 1)))).astype(np.float32)
    M[3, 32:64] = 0.0  # an all-zero block
    M[5, :32] *= 1e-30  # a block far below 1
    q, e = oracle.quantize_blocks_mx(M)
    assert e.shape == (64, 8) and e[3, 1] == 0
    y = np.ldexp(M.astype(np.float64), -np.repeat(e, 32, axis=1))
    ref = torch.from_numpy(y.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(q, ref)
    # no block saturates: its largest scaled value lies in (224, 448], its code (rounded) in [224, 448]
    mags = np.abs(mo.e4m3_decode(q)).reshape(64, 8, 32).max(axis=2)
    nz = np.abs(M).reshape(64, 8, 32).max(axis=2) > 0
    assert np.all((mags[nz] >= 224) & (mags[nz] <= 448))


def test_mx_round_trip_exact_on_representable_blocks_and_error_bound():
    rng = np.random.default_rng(23)
    grid = mo.e4m3_decode(np.arange(0, 127, dtype=np.uint8))
    R, C = 16, 128
    vals = rng.choice(grid, (R, C)) * rng.choice([-1.0, 1.0], (R, C))
    vals[:, ::32] = rng.choice(grid[(grid > 224) & (grid <= 448)], (R, C // 32))  # the block maximum
    ex = rng.integers(-40, 40, (R, C // 32))
    V = np.ldexp(vals, np.repeat(ex, 32, axis=1))
    q, e = oracle.quantize_blocks_mx(V)
    np.testing.assert_array_equal(e, ex)
    np.testing.assert_array_equal(oracle.dequantize_blocks_mx(q, e), V)
    # general inputs: |x - deq| <= max(2^-4 |x|, 2^-10 2^e) (half a mantissa step, or of the subnormal step)
    M = rng.standard_normal((40, 96))
    q, e = oracle.quantize_blocks_mx(M)
    D = oracle.dequantize_blocks_mx(q, e)
    bound = np.maximum(2.0 ** -4 * np.abs(M), 2.0 ** -10 * np.exp2(np.repeat(e, 32, axis=1).astype(np.float64)))
    assert np.all(np.abs(D - M) <= bound) and np.max(np.abs(D - M)) > 0


def _mx_bound(M):
    _, e = oracle.quantize_blocks_mx(M)
    return np.maximum(2.0 ** -4 * np.abs(M), 2.0 ** -10 * np.exp2(np.repeat(e, 32, axis=-1).astype(np.float64)))


def test_mx_forward_reduces_to_bf16_on_representable_inputs():
    # blocks whose elements are e4m3 values times a power of two (maximum in (224, 448] times it) quantize
    # without error, so the gate/up projections and O equal the plain forward's
    rng = np.random.default_rng(24)
    T, d, E, n, K = 24, 64, 4, 32, 2
    X = rng.integers(-3, 4, (T, d)).astype(np.float64)
    X[:, ::32] = 3.5  # the block maximum: 448 2^-7
    W_r = rng.standard_normal((d, E)) * 0.3
    Wg = rng.integers(-1, 2, (E, n, d)).astype(np.float64) * 0.5
    Wu = rng.integers(-1, 2, (E, n, d)).astype(np.float64) * 0.5
    Wg[:, :, ::32] = 0.875
    Wu[:, :, ::32] = -0.875
    Wd = rng.standard_normal((E, d, n)) * 0.2
    Om, cm = oracle.moe_forward_mx(X, W_r, None, Wg, Wu, Wd, K, mx_down=False)
    O, c = mo.moe_forward(X, W_r, None, Wg, Wu, Wd, K)
    np.testing.assert_allclose(Om, O, rtol=1e-12, atol=1e-12)


def test_mx_forward_within_quantization_bound():
    # gate/up: h from the quantized operands within the element-wise bound of the exact product; down
    # projection: y within the bound of A's and W_down's quantization; both differ (the quantization is real)
    rng = np.random.default_rng(25)
    T, d, E, n, K = 32, 64, 4, 64, 2
    X = rng.standard_normal((T, d))
    Wg = rng.standard_normal((E, n, d)) * 0.05
    Wu = rng.standard_normal((E, n, d)) * 0.05
    Wd = rng.standard_normal((E, d, n)) * 0.05
    W_r = rng.standard_normal((d, E)) * 0.3
    Om, cm = oracle.moe_forward_mx(X, W_r, None, Wg, Wu, Wd, K)
    r = cm["routing"]
    dx = _mx_bound(X)
    for e in range(E):
        lo, hi = r.offsets[e], r.offsets[e + 1]
        if hi == lo:
            continue
        rows = r.rows_of(e)
        for W, key in ((Wg[e], "h"), (Wu[e], "u")):
            dw = _mx_bound(W)
            bound = np.abs(X[rows]) @ dw.T + dx[rows] @ np.abs(W).T + dx[rows] @ dw.T
            err = np.abs(cm[key][lo:hi] - X[rows] @ W.T)
            assert np.all(err <= bound * (1 + 1e-9)) and np.max(err) > 0
        a = cm["a"][lo:hi]
        da, dwd = _mx_bound(a), _mx_bound(Wd[e])
        bound = np.abs(a) @ dwd.T + da @ np.abs(Wd[e]).T + da @ dwd.T
        err = np.abs(cm["y_sorted"][lo:hi] - a @ Wd[e].T)
        assert np.all(err <= bound * (1 + 1e-9)) and np.max(err) > 0
    O, _ = mo.moe_forward(X, W_r, None, Wg, Wu, Wd, K)
    assert 0 < np.max(np.abs(Om - O)) < 0.1 * np.max(np.abs(O))


def test_mx_backward_gemms_within_quantization_bound():
    # mx_dact: dA' within the bound of dO's and W_down^T's quantization, dS = <dA', A>; mx_dx: each pair's
    # dX contribution within the bound of [dH | dU]'s and [W_gate; W_up]^T's quantization; the weight
    # gradients of the experts are those of the exact backward when only dX is quantized
    rng = np.random.default_rng(26)
    T, d, E, n, K = 24, 64, 4, 32, 2
    X = rng.standard_normal((T, d))
    Wg = rng.standard_normal((E, n, d)) * 0.1
    Wu = rng.standard_normal((E, n, d)) * 0.1
    Wd = rng.standard_normal((E, d, n)) * 0.1
    W_r = rng.standard_normal((d, E)) * 0.3
    dO = rng.standard_normal((T, d))
    O, cache = mo.moe_forward(X, W_r, None, Wg, Wu, Wd, K)
    g = mo.moe_backward(X, W_r, None, Wg, Wu, Wd, dO, cache)
    gx = mo.moe_backward(X, W_r, None, Wg, Wu, Wd, dO, cache, mx_dx=True)
    ga = mo.moe_backward(X, W_r, None, Wg, Wu, Wd, dO, cache, mx_dact=True)
    for k in ("dW_r", "dlogits", "dw"):
        np.testing.assert_array_equal(gx[k], g[k])
    r, w = cache["routing"], cache["w_full"]
    bound = np.zeros((T, d))
    for e in range(E):
        rows = r.rows_of(e)
        if len(rows) == 0:
            continue
        np.testing.assert_array_equal(gx["dW_gate"][e], g["dW_gate"][e])
        blk = mo.expert_block_backward(X[rows], dO[rows], w[rows, e], Wg[e], Wu[e], Wd[e])
        hu = np.concatenate([blk["dh"], blk["du"]], axis=1)
        B = np.concatenate([Wg[e], Wu[e]], axis=0).T
        dh, db = _mx_bound(hu), _mx_bound(B)
        bound[rows] += np.abs(hu) @ db.T + dh @ np.abs(B).T + dh @ db.T
        Bt = Wd[e].T
        do, dbt = _mx_bound(dO[rows]), _mx_bound(Bt)
        dap_bound = np.abs(dO[rows]) @ dbt.T + do @ np.abs(Bt).T + do @ dbt.T
        oq, oe = oracle.quantize_blocks_mx(dO[rows])
        wq, we = oracle.quantize_blocks_mx(Bt)
        dap = oracle.dequantize_blocks_mx(oq, oe) @ oracle.dequantize_blocks_mx(wq, we).T
        err = np.abs(dap - dO[rows] @ Bt.T)
        assert np.all(err <= dap_bound * (1 + 1e-9)) and np.max(err) > 0
        np.testing.assert_allclose(ga["dw"][rows, e], np.sum(dap * blk["a"], axis=1), rtol=1e-12, atol=1e-12)
    err = np.abs(gx["dX"] - g["dX"])
    assert np.all(err <= bound * (1 + 1e-9) + 1e-12) and np.max(err) > 0


def _token_blocks_brute(M):
    """Block-scaled values with 1 x 32 blocks down each column (the last block partial), written out
    element by element: the block's exponent by search over every admissible e, the code by torch's
    float8_e4m3fn conversion of the exactly scaled value."""
    M = np.asarray(M, dtype=np.float64)
    R, C = M.shape
    out = np.zeros_like(M)
    grid = np.arange(-127, 128)
    for c in range(C):
        for b0 in range(0, R, 32):
            blk = M[b0:b0 + 32, c]
            amax = np.max(np.abs(blk))
            e = 0 if amax == 0 else grid[amax <= 448.0 * np.exp2(grid.astype(np.float64))][0]
            y = torch.from_numpy(np.ldexp(blk, -int(e)).astype(np.float32)).to(torch.float8_e4m3fn)
            out[b0:b0 + 32, c] = np.ldexp(y.to(torch.float64).numpy(), int(e))
    return out


def test_mx_token_blocks_match_brute_force():
    # blocks of 32 rows of one column, the last one over the 13 rows left; magnitudes differ per column and an
    # all-zero block and a block far below 1 are included
    rng = np.random.default_rng(27)
    M = rng.standard_normal((45, 6)) * np.exp2(rng.integers(-12, 12, (1, 6)))
    M[:32, 2] = 0.0
    M[32:, 4] *= 1e-25
    got = oracle.dequantize_token_blocks_mx(M)
    np.testing.assert_array_equal(got, _token_blocks_brute(M))
    assert np.max(np.abs(got - M)) > 0
    # a block's scale depends on its own rows alone: a large value in row 40 leaves rows 0..31 unchanged
    M2 = M.copy()
    M2[40, :] = 1e6
    np.testing.assert_array_equal(oracle.dequantize_token_blocks_mx(M2)[:32], got[:32])


def test_mx_weight_gradients_token_blocks_and_bound():
    # mx_dw: every expert's dW_gate, dW_up, dW_down equal the products of its operands quantized by the
    # brute-force token blocks (blocks starting at the expert's first row), lie within the element-wise
    # quantization bound of the exact gradients, and the other gradients are the exact backward's
    rng = np.random.default_rng(28)
    T, d, E, n, K = 96, 64, 4, 32, 2
    X = rng.standard_normal((T, d))
    Wg = rng.standard_normal((E, n, d)) * 0.1
    Wu = rng.standard_normal((E, n, d)) * 0.1
    Wd = rng.standard_normal((E, d, n)) * 0.1
    W_r = rng.standard_normal((d, E)) * 0.3
    dO = rng.standard_normal((T, d))
    O, cache = mo.moe_forward(X, W_r, None, Wg, Wu, Wd, K)
    g = mo.moe_backward(X, W_r, None, Wg, Wu, Wd, dO, cache)
    gw = mo.moe_backward(X, W_r, None, Wg, Wu, Wd, dO, cache, mx_dw=True)
    for k in ("dX", "dW_r", "dlogits", "dw"):
        np.testing.assert_array_equal(gw[k], g[k])
    r, w = cache["routing"], cache["w_full"]
    seen_ragged = False
    for e in range(E):
        rows = r.rows_of(e)
        if len(rows) == 0:
            continue
        seen_ragged |= len(rows) % 32 != 0 and len(rows) > 32
        blk = mo.expert_block_backward(X[rows], dO[rows], w[rows, e], Wg[e], Wu[e], Wd[e])
        ap = w[rows, e][:, None] * blk["a"]
        qx = _token_blocks_brute(X[rows])
        pairs = ((gw["dW_gate"][e], g["dW_gate"][e], blk["dh"], X[rows], qx),
                 (gw["dW_up"][e], g["dW_up"][e], blk["du"], X[rows], qx),
                 (gw["dW_down"][e], g["dW_down"][e], dO[rows], ap, _token_blocks_brute(ap)))
        for got, exact, A, B, qB in pairs:
            np.testing.assert_allclose(got, _token_blocks_brute(A).T @ qB, rtol=1e-12, atol=1e-13)
            da, db = (np.abs(_token_blocks_brute(M) - M) for M in (A, B))
            bound = np.abs(A).T @ db + da.T @ np.abs(B) + da.T @ db
            err = np.abs(got - exact)
            assert np.all(err <= bound * (1 + 1e-9) + 1e-13) and np.max(err) > 0
    assert seen_ragged  # an expert with a partial last block


# ---------------------------------------------------------------- the metric


def test_metric_scale():
    o = np.array([[1.0, -2.0, 0.0, 4.0], [0.01, 0.0, 0.02, -0.02]])
    assert oracle.rel_error(o, o)["max"] == 0.0
    r = oracle.rel_error(o + np.array([[0.0, 0.0, 0.05, 0.0], [0.0, 0.0, 0.0, 0.0]]), o)
    # a perturbation of an exact zero is judged against its row's rms (sqrt(21/4))
    assert abs(r["max"] - 0.05 / math.sqrt(21 / 4)) < 1e-12
    r = oracle.rel_error(o + np.array([[0.0, 0.0, 0.0, 0.0], [0.0, 0.001, 0.0, 0.0]]), o)
    # in a small row the floor is that row's rms, not the tensor's
    assert abs(r["max"] - 0.001 / math.sqrt(0.0009 / 4)) < 1e-9
    assert r["max_global"] < r["max"]


def test_metric_weight_gradient_floor():
    # [experts, rows, cols]: expert 0 has one tiny row, expert 1 is all zero
    o = np.zeros((2, 2, 3))
    o[0] = [[3.0, -4.0, 0.0], [1e-6, 0.0, -1e-6]]
    g = o.copy()
    g[0, 1, 0] += 1e-7
    # per-row floor: the tiny row judges the perturbation against its own scale (|o| = 1e-6 here)
    r = oracle.rel_error(g, o)
    assert abs(r["max"] - 1e-7 / 1e-6) < 1e-9
    # weight gradient: floor max(row rms, 1e-3 * rms of expert 0's matrix, sqrt((25 + 2e-12) / 6))
    r = oracle.rel_error(g, o, param_axes=oracle.WEIGHT_GRAD)
    assert abs(r["max"] - 1e-7 / (1e-3 * math.sqrt((25 + 2e-12) / 6))) < 1e-12
    # a big row keeps its own floor: a perturbation of its exact zero is judged against the row rms
    g = o.copy()
    g[0, 0, 2] = 0.05
    r = oracle.rel_error(g, o, param_axes=oracle.WEIGHT_GRAD)
    assert abs(r["max"] - 0.05 / math.sqrt(25 / 3)) < 1e-12
    # an all-zero expert is judged against the tensor's rms
    g = o.copy()
    g[1, 0, 2] = 1e-3
    r = oracle.rel_error(g, o, param_axes=oracle.WEIGHT_GRAD)
    assert abs(r["max"] - 1e-3 / math.sqrt((25 + 2e-12) / 12)) < 1e-12


def test_bf16_widening_matches_torch_and_special_values():
    """bf16 bits -> fp64 against torch's own bf16 conversion on random non-NaN bit patterns, and exact values:
    1.0, -2.0, the smallest subnormal 2^-133, the largest finite bf16 and +inf."""
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 1 << 16, 4096, dtype=np.uint32).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # drop inf/NaN exponents
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(mo.bf16_bits_to_f64(bits), ref)
    special = np.array([0x3F80, 0xC000, 0x0001, 0x7F7F, 0x7F80], dtype=np.uint16)
    got = mo.bf16_bits_to_f64(special)
    assert got[0] == 1.0 and got[1] == -2.0 and got[2] == 2.0 ** -133
    assert got[3] == (2 - 2 ** -7) * 2.0 ** 127 and np.isinf(got[4]) and got[4] > 0


def test_router_logits_of_one_hot_tokens_are_router_rows():
    """A token whose row is the unit vector e_i scores every expert with row i of W_r (plus the bias): the
    orientation of the router product (X W_r, not its transpose) and the bias broadcast over experts."""
    d, E = 6, 4
    rng = np.random.default_rng(3)
    W_r = rng.standard_normal((d, E))
    bias = rng.standard_normal(E)
    X = np.eye(d)[[2, 0, 5]]
    L = mo.router_logits(X, W_r, bias)
    np.testing.assert_array_equal(L, W_r[[2, 0, 5]] + bias[None, :])
    np.testing.assert_array_equal(mo.router_logits(X, W_r), W_r[[2, 0, 5]])


@pytest.mark.parametrize("K,pad", [(1, False), (2, False), (3, True)])
def test_router_grad_rows_is_the_derivative_of_the_combine_weights(K, pad):
    """router_grad_rows against central differences of f(l) = sum over the token's final pairs of
    w_e(l) dw_e, with w = combine_weights(l, TopK) and the top-K set held fixed.  With ``pad`` the final set
    also holds an expert outside the top-K (a token rounding pad), whose weight still normalises over the
    top-K.  With K = 1 and no pad the weight is identically 1, so the gradient is zero."""
    rng = np.random.default_rng(11 + K)
    T, E = 5, 6
    L = rng.standard_normal((T, E))
    topk = mo.topk_experts(L, K)
    member = np.zeros((T, E), dtype=bool)
    member[np.arange(T)[:, None], topk] = True
    if pad:
        for t in range(T):
            member[t, [e for e in range(E) if not member[t, e]][0]] = True
    dw = rng.standard_normal((T, E))
    got = mo.router_grad_rows(member, topk, mo.combine_weights(L, topk), dw)
    h = 1e-6
    for t in range(T):
        for e in range(E):
            lp, lm = L.copy(), L.copy()
            lp[t, e] += h
            lm[t, e] -= h
            fp = np.sum(np.where(member, mo.combine_weights(lp, topk) * dw, 0.0)[t])
            fm = np.sum(np.where(member, mo.combine_weights(lm, topk) * dw, 0.0)[t])
            assert abs(got[t, e] - (fp - fm) / (2 * h)) < 1e-7, (t, e)
    if K == 1 and not pad:
        np.testing.assert_allclose(got, 0.0, atol=1e-15)
    if not pad:  # the weights on the top-K set sum to one, so their logit gradient sums to zero
        np.testing.assert_allclose(got.sum(axis=1), 0.0, atol=1e-12)
