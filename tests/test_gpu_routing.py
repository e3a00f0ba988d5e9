"""Routing and grouping on the device vs the oracle's discrete stage.

(i)  Given the device's own fp32 logits (and scores, under token rounding), the oracle reproduces
     topk_ids, counts, offsets, the expert-grouped order and the per-token return map bit for bit.
(ii) Against the oracle's fp64 logits: logits within the float tolerance, and every token whose
     K-th / (K+1)-th margin exceeds the fp32 summation bound has the same top-K set.
(iii) Integer-valued inputs make the logits exact, so the device's selection must equal the
     oracle's own selection with no help from the device's values (ties are frequent and
     exercise the lower-expert rule); under Token Rounding the selection is unique where the
     fp32 scores of different tokens are separated, and valid within that precision elsewhere."""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import moe_oracle as mo

from _helpers import Inputs, check_rounding_near_ties, check_routing_bit_exact, gpu_routing, run_path

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import varlen_grouped_gemm_gb300 as vgg
    return vgg.Context(0)


CASES = [
    synth.WORKLOADS["tiny"],
    synth.scaled(synth.WORKLOADS["c2"], name="c2_small", T=600, d=256, n=128),
    synth.scaled(synth.WORKLOADS["c3"], name="c3_small", T=512, d=512, E=64, n=128),
    synth.scaled(synth.WORKLOADS["c4"], name="c4_small", T=777, d=192, E=128, n=192),
    synth.scaled(synth.WORKLOADS["c5"], name="c5_small", T=2048, d=128, E=64, n=64, m_tile=64),
    synth.scaled(synth.WORKLOADS["c5"], name="c5_tr128", T=4096, d=128, E=32, n=64, m_tile=128),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_routing_bit_exact_given_device_logits(ctx, wl):
    inp = Inputs(wl, with_grad=False)
    buf = run_path(ctx, inp, backward=False)
    g = gpu_routing(buf)
    r = check_routing_bit_exact(g, wl.K, wl.m_tile)
    # weights: top-K weights vs fp64 from the device logits' selection
    L64 = mo.router_logits(inp.X, inp.W_r, inp.bias)
    oracle.compare("logits", g["logits"], L64)
    w_ref = mo.combine_weights(L64, r.topk_ids)
    oracle.compare("topk_w", g["topk_w"], np.take_along_axis(w_ref, r.topk_ids, 1))
    oracle.compare("sorted_w", g["sorted_w"], w_ref[r.sorted_tok, r.sorted_exp])
    if wl.m_tile:
        assert np.all(g["counts"] % wl.m_tile == 0)
        oracle.compare("scores", g["scores"], mo.softmax(L64))


@pytest.mark.parametrize("wl", CASES[:4], ids=lambda w: w.name)
def test_topk_sets_match_fp64_beyond_margin(ctx, wl):
    inp = Inputs(wl, with_grad=False)
    buf = run_path(ctx, inp, backward=False)
    g = gpu_routing(buf)
    X = mo.bf16_bits_to_f64(inp.X)
    Wr = mo.bf16_bits_to_f64(inp.W_r)
    L64 = mo.router_logits(inp.X, inp.W_r, inp.bias)
    own = mo.topk_experts(L64, wl.K)
    srt = -np.sort(-L64, axis=1)
    margin = srt[:, wl.K - 1] - srt[:, wl.K] if wl.K < wl.E else np.full(wl.T, np.inf)
    # fp32 summation bound on each logit: gamma_d * sum |x_i w_ie|, times 2 for two logits
    gamma = wl.d * 2.0 ** -24
    bound = 2 * gamma * (np.abs(X) @ np.abs(Wr)).max(axis=1) + 1e-6
    safe = margin > bound
    same = np.all(np.sort(own, 1) == np.sort(g["topk_ids"], 1), axis=1)
    assert np.all(same[safe]), np.nonzero(~same & safe)[0][:10]
    assert safe.mean() > 0.9


@pytest.mark.parametrize("wl", [
    synth.scaled(synth.WORKLOADS["tiny"], name="tiny_int", integer=True),
    synth.scaled(synth.WORKLOADS["c2"], name="c2_int", T=512, d=128, E=32, n=64, integer=True),
    synth.scaled(synth.WORKLOADS["c5"], name="c5_int_tr", T=1024, d=64, E=16, n=64, m_tile=64, integer=True),
    # thousands of candidates per expert with few distinct scores: the padding's threshold falls among
    # hundreds of equal scores, taken in token order
    synth.scaled(synth.WORKLOADS["c5"], name="c5_int_tr_ties", T=8192, d=64, E=16, n=64, m_tile=128, integer=True),
], ids=lambda w: w.name)
def test_integer_inputs_routing_fully_independent(ctx, wl):
    inp = Inputs(wl, with_grad=False)
    buf = run_path(ctx, inp, backward=False)
    g = gpu_routing(buf)
    L64 = mo.router_logits(inp.X, inp.W_r, inp.bias)
    np.testing.assert_array_equal(g["logits"].astype(np.float64), L64)  # exact integers
    assert (np.diff(np.sort(L64, 1), axis=1) == 0).any(), "integer logits should contain ties"
    # the oracle's own selection from its own logits and, under rounding, its own fp64 scores rounded to
    # fp32 (the precision the device compares in); nothing is taken from the device
    s32 = mo.softmax(L64).astype(np.float32) if wl.m_tile else None
    r = mo.route_discrete(L64, wl.K, wl.m_tile, scores=s32)
    np.testing.assert_array_equal(g["topk_ids"], r.topk_ids)
    np.testing.assert_array_equal(g["counts"], r.counts)
    np.testing.assert_array_equal(g["offsets"], r.offsets)
    if not wl.m_tile:
        np.testing.assert_array_equal(g["sorted_tok"], r.sorted_tok)
        np.testing.assert_array_equal(g["tok_pairs"], r.tok_pairs)
        return
    oracle.compare("scores", g["scores"], s32)
    n_diff = check_rounding_near_ties(g, L64, r)
    print(wl.name, "pairs on a near-tie threshold taken differently:", n_diff)


@pytest.mark.parametrize("reps", [3000, 100])
def test_token_rounding_repeated_tokens(ctx, reps):
    """Token rounding when tokens repeat (groups of `reps` identical rows): every expert's candidates come
    in groups of equal scores, so the threshold of both the drop and the padding selection falls inside
    a group and its equal scores are taken in token order (thousands of ties for reps=3000, tens for 100)."""
    import varlen_grouped_gemm_gb300 as vgg
    T, d, E, K, m_tile = 8192, 64, 16, 4, 128
    rng = np.random.default_rng(reps)
    X = np.repeat(rng.integers(-2, 3, (T // reps + 1, d)), reps, axis=0)[:T]
    W_r = rng.integers(-2, 3, (d, E))
    Xd = torch.tensor(X, dtype=torch.bfloat16, device="cuda")
    Wd = torch.tensor(W_r, dtype=torch.bfloat16, device="cuda")
    buf = vgg.Buffers.allocate(T, d, E, 64, K, m_tile, backward=False)
    vgg.moe_route(ctx, Xd, Wd, None, K, buf.logits, buf.scores, buf.topk_ids, buf.topk_w, buf.ws)
    vgg.moe_permute(ctx, buf.topk_ids, buf.topk_w, buf.logits, buf.scores, E, m_tile, buf.counts, buf.offsets,
                    buf.sorted_tok, buf.sorted_w, buf.tok_ptr, buf.tok_pairs, buf.P, buf.ws)
    rc, code = vgg.moe_get_error(ctx)
    assert rc == vgg.MOE_OK and code == 0, (rc, code)
    g = gpu_routing(buf)
    r = check_routing_bit_exact(g, K, m_tile)
    assert np.all(r.counts % m_tile == 0)
    c = np.bincount(r.topk_ids.reshape(-1), minlength=E)
    assert (r.counts < c).any() and (r.counts > c).any(), "both dropping and padding experts"
