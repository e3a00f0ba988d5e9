"""moe_permute_noalloc against moe_permute.

moe_permute_noalloc serves callers that cannot allocate device memory: it keeps its scratch in a
fixed array inside the library instead of taking a workspace.  Its outputs must be the same as
moe_permute's (the grouping is integer work, so the comparison is exact), on two calls in a row
(the array keeps the previous call's contents, which must not leak into the next result).
This file is collected last so that a run stopping at the first failure has run every other test.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _state(vgg, T, E, K):
    cap = vgg.moe_pair_capacity(T, E, K, 0)
    z = lambda n, dt: torch.full((n,), -7, dtype=dt, device="cuda")
    return dict(counts=z(E, torch.int32), offsets=z(E + 1, torch.int32), sorted_tok=z(cap, torch.int32),
                sorted_w=z(cap, torch.float32), tok_ptr=z(T + 1, torch.int32), tok_pairs=z(cap, torch.int32),
                P=z(1, torch.int32))


@pytest.mark.parametrize("wl", [
    synth.scaled(synth.WORKLOADS["c2"], name="c2_half", T=2048),
    synth.scaled(synth.WORKLOADS["c5_plain"], name="c5_max", T=32768, d=128, n=64),
    synth.WORKLOADS["tiny"],
], ids=lambda w: w.name)
def test_noalloc_permute_matches_permute(wl):
    import varlen_grouped_gemm_gb300 as vgg
    ctx = vgg.Context(0)
    X = torch.from_numpy(synth.make_x(wl).view(np.int16)).view(torch.bfloat16).cuda()
    W_r = torch.from_numpy(synth.make_router(wl).view(np.int16)).view(torch.bfloat16).cuda()
    logits = torch.empty((wl.T, wl.E), device="cuda")
    ids = torch.empty((wl.T, wl.K), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.T, wl.K), device="cuda")
    vgg.moe_route(ctx, X, W_r, None, wl.K, logits, None, ids, w)
    ref = _state(vgg, wl.T, wl.E, wl.K)
    ws = torch.empty(vgg.moe_workspace_bytes(wl.T, wl.d, wl.E, wl.n, wl.K, 0), dtype=torch.uint8, device="cuda")
    vgg.moe_permute(ctx, ids, w, None, None, wl.E, 0, ref["counts"], ref["offsets"], ref["sorted_tok"],
                    ref["sorted_w"], ref["tok_ptr"], ref["tok_pairs"], ref["P"], ws)
    for call in range(2):
        got = _state(vgg, wl.T, wl.E, wl.K)
        vgg.moe_permute_noalloc(ctx, ids, w, wl.E, got["counts"], got["offsets"], got["sorted_tok"],
                                got["sorted_w"], got["tok_ptr"], got["tok_pairs"], got["P"])
        assert vgg.moe_get_error(ctx) == (0, 0)
        for k in ref:
            assert torch.equal(got[k], ref[k]), (call, k)


def _route(vgg, ctx, wl, permute_experts=None):
    X = torch.from_numpy(synth.make_x(wl).view(np.int16)).view(torch.bfloat16).cuda()
    W_r = torch.from_numpy(synth.make_router(wl).view(np.int16)).view(torch.bfloat16).cuda()
    if permute_experts is not None:  # a different routing of the same shape: the router's columns shuffled
        W_r = W_r[:, torch.from_numpy(permute_experts).cuda()].contiguous()
    logits = torch.empty((wl.T, wl.E), device="cuda")
    ids = torch.empty((wl.T, wl.K), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.T, wl.K), device="cuda")
    vgg.moe_route(ctx, X, W_r, None, wl.K, logits, None, ids, w)
    return ids, w


def test_noalloc_after_a_larger_call():
    """The array keeps the previous call's contents: a call at the largest size (T = 32768, E = 512) leaves
    every count slot written, then smaller, differently routed calls must still equal moe_permute."""
    import varlen_grouped_gemm_gb300 as vgg
    ctx = vgg.Context(0)
    big = synth.scaled(synth.WORKLOADS["c5_plain"], name="noalloc_big", T=32768, d=128, n=64)
    ids, w = _route(vgg, ctx, big)
    st = _state(vgg, big.T, big.E, big.K)
    vgg.moe_permute_noalloc(ctx, ids, w, big.E, st["counts"], st["offsets"], st["sorted_tok"], st["sorted_w"],
                            st["tok_ptr"], st["tok_pairs"], st["P"])
    assert vgg.moe_get_error(ctx) == (0, 0)
    small = synth.scaled(synth.WORKLOADS["c2"], name="noalloc_small", T=777, d=128, E=64, K=4)
    for perm_seed in (1, 2):
        ids, w = _route(vgg, ctx, small, np.random.default_rng(perm_seed).permutation(small.E))
        ref = _state(vgg, small.T, small.E, small.K)
        ws = torch.empty(vgg.moe_workspace_bytes(small.T, small.d, small.E, small.n, small.K, 0), dtype=torch.uint8,
                         device="cuda")
        vgg.moe_permute(ctx, ids, w, None, None, small.E, 0, ref["counts"], ref["offsets"], ref["sorted_tok"],
                        ref["sorted_w"], ref["tok_ptr"], ref["tok_pairs"], ref["P"], ws)
        got = _state(vgg, small.T, small.E, small.K)
        vgg.moe_permute_noalloc(ctx, ids, w, small.E, got["counts"], got["offsets"], got["sorted_tok"],
                                got["sorted_w"], got["tok_ptr"], got["tok_pairs"], got["P"])
        assert vgg.moe_get_error(ctx) == (0, 0)
        for k in ref:
            assert torch.equal(got[k], ref[k]), (perm_seed, k)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import varlen_grouped_gemm_gb300 as vgg
    ctx = vgg.Context(0)
    T, E, K = 32768 + 256, 64, 2
    ids = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    ids[:, 1] = 1
    w = torch.full((T, K), 0.5, device="cuda")
    st = _state(vgg, T, E, K)
    with pytest.raises(RuntimeError, match="unsupported"):
        vgg.moe_permute_noalloc(ctx, ids, w, E, st["counts"], st["offsets"], st["sorted_tok"], st["sorted_w"],
                                st["tok_ptr"], st["tok_pairs"], st["P"])
