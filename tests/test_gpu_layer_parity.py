"""The whole layer (forward and backward) on the device vs the fp64 oracle, element by element.

Sizes span several tiles in every dimension with ragged tails (rows per expert not multiples of
128, n or d not multiples of 128/256), empty experts (skewed prior), token rounding, and the
workload shapes of the benchmark configurations scaled down so the oracle finishes in seconds.
Tolerance: max relative error <= 2e-2 and mean <= 3e-3 per tensor (bf16 inputs, fp32 accumulation),
with the relative error of an element taken against max(|ref|, rms(ref)).
The selection of experts is taken from the device's fp32 logits (bit-exactness of that stage is
checked separately), so that the float comparison is not disturbed by near-ties."""
import numpy as np
import pytest
import torch

import synth

from _helpers import Inputs, check_routing_bit_exact, compare_layer, gpu_routing, oracle_layer, run_path

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import varlen_grouped_gemm_gb300 as vgg
    return vgg.Context(0)


CASES = [
    synth.WORKLOADS["tiny"],
    synth.scaled(synth.WORKLOADS["c2"], name="c2_small", T=512, d=256, E=16, n=192, K=4),
    synth.scaled(synth.WORKLOADS["c3"], name="c3_small", T=384, d=448, E=32, n=256, K=8),
    synth.scaled(synth.WORKLOADS["c4"], name="c4_small", T=640, d=320, E=32, n=320, K=4),
    synth.scaled(synth.WORKLOADS["c5"], name="c5_small_tr", T=2048, d=192, E=32, n=128, K=8, m_tile=64),
    synth.scaled(synth.WORKLOADS["c5_plain"], name="c5_small_plain", T=2048, d=192, E=32, n=128, K=8),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_layer_matches_oracle(ctx, wl):
    inp = Inputs(wl)
    buf = run_path(ctx, inp, backward=True, dW_dtype=torch.float32)
    g = gpu_routing(buf)
    check_routing_bit_exact(g, wl.K, wl.m_tile)
    O_ref, cache, grads = oracle_layer(inp, g)
    rep = compare_layer(buf, inp, O_ref, cache, grads)
    if wl.bias == "zipf":
        assert (g["counts"] == 0).any(), "the skewed prior should leave some experts empty"
    print(wl.name, {k: (round(v["max"], 5), round(v["mean"], 6)) for k, v in rep.items()})


@pytest.mark.parametrize("wl", [CASES[1], CASES[2]], ids=lambda w: w.name)
def test_layer_with_cta_pairs(ctx, wl):
    """The same layer with the tiled varlen-M GEMMs and the weight-gradient GEMMs on CTA pairs (two CTAs per
    256-row tile): the same tolerance against the oracle."""
    inp = Inputs(wl)
    ctx.set_cta_pairs(True, True)
    try:
        buf = run_path(ctx, inp, backward=True, dW_dtype=torch.float32)
    finally:
        ctx.set_cta_pairs(False, False)
    g = gpu_routing(buf)
    O_ref, cache, grads = oracle_layer(inp, g)
    compare_layer(buf, inp, O_ref, cache, grads)


def test_dW_bf16_storage(ctx):
    wl = synth.scaled(synth.WORKLOADS["c2"], name="c2_bf16dw", T=256, d=128, E=8, n=128, K=2)
    inp = Inputs(wl)
    buf = run_path(ctx, inp, backward=True, dW_dtype=torch.bfloat16)
    g = gpu_routing(buf)
    O_ref, cache, grads = oracle_layer(inp, g)
    compare_layer(buf, inp, O_ref, cache, grads)


def test_deterministic(ctx):
    wl = synth.scaled(synth.WORKLOADS["c2"], name="c2_det", T=512, d=256, E=16, n=128, K=4)
    inp = Inputs(wl)
    a = run_path(ctx, inp, backward=True)
    b = run_path(ctx, inp, backward=True)
    for name in ("O", "dX", "dW_gate", "dW_up", "dW_down", "dS", "dlogits", "dW_r", "sorted_tok", "tok_pairs"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


def test_forward_only_skips_the_backward_cache(ctx):
    """cache=False (H = U = NULL at the C ABI): the same O bit for bit, and H, U left untouched."""
    import varlen_grouped_gemm_gb300 as vgg
    wl = synth.scaled(synth.WORKLOADS["c2"], name="c2_fwd_only", T=512, d=256, E=16, n=192, K=4)
    inp = Inputs(wl, with_grad=False)
    dv = inp.dev
    buf = vgg.Buffers.allocate(wl.T, wl.d, wl.E, wl.n, wl.K, backward=False)
    vgg.forward(ctx, dv["X"], dv["W_r"], dv["bias"], dv["W_gate"], dv["W_up"], dv["W_down"], buf)
    O_cached = buf.O.clone()
    buf.H.fill_(7.0)
    buf.U.fill_(7.0)
    buf.O.zero_()
    vgg.forward(ctx, dv["X"], dv["W_r"], dv["bias"], dv["W_gate"], dv["W_up"], dv["W_down"], buf, cache=False)
    rc, code = vgg.moe_get_error(ctx)
    assert rc == vgg.MOE_OK and code == 0, (rc, code)
    assert torch.equal(buf.O, O_cached)
    assert bool((buf.H == 7.0).all()) and bool((buf.U == 7.0).all())


def test_step_graph_replays_the_eager_step(ctx):
    """StepGraph: a captured forward + backward replays to the eager results, also after new inputs were
    copied into the captured tensors."""
    import varlen_grouped_gemm_gb300 as vgg
    wl = synth.scaled(synth.WORKLOADS["c2"], name="c2_graph", T=512, d=256, E=16, n=192, K=4)
    inp = Inputs(wl)
    dv = inp.dev
    X, dO = dv["X"].clone(), dv["dO"].clone()
    buf = vgg.Buffers.allocate(wl.T, wl.d, wl.E, wl.n, wl.K, backward=True)
    g = vgg.StepGraph(ctx, X, dv["W_r"], dv["bias"], dv["W_gate"], dv["W_up"], dv["W_down"], dO, buf)
    X.copy_(dv["X"].flip(0))  # other tokens in the same tensor
    dO.copy_(dv["dO"] * 0.5)
    g.replay()
    torch.cuda.synchronize()
    got = {k: getattr(buf, k).clone() for k in ("O", "dX", "dW_gate", "dW_up", "dW_down", "dW_r", "dlogits")}
    ref = vgg.Buffers.allocate(wl.T, wl.d, wl.E, wl.n, wl.K, backward=True)
    vgg.forward_backward(ctx, X, dv["W_r"], dv["bias"], dv["W_gate"], dv["W_up"], dv["W_down"], dO, ref)
    rc, code = vgg.moe_get_error(ctx)
    assert rc == vgg.MOE_OK and code == 0, (rc, code)
    for k, v in got.items():
        assert torch.equal(v, getattr(ref, k)), k
