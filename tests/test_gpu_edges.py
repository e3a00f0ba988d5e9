"""Edge cases of the whole layer (forward and backward) against the fp64 oracle.

The degenerate cases of the method and the limits of the C ABI: a single token, top-1 routing, K = E
(every expert takes every token), a token count that fills no block, most experts empty, token
rounding where experts round down to nothing, the capacity dispatch with a single token, the largest
expert count (1024: the widest group tables and top-K), and the largest token counts the entry points
take (65536 plain, 32768 with token rounding).  Routing bit for bit, every float output within the
usual tolerance.
"""
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


base = synth.WORKLOADS["c2"]
CASES = [
    synth.scaled(base, name="one_token_top1", T=1, d=64, E=8, n=64, K=1),
    synth.scaled(base, name="top1", T=300, d=128, E=16, n=128, K=1),
    synth.scaled(base, name="k_equals_e", T=33, d=64, E=8, n=64, K=8),
    synth.scaled(base, name="ragged_tokens", T=37, d=192, E=16, n=192, K=3),
    synth.scaled(synth.WORKLOADS["c4"], name="mostly_empty", T=5, d=64, E=64, n=64, K=2),
    synth.scaled(synth.WORKLOADS["c5"], name="tr_small_counts", T=100, d=64, E=16, n=64, K=2, m_tile=64),
    synth.scaled(synth.WORKLOADS["c2_cap"], name="cap_one_token", T=1, d=64, E=8, n=64, K=2),
    synth.scaled(base, name="e1024", T=2048, d=64, E=1024, n=64, K=8),
    synth.scaled(base, name="t65536", T=65536, d=64, E=8, n=64, K=1),
    synth.scaled(synth.WORKLOADS["c5"], name="t32768_tr", T=32768, d=64, E=32, n=64, K=2, m_tile=128),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_edge_case_layer(ctx, wl):
    inp = Inputs(wl)
    buf = run_path(ctx, inp, backward=True, dW_dtype=torch.float32)
    g = gpu_routing(buf)
    if wl.capacity_factor:
        import oracle
        from oracle import moe_oracle as mo
        C = mo.expert_capacity(wl.T, wl.E, wl.K, wl.capacity_factor)
        O_ref, cache = mo.moe_forward(inp.X, inp.W_r, inp.bias, inp.W_gate, inp.W_up, inp.W_down, wl.K,
                                      logits_for_routing=g["logits"], capacity=C, policy=wl.drop_policy,
                                      drop_keys=g["topk_w"])
        oracle.compare("O", buf.O.float().cpu().numpy().astype(np.float64), O_ref)
        return
    check_routing_bit_exact(g, wl.K, wl.m_tile)
    O_ref, cache, grads = oracle_layer(inp, g)
    # e1024: about 16 rows per expert, where a single bf16 rounding of the weight-gradient operands would cost
    # up to 2.8e-2 on dW_down; the two-part operands keep every tensor within the bound of the exact gradient
    rep = compare_layer(buf, inp, O_ref, cache, grads)
    if wl.m_tile:
        assert np.all(g["counts"] % wl.m_tile == 0)
    print(wl.name, "P", g["P"], {k: (round(v["max"], 5), round(v["mean"], 6)) for k, v in rep.items()})


def test_nan_poisoned_buffers_token_rounding(ctx):
    """Every float buffer and the workspace start as NaN bit patterns.  Token rounding leaves rows past the
    last pair in the pair-indexed buffers (P < cap), which the GEMMs load with their last tiles and stages;
    neither those rows nor any scratch may reach an output."""
    import varlen_grouped_gemm_gb300 as vgg
    wl = synth.scaled(synth.WORKLOADS["c5"], name="tr_poisoned", T=600, d=320, E=16, n=192, K=4, m_tile=64)
    inp = Inputs(wl)
    dv = inp.dev
    buf = vgg.Buffers.allocate(wl.T, wl.d, wl.E, wl.n, wl.K, wl.m_tile, backward=True, dW_dtype=torch.float32)
    for name in ("logits", "scores", "topk_w", "sorted_w", "H", "U", "A", "Yw", "O", "dX", "dW_gate", "dW_up",
                 "dW_down", "dS", "dlogits", "dW_r", "ws"):
        t = getattr(buf, name)
        if t is not None:
            t.view(torch.uint8).fill_(0xFF)
    vgg.forward(ctx, dv["X"], dv["W_r"], dv["bias"], dv["W_gate"], dv["W_up"], dv["W_down"], buf)
    vgg.backward(ctx, dv["dO"], dv["X"], dv["W_r"], dv["W_gate"], dv["W_up"], dv["W_down"], buf)
    rc, code = vgg.moe_get_error(ctx)
    assert rc == vgg.MOE_OK and code == 0, (rc, code)
    g = gpu_routing(buf)
    assert g["P"] + 16 <= buf.sorted_tok.numel(), "the case must leave rows past the last pair"
    check_routing_bit_exact(g, wl.K, wl.m_tile)
    O_ref, cache, grads = oracle_layer(inp, g)
    compare_layer(buf, inp, O_ref, cache, grads)
