"""Every element of every output at the full c2 size (T=4096, d=2048, E=128, n=512, K=8), against the
complete fp64 oracle (forward and backward over all 128 experts, a few seconds on the host's cores).

The path runs as the benchmark times it (route, permute, grouped GEMMs, combine and the whole backward
through the C ABI, bf16 weight gradients).  Routing: every index array bit for bit against the oracle's
discrete stage on the device's fp32 logits (contract (i)); the float outputs O, dX, dS, dlogits, dW_r and
dW_gate, dW_up, dW_down of all experts element by element, max relative error <= 2e-2 and mean <= 3e-3
under both the row floor and the tensor-wide floor.
"""
import gc

import numpy as np
import pytest
import torch

import synth

from _helpers import Inputs, check_routing_bit_exact, compare_layer, gpu_routing, oracle_layer

pytestmark = pytest.mark.gpu


def test_c2_every_element():
    import varlen_grouped_gemm_gb300 as vgg
    ctx = vgg.Context(0)
    wl = synth.WORKLOADS["c2"]
    inp = Inputs(wl)
    dv = inp.dev
    buf = vgg.Buffers.allocate(wl.T, wl.d, wl.E, wl.n, wl.K, wl.m_tile, backward=True, dW_dtype=torch.bfloat16)
    vgg.forward_backward(ctx, dv["X"], dv["W_r"], dv["bias"], dv["W_gate"], dv["W_up"], dv["W_down"], dv["dO"], buf)
    rc, code = vgg.moe_get_error(ctx)
    assert rc == vgg.MOE_OK and code == 0, (rc, code)
    try:
        g = gpu_routing(buf)
        check_routing_bit_exact(g, wl.K, wl.m_tile)
        O_ref, cache, grads = oracle_layer(inp, g)
        rep = compare_layer(buf, inp, O_ref, cache, grads)
        print("c2 every element", {k: (float(f"{v['max']:.2e}"), float(f"{v['mean']:.2e}"),
                                      float(f"{v['max_global']:.2e}")) for k, v in rep.items()})
    finally:
        del buf
        gc.collect()
        torch.cuda.empty_cache()
