"""The capacity (drop/pad) dispatch variant on the device vs the fp64 oracle.

[DEP] "Drop/Padding 방식": the pairs are laid out as [E, C] slots; an expert keeps at most C of its routed
tokens ("position": the first C in token order, "probs": the C with the largest routing probability) and is
padded to C.  Checked: the kept sets, counts, slot layout and per-token return map bit for bit against the
oracle's discrete stage on the device's own fp32 logits and probabilities; then every float output of the
layer, forward and backward, within the usual tolerance.  Capacity factors below, at and above the mean
load (dropping many pairs, some, none).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import moe_oracle as mo

from _helpers import Inputs, dev_to_f64, run_path

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import varlen_grouped_gemm_gb300 as vgg
    return vgg.Context(0)


def _check_slots(buf, wl, r, C):
    """Device [E, C] slot layout against the oracle's grouping of the kept pairs."""
    E = wl.E
    st = buf.sorted_tok.cpu().numpy()
    sw = buf.sorted_w.cpu().numpy()
    np.testing.assert_array_equal(buf.counts.cpu().numpy(), r.counts)
    np.testing.assert_array_equal(buf.offsets.cpu().numpy(), np.arange(E + 1) * C)
    assert int(buf.P.item()) == E * C
    for e in range(E):
        k = int(r.counts[e])
        np.testing.assert_array_equal(st[e * C:e * C + k], r.rows_of(e))
        assert np.all(st[e * C + k:(e + 1) * C] == -1) and np.all(sw[e * C + k:(e + 1) * C] == 0)
    np.testing.assert_array_equal(buf.tok_ptr.cpu().numpy(), r.tok_ptr)
    slot_of = np.concatenate([e * C + np.arange(r.counts[e]) for e in range(E)]).astype(np.int64)
    np.testing.assert_array_equal(buf.tok_pairs[:r.P].cpu().numpy(), slot_of[r.tok_pairs])
    return slot_of


CASES = [
    synth.scaled(synth.WORKLOADS["c2_cap"], name="cap_f05", T=512, d=256, E=16, n=192, K=4, capacity_factor=0.5),
    synth.scaled(synth.WORKLOADS["c2_cap"], name="cap_f1", T=512, d=256, E=16, n=192, K=4),
    synth.scaled(synth.WORKLOADS["c2_cap_probs"], name="cap_f1_probs", T=512, d=256, E=16, n=192, K=4),
    synth.scaled(synth.WORKLOADS["c2_cap_probs"], name="cap_f05_probs_bias", T=768, d=192, E=32, n=128, K=4,
                 capacity_factor=0.5, bias="normal"),
    synth.scaled(synth.WORKLOADS["c2_cap"], name="cap_f2", T=256, d=128, E=8, n=128, K=2, capacity_factor=2.0),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_capacity_layer_matches_oracle(ctx, wl):
    inp = Inputs(wl)
    buf = run_path(ctx, inp, backward=True, dW_dtype=torch.float32)
    C = mo.expert_capacity(wl.T, wl.E, wl.K, wl.capacity_factor)
    assert buf.capacity == C
    L = buf.logits.cpu().numpy()
    w_dev = buf.topk_w.cpu().numpy()
    O_ref, cache = mo.moe_forward(inp.X, inp.W_r, inp.bias, inp.W_gate, inp.W_up, inp.W_down, wl.K,
                                  logits_for_routing=L, capacity=C, policy=wl.drop_policy, drop_keys=w_dev)
    r = cache["routing"]
    np.testing.assert_array_equal(buf.topk_ids.cpu().numpy(), r.topk_ids)
    slot_of = _check_slots(buf, wl, r, C)
    c = np.bincount(r.topk_ids.reshape(-1), minlength=wl.E)
    if wl.capacity_factor < 1:
        assert r.P < wl.T * wl.K, "capacity below the mean load drops pairs"
    if wl.capacity_factor >= 2:
        assert r.P == wl.T * wl.K and (c < C).any(), "a large capacity keeps every pair and pads"
    g = mo.moe_backward(inp.X, inp.W_r, inp.bias, inp.W_gate, inp.W_up, inp.W_down, inp.dO, cache)
    oracle.compare("O", dev_to_f64(buf.O), O_ref)
    oracle.compare("dX", dev_to_f64(buf.dX), g["dX"])
    for name, key in (("dW_gate", "dW_gate"), ("dW_up", "dW_up"), ("dW_down", "dW_down")):
        got = dev_to_f64(getattr(buf, name))
        ref = np.stack([g[key][e] for e in range(wl.E)])
        oracle.compare(name, got, ref, param_axes=oracle.WEIGHT_GRAD)
    dS = dev_to_f64(buf.dS)
    oracle.compare("dS", dS[slot_of], g["dw"][r.sorted_tok, r.sorted_exp])
    oracle.compare("dlogits", dev_to_f64(buf.dlogits), g["dlogits"])
    oracle.compare("dW_r", dev_to_f64(buf.dW_r), g["dW_r"])
