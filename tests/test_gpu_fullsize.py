"""The whole layer at the benchmark's full sizes, in the configuration the benchmark times
(bf16 weight gradients, the whole path launched through the C ABI), against the fp64 oracle.

The oracle cannot run a full layer at these sizes in seconds, so the float outputs are checked on
sampled outputs it computes one by one, and the rest through properties that hold at any size:

* routing: every index array (top-K, counts, offsets, sorted order, per-token return map) bit for
  bit against the oracle's discrete stage on the device's own fp32 logits (and scores under token
  rounding), for all T tokens;
* per token (a row of O, dX, dlogits and its pairs' dS): every expert's contribution depends only
  on that token's row of X and dO, so the oracle evaluates exactly those rows, with the experts'
  weights regenerated from the seeded generator; sampled tokens are the first and last token, two
  tokens of the heaviest expert and 16 random ones;
* dW of whole experts: the heaviest and the lightest non-empty expert, all of their rows;
* whole columns of dW_r = X^T dlogits (the lightest non-empty expert's and a random one), from the
  oracle's own dlogits of every token that has a nonzero entry in the column;
* experts that receive no pair get exactly zero weight gradients.

Tolerance: the one the small parity tests use (max relative error <= 2e-2, mean <= 3e-3, under both the
row floor and the tensor-wide floor of the compared set).
The complete element-by-element comparison at c2 is in test_gpu_full_c2.py.
"""
import gc

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import moe_oracle as mo

from _helpers import bits_to_dev, check_routing_bit_exact, dev_to_f64, gpu_routing

pytestmark = pytest.mark.gpu

CONFIGS = ["c2", "c3", "c4", "c5", "c5_plain"]


@pytest.fixture(scope="module")
def ctx():
    import varlen_grouped_gemm_gb300 as vgg
    return vgg.Context(0)


def _run_full(ctx, wl):
    """The whole path at full size; returns (buffers, the device inputs)."""
    import varlen_grouped_gemm_gb300 as vgg
    dev = {}
    for name, make in (("X", synth.make_x), ("dO", synth.make_dout), ("W_r", synth.make_router),
                       ("W_gate", synth.make_w_gate), ("W_up", synth.make_w_up), ("W_down", synth.make_w_down)):
        dev[name] = bits_to_dev(make(wl))
        gc.collect()
    bias = synth.make_bias(wl)
    dev["bias"] = None if bias is None else torch.from_numpy(bias).cuda()
    buf = vgg.Buffers.allocate(wl.T, wl.d, wl.E, wl.n, wl.K, wl.m_tile, backward=True, dW_dtype=torch.bfloat16)
    vgg.forward_backward(ctx, dev["X"], dev["W_r"], dev["bias"], dev["W_gate"], dev["W_up"], dev["W_down"],
                         dev["dO"], buf)
    rc, code = vgg.moe_get_error(ctx)
    assert rc == vgg.MOE_OK and code == 0, (rc, code)
    return buf, dev


def _token_oracle(wl, r: mo.Routing, toks, W_r_bits, bias):
    """fp64 O, dX, dlogits and per-pair dS of the given tokens, from their rows alone."""
    X = synth.make_x(wl, rows=toks)
    dO = synth.make_dout(wl, rows=toks)
    L = mo.router_logits(X, W_r_bits, bias)
    topk = r.topk_ids[toks]
    w = mo.combine_weights(L, topk)
    member = r.member[toks]
    S, d = len(toks), wl.d
    O = np.zeros((S, d))
    dX = np.zeros((S, d))
    dw = np.zeros((S, wl.E))
    experts = sorted(set(np.nonzero(member)[1].tolist()))
    for e in experts:
        rows = np.nonzero(member[:, e])[0]
        Wg, Wu, Wd = synth.make_w_gate(wl, [e])[0], synth.make_w_up(wl, [e])[0], synth.make_w_down(wl, [e])[0]
        g = mo.expert_block_backward(X[rows], dO[rows], w[rows, e], Wg, Wu, Wd)
        O[rows] += w[rows, e][:, None] * g["y"]
        dX[rows] += g["dx"]
        dw[rows, e] = g["dw"]
    dL = mo.router_grad_rows(member, topk, w, dw)
    dX += dL @ mo.bf16_bits_to_f64(W_r_bits).T
    return O, dX, dL, dw


def _expert_dw_oracle(wl, r: mo.Routing, e, W_r_bits, bias):
    """fp64 dW_gate, dW_up, dW_down of expert e over all of its rows."""
    rows = r.rows_of(e)
    X = synth.make_x(wl, rows=rows)
    dO = synth.make_dout(wl, rows=rows)
    L = mo.router_logits(X, W_r_bits, bias)
    w = mo.combine_weights(L, r.topk_ids[rows])[:, e]
    g = mo.expert_block_backward(X, dO, w, synth.make_w_gate(wl, [e])[0], synth.make_w_up(wl, [e])[0],
                                 synth.make_w_down(wl, [e])[0])
    return g["dWg"], g["dWu"], g["dWd"]


@pytest.mark.parametrize("name", CONFIGS)
def test_fullsize_parity(ctx, name):
    wl = synth.WORKLOADS[name]
    buf, dev = _run_full(ctx, wl)
    try:
        g = gpu_routing(buf)
        r = check_routing_bit_exact(g, wl.K, wl.m_tile)
        assert int(r.counts.sum()) == r.P
        if wl.m_tile:
            assert np.all(r.counts % wl.m_tile == 0), "token rounding: counts are multiples of M_tile"
        else:
            assert r.P == wl.T * wl.K
        if wl.bias == "zipf":
            mean = wl.T * wl.K / wl.E
            assert (r.counts == 0).any() and r.counts.max() > 10 * mean, "the skewed prior: empty and >10x experts"

        W_r_bits = synth.make_router(wl)
        bias = synth.make_bias(wl)
        rng = np.random.default_rng(1234)
        heavy = int(np.argmax(r.counts))
        lightest = int(np.argmin(np.where(r.counts > 0, r.counts, np.iinfo(np.int64).max)))
        hrows = r.rows_of(heavy)
        toks = np.unique(np.concatenate([[0, wl.T - 1], hrows[[0, len(hrows) - 1]],
                                         rng.choice(wl.T, 16, replace=False)])).astype(np.int64)
        O_ref, dX_ref, dL_ref, dw_ref = _token_oracle(wl, r, toks, W_r_bits, bias)
        tsel = torch.from_numpy(toks).cuda()
        rep = {}
        rep["O"] = oracle.compare("O (sampled tokens)", dev_to_f64(buf.O[tsel]), O_ref)
        rep["dX"] = oracle.compare("dX (sampled tokens)", dev_to_f64(buf.dX[tsel]), dX_ref)
        rep["dlogits"] = oracle.compare("dlogits (sampled tokens)", dev_to_f64(buf.dlogits[tsel]), dL_ref)
        # dS of every pair of the sampled tokens, at its sorted position
        dS = buf.dS.cpu().numpy().astype(np.float64)
        got, ref = [], []
        for i, t in enumerate(toks):
            for j in r.tok_pairs[r.tok_ptr[t]:r.tok_ptr[t + 1]]:
                got.append(dS[j])
                ref.append(dw_ref[i, r.sorted_exp[j]])
        rep["dS"] = oracle.compare("dS (sampled pairs)", np.array(got)[None, :], np.array(ref)[None, :])

        # whole columns of dW_r = X^T dlogits, from the oracle's own dlogits of every token whose row of dlogits
        # is nonzero in that column (the tokens routed to the expert or holding it in their top-K): the
        # lightest non-empty expert and one drawn at random
        routed = np.zeros((wl.T, wl.E), dtype=bool)
        routed[np.arange(wl.T)[:, None], r.topk_ids] = True
        cols = sorted({lightest, int(rng.integers(wl.E))})
        ref_cols = []
        for e in cols:
            tk = np.nonzero(r.member[:, e] | routed[:, e])[0].astype(np.int64)
            if len(tk) == 0:
                ref_cols.append(np.zeros(wl.d))
                continue
            _, _, dL_e, _ = _token_oracle(wl, r, tk, W_r_bits, bias)
            ref_cols.append(mo.bf16_bits_to_f64(synth.make_x(wl, rows=tk)).T @ dL_e[:, e])
        got_cols = dev_to_f64(buf.dW_r[:, torch.tensor(cols, device="cuda")]).T
        rep["dW_r"] = oracle.compare(f"dW_r columns {cols}", got_cols, np.stack(ref_cols))

        for e in sorted({heavy, lightest}):
            dWg, dWu, dWd = _expert_dw_oracle(wl, r, e, W_r_bits, bias)
            for nm, got_e, ref_e in (("dW_gate", buf.dW_gate[e], dWg), ("dW_up", buf.dW_up[e], dWu),
                                     ("dW_down", buf.dW_down[e], dWd)):
                rep[f"{nm}[{e}]"] = oracle.compare(f"{nm}[{e}]", dev_to_f64(got_e), ref_e,
                                                   param_axes=oracle.WEIGHT_GRAD)

        empty = np.nonzero(r.counts == 0)[0]
        if len(empty):
            esel = torch.from_numpy(empty).cuda()
            for nm in ("dW_gate", "dW_up", "dW_down"):
                assert not torch.any(getattr(buf, nm)[esel] != 0).item(), f"{nm}: empty experts must be zero"
        print(name, "P", r.P, "max rows", int(r.counts.max()), "empty", len(empty), "sampled", len(toks),
              {k: (float(f"{v['max']:.2e}"), float(f"{v['mean']:.2e}")) for k, v in rep.items()})
    finally:
        del buf, dev
        gc.collect()
        torch.cuda.empty_cache()
