"""Shared helpers for the GPU tests: synthetic inputs on the device, the whole path, and oracle runs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
from oracle import moe_oracle as mo


def bits_to_dev(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bits (host) -> bf16 tensor on the device."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


class Inputs:
    """Host bits (for the oracle) and device tensors (for the CUDA path) of one workload."""

    def __init__(self, wl: synth.Workload, with_grad: bool = True):
        self.wl = wl
        self.X = synth.make_x(wl)
        self.W_r = synth.make_router(wl)
        self.bias = synth.make_bias(wl)
        self.W_gate = synth.make_w_gate(wl)
        self.W_up = synth.make_w_up(wl)
        self.W_down = synth.make_w_down(wl)
        self.dO = synth.make_dout(wl) if with_grad else None
        self.dev = dict(
            X=bits_to_dev(self.X), W_r=bits_to_dev(self.W_r),
            bias=None if self.bias is None else torch.from_numpy(self.bias).cuda(),
            W_gate=bits_to_dev(self.W_gate), W_up=bits_to_dev(self.W_up), W_down=bits_to_dev(self.W_down),
            dO=None if self.dO is None else bits_to_dev(self.dO))


def run_path(ctx, inp: Inputs, backward=True, dW_dtype=torch.float32):
    import varlen_grouped_gemm_gb300 as vgg
    wl, dv = inp.wl, inp.dev
    buf = vgg.Buffers.allocate(wl.T, wl.d, wl.E, wl.n, wl.K, wl.m_tile, backward=backward, dW_dtype=dW_dtype,
                               capacity_factor=wl.capacity_factor, drop_policy=wl.drop_policy)
    vgg.forward(ctx, dv["X"], dv["W_r"], dv["bias"], dv["W_gate"], dv["W_up"], dv["W_down"], buf)
    if backward:
        vgg.backward(ctx, dv["dO"], dv["X"], dv["W_r"], dv["W_gate"], dv["W_up"], dv["W_down"], buf)
    rc, code = vgg.moe_get_error(ctx)
    assert rc == vgg.MOE_OK and code == 0, (rc, code)
    return buf


def gpu_routing(buf):
    """The device's discrete routing state as host arrays, trimmed to P pairs."""
    P = int(buf.P.item())
    return dict(
        P=P, topk_ids=buf.topk_ids.cpu().numpy(), topk_w=buf.topk_w.cpu().numpy(),
        counts=buf.counts.cpu().numpy(), offsets=buf.offsets.cpu().numpy(),
        sorted_tok=buf.sorted_tok[:P].cpu().numpy(), sorted_w=buf.sorted_w[:P].cpu().numpy(),
        tok_ptr=buf.tok_ptr.cpu().numpy(), tok_pairs=buf.tok_pairs[:P].cpu().numpy(),
        logits=buf.logits.cpu().numpy(), scores=None if buf.scores is None else buf.scores.cpu().numpy())


def check_routing_bit_exact(g, K, m_tile):
    """Contract (i): the oracle's discrete stage on the device's own fp32 logits/scores reproduces
    every index array bit for bit.  Returns the oracle Routing."""
    r = mo.route_discrete(g["logits"], K, m_tile, scores=g["scores"])
    np.testing.assert_array_equal(g["topk_ids"], r.topk_ids)
    np.testing.assert_array_equal(g["counts"], r.counts)
    np.testing.assert_array_equal(g["offsets"], r.offsets)
    assert g["P"] == r.P
    np.testing.assert_array_equal(g["sorted_tok"], r.sorted_tok)
    np.testing.assert_array_equal(g["tok_ptr"], r.tok_ptr)
    np.testing.assert_array_equal(g["tok_pairs"], r.tok_pairs)
    return r


def oracle_layer(inp: Inputs, g=None, backward=True):
    """fp64 oracle forward (+ backward) with the selection taken from the device's fp32 logits/scores
    when ``g`` is given (so that routing decisions coincide), else from the oracle's own logits."""
    wl = inp.wl
    O, cache = mo.moe_forward(inp.X, inp.W_r, inp.bias, inp.W_gate, inp.W_up, inp.W_down, wl.K, wl.m_tile,
                              logits_for_routing=None if g is None else g["logits"],
                              scores_for_routing=None if g is None else g["scores"])
    grads = mo.moe_backward(inp.X, inp.W_r, inp.bias, inp.W_gate, inp.W_up, inp.W_down, inp.dO, cache) \
        if backward else None
    return O, cache, grads


def compare_layer(buf, inp: Inputs, O_ref, cache, grads, report=None, skip=()):
    """Element-wise comparison of every float output with the fp64 oracle (max/mean metric, both floors).
    Tensors named in ``skip`` are left to the caller (a variant with its own tolerance)."""
    rep = {} if report is None else report
    rep["O"] = oracle.compare("O", dev_to_f64(buf.O), O_ref)
    if grads is None:
        return rep
    r: mo.Routing = cache["routing"]
    E = inp.wl.E
    if "dX" not in skip:
        rep["dX"] = oracle.compare("dX", dev_to_f64(buf.dX), grads["dX"])
    for name, key in (("dW_gate", "dW_gate"), ("dW_up", "dW_up"), ("dW_down", "dW_down")):
        got = dev_to_f64(getattr(buf, name))
        if name not in skip:
            ref = np.stack([grads[key][e] for e in range(E)])
            rep[name] = oracle.compare(name, got, ref, param_axes=oracle.WEIGHT_GRAD)
        empty = np.nonzero(r.counts == 0)[0]
        assert not np.any(got[empty]), f"{name}: experts without pairs must get exactly zero"
    dS_ref = grads["dw"][r.sorted_tok, r.sorted_exp]
    rep["dS"] = oracle.compare("dS", dev_to_f64(buf.dS)[:r.P], dS_ref)
    rep["dlogits"] = oracle.compare("dlogits", dev_to_f64(buf.dlogits), grads["dlogits"])
    rep["dW_r"] = oracle.compare("dW_r", dev_to_f64(buf.dW_r), grads["dW_r"])
    return rep


def check_dw_single_bf16(buf, blocks, X64, dO64, r, w_full):
    """Weight gradients of the e4m3 and block-scaled backward, whose operands dH, dU and A' = w A the device rounds
    once to bf16 from its fp32 values (X and dO are bf16 inputs): every element within that rounding's bound of
    the oracle's gradient of the same variant,

        |dev - sum_t a_t b_t| <= 2^-8 sum_t |a_t| |b_t| + 2^-16 max_t |a_t| sum_t |b_t|

    (half a bf16 ulp is 2^-9 of a value; the rest covers the fp32 arithmetic before the rounding and the fp32
    accumulation), with (a, b) = (dH, X), (dU, X) and (A', dO) per expert, and normwise within 2^-7 of the
    product per expert.  ``blocks[e]`` holds the oracle's exact dh, du, a of expert e.  Experts without pairs
    must get exact zeros.  Returns the worst error over its bound."""
    worst = 0.0
    got = {k: dev_to_f64(getattr(buf, k)) for k in ("dW_gate", "dW_up", "dW_down")}
    E = len(r.counts)
    for e in range(E):
        lo, hi = r.offsets[e], r.offsets[e + 1]
        if hi == lo:
            for k in got:
                assert not np.any(got[k][e]), f"{k}: an expert without pairs must get exactly zero"
            continue
        toks = r.sorted_tok[lo:hi]
        dh, du, a = blocks[e]
        ap = w_full[toks, e][:, None] * a
        for k, A, B in (("dW_gate", dh, X64[toks]), ("dW_up", du, X64[toks]), ("dW_down", dO64[toks], ap)):
            if k == "dW_down":  # dW_down[e] = dO^T A': the rounded operand is the second one
                ref = A.T @ B
                bound = 2.0 ** -8 * (np.abs(A).T @ np.abs(B)) + 2.0 ** -16 * np.outer(np.abs(A).sum(0), np.abs(B).max(0))
            else:
                ref = A.T @ B
                bound = 2.0 ** -8 * (np.abs(A).T @ np.abs(B)) + 2.0 ** -16 * np.outer(np.abs(A).max(0), np.abs(B).sum(0))
            err = np.abs(got[k][e] - ref)
            assert np.all(err <= bound + 1e-30), (k, e, float(np.max(err / (bound + 1e-30))))
            worst = max(worst, float(np.max(err / (bound + 1e-30))))
            # independent roundings leave about 2^-9 / sqrt(3) of the product's norm; a dropped or doubled token
            # would leave about 1 / sqrt(rows)
            assert np.linalg.norm(err) <= 2.0 ** -7 * np.linalg.norm(ref) + 1e-30, (k, e, "normwise")
    return worst


def check_rounding_near_ties(g, L64, r: mo.Routing, eps=8 * 2.0 ** -24):
    """Token Rounding on exact logits, against the oracle's own selection ``r``.

    Token Rounding compares the scores of different tokens: two tokens whose exact scores lie within the
    fp32 evaluation error of each other may be taken in either order, so the selection is unique only
    where the scores are separated.  Every token on which the device and the oracle disagree must sit on
    the expert's selection threshold within ``eps`` (a few fp32 ulps of a score in (0, 1]), and the
    device's own choice must be a valid rounding under the exact scores up to ``eps``: kept routed tokens
    outrank dropped ones, padded tokens outrank the unpadded.  The device's sorted order must be that of
    its own selection.  Returns the number of pairs taken differently (at most 1% of the pairs)."""
    T, E = L64.shape
    s64 = mo.softmax(L64)
    dev_member = np.zeros((T, E), dtype=bool)
    dev_member[g["sorted_tok"], np.repeat(np.arange(E), np.diff(g["offsets"]))] = True
    routed = np.zeros((T, E), dtype=bool)
    routed[np.arange(T)[:, None], r.topk_ids] = True
    n_diff = 0
    for e in range(E):
        col, dm, om, ro = s64[:, e], dev_member[:, e], r.member[:, e], routed[:, e]
        if (ro & dm).any() and (ro & ~dm).any():
            assert col[ro & dm].min() >= col[ro & ~dm].max() - eps, f"expert {e}: drop order"
        if (~ro & dm).any() and (~ro & ~dm).any():
            assert col[~ro & dm].min() >= col[~ro & ~dm].max() - eps, f"expert {e}: padding order"
        diff = dm != om
        n_diff += int(diff.sum())
        if diff.any():
            # a dropping expert selects among its routed tokens, a padding one among the others
            pool = ro if r.counts[e] < ro.sum() else ~ro
            assert np.all(pool[diff]), f"expert {e}: a disagreement outside the pool it selects from"
            threshold = col[om & pool].min()  # the oracle's last taken score
            assert np.all(np.abs(col[diff] - threshold) <= eps), (e, col[diff], threshold)
    tt, ee = np.nonzero(dev_member)
    order = np.lexsort((tt, ee))
    np.testing.assert_array_equal(g["sorted_tok"], tt[order])
    assert n_diff <= 0.01 * r.P, n_diff
    return n_diff
