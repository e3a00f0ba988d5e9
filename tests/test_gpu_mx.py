"""The block-scaled (1 x 32) e4m3 forward on the device vs the oracle's block-scaled forward.

[GG] "한계": a fine-grained FP8 grouped GEMM as the next step after bf16; the recipe (blocks of 32 along the
reduction dimension, power-of-two scales, e the smallest exponent with max|block| <= 448 2^e, codes rounded
to nearest even) is the library's reading.  Checked: the quantized operands (codes and block scales of X, of
W_gate / W_up and of W_down, every scale layout unpacked here) bit for bit against the oracle's quantization
of the same bf16 inputs; the routing bit for bit; H and U per sorted pair within the usual tolerance of the
oracle's fp64 products of the same codes; the activation codes A, which the gate/up epilogue quantizes from
its fp32 SwiGLU values, against the oracle's quantization of its exact values (equal but for values within
fp32 rounding of a rounding boundary: at most one code step, at most a few per hundred thousand); O within
the usual tolerance of the oracle's fp64 forward.  Cases: ragged tails, n and d with a half last stage of
128 codes, empty experts (skewed prior), token rounding, 512 experts, the capacity dispatch with empty slots.
The backward: both activation-gradient GEMMs block-scaled, and the weight gradients either two-part bf16 (the
usual tolerance) or block-scaled along tokens (the element-wise bound derived from the arithmetic: the oracle's
block-scaled product within fp32 accumulation, plus one code step where a device operand value may round
differently).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import moe_oracle as mo

from _helpers import Inputs, bits_to_dev, check_dw_single_bf16, check_routing_bit_exact, dev_to_f64, gpu_routing

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import varlen_grouped_gemm_gb300 as vgg
    return vgg.Context(0)


def _bf16_bits(M: np.ndarray) -> np.ndarray:
    return torch.from_numpy(M).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _block_off(r, b):
    """Byte of operand row r (0..127 within its block row) and 32-column block b (0..3 within its stage)."""
    return (r % 32) * 16 + (r // 32) * 4 + b


TILE = 192  # the gate/up pair's tile: 96 + 96 rows of W_gate and W_up


def _tile_cols(N: int) -> int:
    """The plain block-scaled GEMMs' tile width for N output columns, as the header states it: 192, or 128
    when 192-row tiles would pass N by more than N / 4 and 128-row tiles by less."""
    w192, w128 = -(-N // 192) * 192 - N, -(-N // 128) * 128 - N
    return 128 if (4 * w192 > N and w128 < w192) else 192


def _weight_index(E: int, R: int, C: int, rows_per_tile: int, row0: int, tile_rows: int = TILE) -> np.ndarray:
    """Byte index [E, R, C/32] of each (row, 32-column block) scale of one weight in its scale buffer:
    [E][tiles][ceil(C/128)] groups of ceil(tile_rows / 128) 512-byte blocks, tile row i = row0 + row % rows_per_tile
    in block i // 128."""
    kst = -(-C // 128)
    nblk = -(-tile_rows // 128)
    tiles = -(-R // rows_per_tile)
    rows = np.arange(R)[:, None]
    cols = np.arange(C // 32)[None, :]
    t, tr = rows // rows_per_tile, row0 + rows % rows_per_tile
    off = ((t * kst + cols // 4) * nblk + tr // 128) * 512 + _block_off(tr % 128, cols % 4)
    return np.arange(E)[:, None, None] * (tiles * kst * nblk * 512) + off[None]


def _unpack_weight_blocks(sf: np.ndarray, E: int, R: int, C: int, rows_per_tile: int, row0: int) -> np.ndarray:
    """Exponents [E, R, C/32] of one weight from its scale buffer."""
    return sf[_weight_index(E, R, C, rows_per_tile, row0)].astype(np.int64) - 127


def _unpack_act_blocks(sf: np.ndarray, offsets: np.ndarray, n: int, rows: np.ndarray) -> np.ndarray:
    """Exponents [len(rows), n/32] of the activation rows (sorted positions) from the per-row-tile blocks."""
    kst = -(-n // 128)
    E = len(offsets) - 1
    tiles_before = np.concatenate([[0], np.cumsum(-(-np.diff(offsets) // 128))])
    e = np.searchsorted(offsets, rows, side="right") - 1
    r = rows - offsets[e]
    rt = tiles_before[e] + r // 128
    cols = np.arange(n // 32)
    idx = (rt[:, None] * kst + cols[None, :] // 4) * 512 + _block_off(r[:, None] % 128, cols[None, :] % 4)
    assert e.max() < E
    return sf[idx].astype(np.int64) - 127


def test_mx_quantize_rows_bit_exact(ctx):
    import varlen_grouped_gemm_gb300 as vgg
    rng = np.random.default_rng(31)
    for rows, cols in ((300, 320), (64, 2048)):
        # row and block magnitudes over many binades (subnormal codes, the clamped exponent), zero blocks
        M = rng.standard_normal((rows, cols)) * np.exp2(rng.uniform(-60, 60, (rows, cols // 32))).repeat(32, axis=1)
        M[3] = 0.0
        M[4, 32:64] = 0.0
        M[5, :32] *= 2.0 ** -80
        bits = _bf16_bits(M)
        Md = bits_to_dev(bits)
        q = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
        sf = torch.full((rows, vgg.mx_sf_cols(cols)), 0, dtype=torch.uint8, device="cuda")
        vgg.moe_quantize_rows_mx(ctx, Md, q, sf)
        qo, eo = oracle.quantize_blocks_mx(bits)
        np.testing.assert_array_equal(q.cpu().numpy(), qo)
        got = sf.cpu().numpy().astype(np.int64)
        np.testing.assert_array_equal(got[:, :cols // 32] - 127, eo)
        assert np.all(got[:, cols // 32:] == 127), "padding entries hold scale 1"
        assert eo[3].max() == 0 and eo[4, 1] == 0


@pytest.mark.parametrize("E,d,n", [(4, 256, 192), (3, 320, 320), (2, 2048, 512)])
def test_mx_weights_bit_exact(ctx, E, d, n):
    import varlen_grouped_gemm_gb300 as vgg
    rng = np.random.default_rng(32 + d)
    Wg = _bf16_bits(rng.standard_normal((E, n, d)) * 0.05)
    Wu = _bf16_bits(rng.standard_normal((E, n, d)) * 0.05 * np.exp2(rng.integers(-8, 8, (E, n, 1))))
    Wd = _bf16_bits(rng.standard_normal((E, d, n)) * 0.05)
    w = vgg.MxWeights.quantize(ctx, bits_to_dev(Wg), bits_to_dev(Wu), bits_to_dev(Wd))
    gu = w.gu_sf.cpu().numpy()
    dn = w.dn_sf.cpu().numpy()
    bd = _tile_cols(d)
    assert gu.size == E * -(-n // (TILE // 2)) * -(-d // 128) * 1024
    assert dn.size == E * -(-d // bd) * -(-n // 128) * 512 * -(-bd // 128)
    want = {"gu": np.full_like(gu, 127), "dn": np.full_like(dn, 127)}
    for got_q, W, R, C, key, rpt, r0, tr in ((w.Wg_q, Wg, n, d, "gu", TILE // 2, 0, TILE),
                                             (w.Wu_q, Wu, n, d, "gu", TILE // 2, TILE // 2, TILE),
                                             (w.Wd_q, Wd, d, n, "dn", bd, 0, bd)):
        q, e = oracle.quantize_blocks_mx(W.reshape(E * R, C))
        np.testing.assert_array_equal(got_q.cpu().numpy().reshape(E * R, C), q)
        # the whole scale buffer, built here from the oracle's exponents: entries no weight row or column
        # fills hold scale 1 (byte 127)
        want[key][_weight_index(E, R, C, rpt, r0, tr)] = e.reshape(E, R, -1) + 127
    np.testing.assert_array_equal(gu, want["gu"])
    np.testing.assert_array_equal(dn, want["dn"])


CASES = [
    synth.scaled(synth.WORKLOADS["c2"], name="c2_small", T=512, d=256, E=16, n=192, K=4),
    synth.scaled(synth.WORKLOADS["c2"], name="c2_medium", T=1024, d=1024, E=32, n=256, K=4),
    # d = n = 320: both GEMMs end on a half stage of 128 codes; skewed prior: empty experts
    synth.scaled(synth.WORKLOADS["c4"], name="c4_small_320", T=640, d=320, E=32, n=320, K=4),
    synth.scaled(synth.WORKLOADS["c5"], name="c5_small_tr", T=2048, d=256, E=32, n=128, K=8, m_tile=64),
    synth.scaled(synth.WORKLOADS["c5_plain"], name="c5_small_e512", T=2048, d=256, E=512, n=128, K=8),
    # capacity factor 1 under a skewed load: some experts drop pairs, others leave slots empty
    synth.scaled(synth.WORKLOADS["c2_cap"], name="cap_f1_bias", T=512, d=256, E=16, n=192, K=4, bias="normal"),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_mx_forward_matches_oracle(ctx, wl):
    import varlen_grouped_gemm_gb300 as vgg
    inp = Inputs(wl, with_grad=False)
    dv = inp.dev
    E, n, d = wl.E, wl.n, wl.d
    buf = vgg.Buffers.allocate(wl.T, d, E, n, wl.K, wl.m_tile, backward=False, capacity_factor=wl.capacity_factor,
                               drop_policy=wl.drop_policy, mx=True)
    buf.masf.fill_(255)  # scale bytes the forward must write are never left at this (NaN) pattern
    wmx = vgg.MxWeights.quantize(ctx, dv["W_gate"], dv["W_up"], dv["W_down"])
    vgg.forward_mx(ctx, dv["X"], dv["W_r"], dv["bias"], wmx, buf)
    rc, code = vgg.moe_get_error(ctx)
    assert rc == vgg.MOE_OK and code == 0, (rc, code)

    xq, xe = oracle.quantize_blocks_mx(inp.X)
    np.testing.assert_array_equal(buf.mxq.cpu().numpy(), xq)
    np.testing.assert_array_equal(buf.mxsf.cpu().numpy()[:, :d // 32].astype(np.int64) - 127, xe)

    g = gpu_routing(buf)
    C = buf.capacity
    O_ref, cache = oracle.moe_forward_mx(inp.X, inp.W_r, inp.bias, inp.W_gate, inp.W_up, inp.W_down, wl.K,
                                         wl.m_tile, logits_for_routing=g["logits"], scores_for_routing=g["scores"],
                                         capacity=C, policy=wl.drop_policy, drop_keys=g["topk_w"] if C else None)
    r = cache["routing"]
    if C:
        # slots e*C + rank hold the kept pairs; the rest are empty (zero rows)
        slot_of = np.concatenate([e * C + np.arange(r.counts[e]) for e in range(E)]).astype(np.int64)
        empty = np.setdiff1d(np.arange(E * C), slot_of)
        assert r.P < wl.T * wl.K and len(empty) > 0
        assert not torch.any(buf.H[torch.from_numpy(empty).cuda()] != 0).item(), "empty slots give zero rows"
        assert not torch.any(buf.maq[torch.from_numpy(empty).cuda()] != 0).item()
        rows = slot_of
        offs = np.arange(E + 1) * C
    else:
        check_routing_bit_exact(g, wl.K, wl.m_tile)
        rows = np.arange(r.P)
        offs = r.offsets
    sel = torch.from_numpy(rows).cuda()
    rep = {"O": oracle.compare("O", dev_to_f64(buf.O), O_ref)}
    rep["H"] = oracle.compare("H", dev_to_f64(buf.H[sel]), cache["h"])
    rep["U"] = oracle.compare("U", dev_to_f64(buf.U[sel]), cache["u"])
    # A's codes and block scales: the device quantizes its fp32 SwiGLU values, the oracle the exact ones
    aq = buf.maq[sel].cpu().numpy()
    ae = _unpack_act_blocks(buf.masf.cpu().numpy(), offs, n, rows)
    diff_e = ae != cache["ae"]
    assert diff_e.sum() <= max(2, diff_e.size // 10000), ("block scales of A", int(diff_e.sum()), diff_e.size)
    same_blocks = np.repeat(~diff_e, 32, axis=1)
    dq = np.abs(mo.e4m3_decode(aq) - mo.e4m3_decode(cache["aq"]))
    step = np.maximum(np.abs(mo.e4m3_decode(cache["aq"])) * 2.0 ** -3, 2.0 ** -9)
    bad = same_blocks & (dq > 0)
    assert bad.sum() <= max(4, aq.size // 20000), ("A codes", int(bad.sum()), aq.size)
    assert np.all(dq[bad] <= step[bad] * (1 + 1e-12)), "a differing code is one step away"
    # the activation scale blocks of every row tile hold scale 1 past n
    if wl.bias == "zipf":
        assert (r.counts == 0).any(), "the skewed prior should leave some experts empty"
    print(wl.name, {k: (round(v["max"], 6), round(v["mean"], 7)) for k, v in rep.items()},
          "A codes differing:", int(bad.sum()), "of", aq.size)


def test_mx_forward_only(ctx):
    """cache=False: the same O bit for bit, H and U left untouched."""
    import varlen_grouped_gemm_gb300 as vgg
    wl = synth.scaled(synth.WORKLOADS["c2"], name="c2_small_n256", T=512, d=256, E=16, n=256, K=4)
    inp = Inputs(wl, with_grad=False)
    dv = inp.dev
    buf = vgg.Buffers.allocate(wl.T, wl.d, wl.E, wl.n, wl.K, backward=False, mx=True)
    wmx = vgg.MxWeights.quantize(ctx, dv["W_gate"], dv["W_up"], dv["W_down"])
    vgg.forward_mx(ctx, dv["X"], dv["W_r"], dv["bias"], wmx, buf)
    O_cached = buf.O.clone()
    buf.H.fill_(7.0)
    buf.U.fill_(7.0)
    buf.O.zero_()
    vgg.forward_mx(ctx, dv["X"], dv["W_r"], dv["bias"], wmx, buf, cache=False)
    assert torch.equal(buf.O, O_cached)
    assert torch.all(buf.H == 7.0).item() and torch.all(buf.U == 7.0).item()


BWD_CASES = [
    synth.scaled(synth.WORKLOADS["c2"], name="c2_small", T=512, d=256, E=16, n=192, K=4),
    # n = 320: a partial 192-column tile; d = 320: the dSwiGLU GEMM ends on a half stage; empty experts
    synth.scaled(synth.WORKLOADS["c4"], name="c4_small_320", T=640, d=320, E=32, n=320, K=4),
    synth.scaled(synth.WORKLOADS["c5"], name="c5_small_tr", T=2048, d=256, E=32, n=128, K=8, m_tile=64),
    synth.scaled(synth.WORKLOADS["c2_cap"], name="cap_f1_bias", T=512, d=256, E=16, n=192, K=4, bias="normal"),
]


def _token_block_slack(M, rel=0.0, amax_frac=0.0):
    """An expert's [rows, C] operand (exact values) quantized in blocks of 32 tokens of one column: the oracle's
    block-scaled values, and per element the slack that a device value within rel |x| + amax_frac amax of x
    (amax: the block's largest magnitude) allows in its dequantized value.  Zero where every such value gets
    the same code under the same block exponent; one code step (plus the deviation) where the code may be the
    neighbouring one; two steps of the coarser exponent where the block's exponent itself may differ by one.
    rel = amax_frac = 0 (operands the device reads as the same bf16 values): no slack."""
    A = np.asarray(M, dtype=np.float64)
    R, C = A.shape
    Rp = -(-R // 32) * 32
    pad = np.zeros((Rp, C))
    pad[:R] = A
    B = pad.T.reshape(C, Rp // 32, 32)
    amax = np.abs(B).max(axis=-1)
    e = oracle.mx_block_exponents(amax)
    sc = np.exp2(e.astype(np.float64))[..., None]
    q = oracle.e4m3_round(B / sc) * sc
    dev = rel * np.abs(B) + amax_frac * amax[..., None]
    amb = oracle.e4m3_round((B - dev) / sc) != oracle.e4m3_round((B + dev) / sc)
    da = (rel + amax_frac) * amax
    blk = (oracle.mx_block_exponents(np.maximum(amax - da, 0.0)) != e) | (oracle.mx_block_exponents(amax + da) != e)
    step = 2.0 ** -3 * (np.abs(B) + dev) + 2.0 ** -9 * sc
    slack = np.where(amb, step + dev, 0.0)
    slack = np.where(blk[..., None], 2 * step + 2.0 ** -9 * sc + dev, slack)
    back = lambda Z: Z.reshape(C, Rp).T[:R]
    return back(q), back(slack)


def _check_mx_dw(got, Aq, As, Bq, Bs, name):
    """got = sum over the expert's tokens of dq(A)^T dq(B) on the device: within fp32 accumulation of the
    oracle's product of its block-scaled operands, plus what the operands' slack (``_token_block_slack``)
    allows.  Returns the summed slack, the summed magnitude sum |dq(A)| |dq(B)| and the worst error relative to
    the bound."""
    mag = np.abs(Aq).T @ np.abs(Bq)
    ref = Aq.T @ Bq
    slack = As.T @ (np.abs(Bq) + Bs) + np.abs(Aq).T @ Bs
    bound = 2.0 ** -14 * mag + slack + 1e-30
    err = np.abs(got - ref)
    assert np.all(err <= bound), (name, float(np.max(err / bound)), float(np.max(err)))
    return float(slack.sum()), float(mag.sum()), float(np.max(err / bound))


def _act_exps(sf: torch.Tensor, offsets: np.ndarray, cols: int, rows: np.ndarray) -> np.ndarray:
    return _unpack_act_blocks(sf.cpu().numpy(), offsets, cols, rows)


@pytest.mark.parametrize("wl,dw", [(w, True) for w in BWD_CASES] + [(BWD_CASES[0], False)],
                         ids=lambda v: v.name if hasattr(v, "name") else ("mx_dw" if v else "bf16_dw"))
def test_mx_backward_matches_oracle(ctx, wl, dw):
    """moe_backward_mx against the oracle's backward with both activation-gradient GEMMs block-scaled and, with
    ``dw``, the weight gradients on operands quantized in blocks of 32 tokens of one expert (else two-part bf16):
    * the weight codes and scale blocks (W_down^T and [W_gate; W_up]^T) bit for bit, padding included;
    * the sorted dO codes and their scale blocks bit for bit (decided on the exact bf16 dO);
    * the [dH | dU] codes, which the dSwiGLU epilogue quantizes from its fp32 values, against the oracle's
      quantization of its exact values: equal but for values within fp32 rounding of a boundary (one code step,
      a few per hundred thousand; a block whose scale differs is left out);
    * dX, dS, dlogits, dW_r within the usual tolerance of the oracle's block-scaled backward, both floors;
    * the weight gradients: block-scaled, within the bound derived for them; else on operands rounded once to
      bf16, within that rounding's bound (``check_dw_single_bf16``)."""
    import varlen_grouped_gemm_gb300 as vgg
    from _helpers import compare_layer
    inp = Inputs(wl)
    dv = inp.dev
    E, n, d = wl.E, wl.n, wl.d
    buf = vgg.Buffers.allocate(wl.T, d, E, n, wl.K, wl.m_tile, backward=True, dW_dtype=torch.float32,
                               capacity_factor=wl.capacity_factor, drop_policy=wl.drop_policy, mx=True)
    buf.mhusf.fill_(255)
    buf.mdosft.fill_(255)
    wmx = vgg.MxWeights.quantize(ctx, dv["W_gate"], dv["W_up"], dv["W_down"], backward=True)
    vgg.forward(ctx, dv["X"], dv["W_r"], dv["bias"], dv["W_gate"], dv["W_up"], dv["W_down"], buf)
    vgg.backward_mx(ctx, dv["dO"], dv["X"], dv["W_r"], dv["W_gate"], dv["W_up"], dv["W_down"], wmx, buf, dw=dw)
    rc, code = vgg.moe_get_error(ctx)
    assert rc == vgg.MOE_OK and code == 0, (rc, code)

    Wg, Wu, Wd = (mo.bf16_bits_to_f64(a) for a in (inp.W_gate, inp.W_up, inp.W_down))
    Wdt = Wd.transpose(0, 2, 1)  # [E, n, d]
    Wgu = np.concatenate([Wg, Wu], axis=1).transpose(0, 2, 1)  # [E, d, 2n]
    for got_q, got_sf, W, R, C in ((wmx.Wdt_q, wmx.wdt_sf, Wdt, n, d), (wmx.Wgu_q, wmx.wgu_sf, Wgu, d, 2 * n)):
        q, e = oracle.quantize_blocks_mx(W.reshape(E * R, C))
        np.testing.assert_array_equal(got_q.cpu().numpy().reshape(E * R, C), q)
        sf = got_sf.cpu().numpy()
        want = np.full_like(sf, 127)
        want[_weight_index(E, R, C, _tile_cols(R), 0, _tile_cols(R))] = e.reshape(E, R, -1) + 127
        np.testing.assert_array_equal(sf, want)

    g = gpu_routing(buf)
    C = buf.capacity
    O_ref, cache = mo.moe_forward(inp.X, inp.W_r, inp.bias, inp.W_gate, inp.W_up, inp.W_down, wl.K, wl.m_tile,
                                  logits_for_routing=g["logits"], scores_for_routing=g["scores"], capacity=C,
                                  policy=wl.drop_policy, drop_keys=g["topk_w"] if C else None)
    grads = mo.moe_backward(inp.X, inp.W_r, inp.bias, inp.W_gate, inp.W_up, inp.W_down, inp.dO, cache,
                            mx_dx=True, mx_dact=True, mx_dw=dw)
    r = cache["routing"]
    if C:
        rows = np.concatenate([e * C + np.arange(r.counts[e]) for e in range(E)]).astype(np.int64)
        offs = np.arange(E + 1) * C
    else:
        check_routing_bit_exact(g, wl.K, wl.m_tile)
        rows = np.arange(r.P)
        offs = r.offsets
    # dO's codes at the sorted positions and their scale blocks per row tile, bit for bit
    oq, oe = oracle.quantize_blocks_mx(inp.dO[r.sorted_tok])
    np.testing.assert_array_equal(buf.mdoq.cpu().numpy()[rows], oq)
    np.testing.assert_array_equal(_act_exps(buf.mdosft, offs, d, rows), oe)
    # [dH | dU] codes against the oracle's quantization of its exact values
    X64, dO64 = mo.bf16_bits_to_f64(inp.X), mo.bf16_bits_to_f64(inp.dO)
    hu_ref = np.zeros((r.P, 2 * n))
    # block-scaled weight gradients: every element within fp32 accumulation of the oracle's block-scaled product,
    # plus the slack of operand values (dH, dU, A', which the device computes in fp32) that lie within the
    # device's deviation of a rounding boundary; X and dO are the same bf16 values on both sides (no slack)
    dw_rep = {"slack": 0.0, "magnitude": 0.0, "worst": 0.0}
    blocks = {}
    dev_dw = {k: dev_to_f64(getattr(buf, k)) for k in ("dW_gate", "dW_up", "dW_down")} if dw else None
    for e in range(E):
        lo, hi = r.offsets[e], r.offsets[e + 1]
        if hi == lo:
            continue
        toks = r.sorted_tok[lo:hi]
        q1, e1 = oracle.quantize_blocks_mx(dO64[toks])
        q2, e2 = oracle.quantize_blocks_mx(Wdt[e])
        dap = oracle.dequantize_blocks_mx(q1, e1) @ oracle.dequantize_blocks_mx(q2, e2).T
        blk = mo.expert_block_backward(X64[toks], dO64[toks], cache["w_full"][toks, e], inp.W_gate[e], inp.W_up[e],
                                       inp.W_down[e], dap=dap)
        hu_ref[lo:hi] = np.concatenate([blk["dh"], blk["du"]], axis=1)
        blocks[e] = (blk["dh"], blk["du"], blk["a"])
        if dw:
            xq, xs = _token_block_slack(X64[toks])
            oq, os_ = _token_block_slack(dO64[toks])
            ops = (("dW_gate", blk["dh"], X64), ("dW_up", blk["du"], X64))
            for name, G, _ in ops:
                gq, gs = _token_block_slack(G, 2.0 ** -14, 2.0 ** -16)
                sl, mg, worst = _check_mx_dw(dev_dw[name][e], gq, gs, xq, xs, name)
                np.testing.assert_allclose(gq.T @ xq, grads[name][e], rtol=1e-9, atol=1e-12)
                dw_rep["slack"] += sl
                dw_rep["magnitude"] += mg
                dw_rep["worst"] = max(dw_rep["worst"], worst)
            aq, as_ = _token_block_slack(cache["w_full"][toks, e][:, None] * blk["a"], 2.0 ** -14, 2.0 ** -16)
            sl, mg, worst = _check_mx_dw(dev_dw["dW_down"][e], oq, os_, aq, as_, "dW_down")
            np.testing.assert_allclose(oq.T @ aq, grads["dW_down"][e], rtol=1e-9, atol=1e-12)
            dw_rep["slack"] += sl
            dw_rep["magnitude"] += mg
            dw_rep["worst"] = max(dw_rep["worst"], worst)
    if not dw:  # single-part bf16 operands: the rounding bound
        dw_rep["worst"] = check_dw_single_bf16(buf, blocks, X64, dO64, r, cache["w_full"])
    if dw:
        # the slack is a small part of the bound: summed over all elements it stays below 1% of the summed
        # magnitudes of the products (a few operand values near a boundary, one code step each)
        assert dw_rep["slack"] <= 1e-2 * dw_rep["magnitude"], dw_rep
        for k in ("dW_gate", "dW_up", "dW_down"):
            assert not np.any(dev_dw[k][r.counts == 0]), f"{k}: experts without pairs must get exactly zero"
    hq_ref, he_ref = oracle.quantize_blocks_mx(hu_ref)
    hq = buf.mhuq.cpu().numpy()[rows]
    he = _act_exps(buf.mhusf, offs, 2 * n, rows)
    diff_e = he != he_ref
    assert diff_e.sum() <= max(2, diff_e.size // 10000), ("[dH|dU] block scales", int(diff_e.sum()), diff_e.size)
    same = np.repeat(~diff_e, 32, axis=1)
    dq = np.abs(mo.e4m3_decode(hq) - mo.e4m3_decode(hq_ref))
    step = np.maximum(np.abs(mo.e4m3_decode(hq_ref)) * 2.0 ** -3, 2.0 ** -9)
    bad = same & (dq > 0)
    assert bad.sum() <= max(4, hq.size // 20000), ("[dH|dU] codes", int(bad.sum()), hq.size)
    assert np.all(dq[bad] <= step[bad] * (1 + 1e-12))
    if C:
        rep = {"O": oracle.compare("O", dev_to_f64(buf.O), O_ref),
               "dX": oracle.compare("dX", dev_to_f64(buf.dX), grads["dX"])}

        rep["dS"] = oracle.compare("dS", dev_to_f64(buf.dS)[rows], grads["dw"][r.sorted_tok, r.sorted_exp])
        rep["dlogits"] = oracle.compare("dlogits", dev_to_f64(buf.dlogits), grads["dlogits"])
        rep["dW_r"] = oracle.compare("dW_r", dev_to_f64(buf.dW_r), grads["dW_r"])
    else:
        rep = compare_layer(buf, inp, O_ref, cache, grads, skip=("dW_gate", "dW_up", "dW_down"))
    if dw:
        print(wl.name, "block-scaled dW: slack / magnitude", dw_rep["slack"] / dw_rep["magnitude"],
              "worst error / bound", round(dw_rep["worst"], 4))
    else:
        print(wl.name, "single-part bf16 dW: worst error / bound", round(dw_rep["worst"], 4))
    print(wl.name, "mx_dw" if dw else "bf16_dw", "[dH|dU] codes differing:", int(bad.sum()), "of", hq.size,
          {k: (round(v["max"], 5), round(v["mean"], 6)) for k, v in rep.items()})


def test_mx_fullsize_c2(ctx):
    """The c2 shape at full size (the configuration the benchmark's block-scaled arm times), on sampled tokens:
    every expert contribution of a token depends only on its own row and the experts' weights.  X's codes and
    scales of the sampled tokens and the codes and scale blocks of every expert they reach bit for bit; O of the
    sampled tokens within the usual tolerance of the oracle's block-scaled forward."""
    import gc
    import varlen_grouped_gemm_gb300 as vgg
    wl = synth.WORKLOADS["c2"]
    dev = {name: bits_to_dev(make(wl)) for name, make in (
        ("X", synth.make_x), ("W_r", synth.make_router), ("W_gate", synth.make_w_gate), ("W_up", synth.make_w_up),
        ("W_down", synth.make_w_down))}
    buf = vgg.Buffers.allocate(wl.T, wl.d, wl.E, wl.n, wl.K, backward=False, mx=True)
    wmx = vgg.MxWeights.quantize(ctx, dev["W_gate"], dev["W_up"], dev["W_down"])
    vgg.forward_mx(ctx, dev["X"], dev["W_r"], None, wmx, buf)
    rc, code = vgg.moe_get_error(ctx)
    assert rc == vgg.MOE_OK and code == 0, (rc, code)
    try:
        g = gpu_routing(buf)
        r = check_routing_bit_exact(g, wl.K, 0)
        rng = np.random.default_rng(78)
        toks = np.unique(np.concatenate([[0, wl.T - 1], rng.choice(wl.T, 6, replace=False)])).astype(np.int64)
        X = synth.make_x(wl, rows=toks)
        xq, xe = oracle.quantize_blocks_mx(X)
        tsel = torch.from_numpy(toks).cuda()
        np.testing.assert_array_equal(buf.mxq[tsel].cpu().numpy(), xq)
        np.testing.assert_array_equal(buf.mxsf[tsel].cpu().numpy()[:, :wl.d // 32].astype(np.int64) - 127, xe)
        Xd = oracle.dequantize_blocks_mx(xq, xe)
        L = mo.router_logits(X, synth.make_router(wl), None)
        w = mo.combine_weights(L, r.topk_ids[toks])
        gu_sf, dn_sf = wmx.gu_sf.cpu().numpy(), wmx.dn_sf.cpu().numpy()
        O = np.zeros((len(toks), wl.d))
        member = r.member[toks]
        E, n, d = wl.E, wl.n, wl.d
        gi = _weight_index(E, n, d, TILE // 2, 0)
        ui = _weight_index(E, n, d, TILE // 2, TILE // 2)
        di = _weight_index(E, d, n, _tile_cols(d), 0, _tile_cols(d))
        for e in sorted(set(np.nonzero(member)[1].tolist())):
            rows = np.nonzero(member[:, e])[0]
            gq, ge = oracle.quantize_blocks_mx(synth.make_w_gate(wl, [e])[0])
            uq, ue = oracle.quantize_blocks_mx(synth.make_w_up(wl, [e])[0])
            dq, de = oracle.quantize_blocks_mx(synth.make_w_down(wl, [e])[0])
            np.testing.assert_array_equal(wmx.Wg_q[e].cpu().numpy(), gq)
            np.testing.assert_array_equal(wmx.Wu_q[e].cpu().numpy(), uq)
            np.testing.assert_array_equal(wmx.Wd_q[e].cpu().numpy(), dq)
            np.testing.assert_array_equal(gu_sf[gi[e]].astype(np.int64) - 127, ge)
            np.testing.assert_array_equal(gu_sf[ui[e]].astype(np.int64) - 127, ue)
            np.testing.assert_array_equal(dn_sf[di[e]].astype(np.int64) - 127, de)
            h = Xd[rows] @ oracle.dequantize_blocks_mx(gq, ge).T
            u = Xd[rows] @ oracle.dequantize_blocks_mx(uq, ue).T
            aq, ae = oracle.quantize_blocks_mx(mo.silu(h) * u)
            y = oracle.dequantize_blocks_mx(aq, ae) @ oracle.dequantize_blocks_mx(dq, de).T
            O[rows] += w[rows, e][:, None] * y
        rep = oracle.compare("O (sampled tokens)", dev_to_f64(buf.O[tsel]), O)
        print("c2 block-scaled", len(toks), "tokens", (rep["max"], rep["mean"]))
    finally:
        del buf, dev, wmx
        gc.collect()
        torch.cuda.empty_cache()
