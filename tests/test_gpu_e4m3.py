"""The e4m3 gate/up forward on the device vs the oracle's e4m3 forward.

[GG] "한계": a fine-grained FP8 grouped GEMM as the next step after bf16; the recipe (per-row scales,
s = max|row| / 448 in fp32, codes rounded to nearest even and saturated) is the library's reading.
Checked: the quantized operands (codes and scales of X and of W_gate / W_up) bit for bit against the
oracle's quantization of the same bf16 inputs; the routing bit for bit (as in the bf16 path); H, U, A
per sorted pair and O within the usual tolerance against the oracle's fp64 forward from the same
e4m3 operands (the device accumulates the code products in fp32).  Cases: ragged tails, empty experts
(skewed prior), token rounding, the capacity dispatch with empty slots, and the benchmark's c2 shape at
full size on sampled tokens.
"""
import gc

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


def test_quantize_rows_bit_exact(ctx):
    import varlen_grouped_gemm_gb300 as vgg
    rng = np.random.default_rng(21)
    rows, cols = 300, 272
    # row magnitudes over many binades, so that codes land in the subnormal range too
    M = rng.standard_normal((rows, cols)) * np.exp2(rng.uniform(-40, 20, (rows, 1)))
    M[3] = 0.0
    M[4] = 0.0
    M[4, 17] = -3.0
    M[5, ::7] *= 1e-6
    bits = _bf16_bits(M)
    for shape in ((rows, cols), (3, 100, cols)):
        b = np.concatenate([bits, bits])[:int(np.prod(shape[:-1]))].reshape(shape)
        Md = bits_to_dev(b)
        q = torch.empty(shape, dtype=torch.uint8, device="cuda")
        s = torch.empty(shape[:-1], dtype=torch.float32, device="cuda")
        vgg.moe_quantize_rows_e4m3(ctx, Md, q, s)
        qo, so = mo.quantize_rows_e4m3(b.reshape(-1, cols))
        np.testing.assert_array_equal(q.cpu().numpy().reshape(-1, cols), qo)
        np.testing.assert_array_equal(s.cpu().numpy().reshape(-1), so)
    assert so[3] == 1.0 and np.all(qo[3] == 0), "a zero row: scale 1, zero codes"


CASES = [
    synth.scaled(synth.WORKLOADS["c2"], name="c2_small", T=512, d=256, E=16, n=192, K=4),
    synth.scaled(synth.WORKLOADS["c4"], name="c4_small", T=640, d=384, E=32, n=320, K=4),
    # d = 320: the last K stage holds 64 of its 128 codes (zeros past K)
    synth.scaled(synth.WORKLOADS["c4"], name="c4_small_d320", T=640, d=320, E=32, n=320, K=4),
    synth.scaled(synth.WORKLOADS["c5"], name="c5_small_tr", T=2048, d=256, E=32, n=128, K=8, m_tile=64),
    # capacity factor 1 under a skewed load: some experts drop pairs, others leave slots empty
    synth.scaled(synth.WORKLOADS["c2_cap"], name="cap_f1_bias", T=512, d=256, E=16, n=192, K=4, bias="normal"),
]


def _run(ctx, wl, dev, fp8_down=False):
    import varlen_grouped_gemm_gb300 as vgg
    buf = vgg.Buffers.allocate(wl.T, wl.d, wl.E, wl.n, wl.K, wl.m_tile, backward=False,
                               capacity_factor=wl.capacity_factor, drop_policy=wl.drop_policy, e4m3=True)
    w8 = vgg.E4m3Weights.quantize(ctx, dev["W_gate"], dev["W_up"], dev["W_down"] if fp8_down else None)
    vgg.forward_e4m3(ctx, dev["X"], dev["W_r"], dev["bias"], w8, dev["W_down"], buf)
    rc, code = vgg.moe_get_error(ctx)
    assert rc == vgg.MOE_OK and code == 0, (rc, code)
    return buf, w8


DOWN8_CASES = [
    synth.scaled(synth.WORKLOADS["c2"], name="c2_small_n256", T=512, d=256, E=16, n=256, K=4),
    synth.scaled(synth.WORKLOADS["c5"], name="c5_small_tr", T=2048, d=256, E=32, n=128, K=8, m_tile=64),
    synth.scaled(synth.WORKLOADS["c2_cap"], name="cap_f1_bias_n256", T=512, d=256, E=16, n=256, K=4, bias="normal"),
    synth.scaled(synth.WORKLOADS["c4"], name="c4_small_zipf_n384", T=640, d=384, E=32, n=384, K=4),
    # 512 experts: the group table leaves no room for a fourth stage (the three-stage form)
    synth.scaled(synth.WORKLOADS["c5_plain"], name="c5_small_e512", T=2048, d=256, E=512, n=128, K=8),
    # d = n = 320: both e4m3 GEMMs end on a half stage
    synth.scaled(synth.WORKLOADS["c4"], name="c4_small_320", T=640, d=320, E=32, n=320, K=4),
]


@pytest.mark.parametrize("wl,fp8_down", [(w, False) for w in CASES] + [(w, True) for w in DOWN8_CASES],
                         ids=lambda x: x.name if hasattr(x, "name") else ("down8" if x else "down16"))
def test_e4m3_forward_matches_oracle(ctx, wl, fp8_down):
    inp = Inputs(wl, with_grad=False)
    buf, w8 = _run(ctx, wl, inp.dev, fp8_down)
    E, n, d = wl.E, wl.n, wl.d
    xq, xs = mo.quantize_rows_e4m3(inp.X)
    np.testing.assert_array_equal(buf.xq.cpu().numpy(), xq)
    np.testing.assert_array_equal(buf.xs.cpu().numpy(), xs)
    for got_q, got_s, Wb in ((w8.Wg_q, w8.wg_scale, inp.W_gate), (w8.Wu_q, w8.wu_scale, inp.W_up)):
        q, s = mo.quantize_rows_e4m3(Wb.reshape(E * n, d))
        np.testing.assert_array_equal(got_q.cpu().numpy().reshape(E * n, d), q)
        np.testing.assert_array_equal(got_s.cpu().numpy().reshape(-1), s)

    g = gpu_routing(buf)
    C = buf.capacity
    O_ref, cache = mo.moe_forward_fp8(inp.X, inp.W_r, inp.bias, inp.W_gate, inp.W_up, inp.W_down, wl.K, wl.m_tile,
                                      logits_for_routing=g["logits"], scores_for_routing=g["scores"], capacity=C,
                                      policy=wl.drop_policy, drop_keys=g["topk_w"] if C else None,
                                      fp8_down=fp8_down)
    if fp8_down:
        # W_down's codes, and A's codes against the oracle's quantization of the device's own bf16 A rows
        q, s = mo.quantize_rows_e4m3(inp.W_down.reshape(E * d, n))
        np.testing.assert_array_equal(w8.Wd_q.cpu().numpy().reshape(E * d, n), q)
        np.testing.assert_array_equal(w8.wd_scale.cpu().numpy().reshape(-1), s)
        rows = int(buf.offsets[E].item())
        A_bits = buf.A[:rows].view(torch.int16).cpu().numpy().view(np.uint16)
        qa, sa = mo.quantize_rows_e4m3(A_bits)
        np.testing.assert_array_equal(buf.aq[:rows].cpu().numpy(), qa)
        np.testing.assert_array_equal(buf.as_[:rows].cpu().numpy(), sa)
    r = cache["routing"]
    rep = {"O": oracle.compare("O", dev_to_f64(buf.O), O_ref)}
    if C:
        # slots e*C + rank hold the kept pairs; the rest are empty (zero rows)
        slot_of = np.concatenate([e * C + np.arange(r.counts[e]) for e in range(E)]).astype(np.int64)
        empty = np.setdiff1d(np.arange(E * C), slot_of)
        assert r.P < wl.T * wl.K and len(empty) > 0
        assert not torch.any(buf.H[torch.from_numpy(empty).cuda()] != 0).item(), "empty slots give zero rows"
        sel = torch.from_numpy(slot_of).cuda()
        H, U, A = buf.H[sel], buf.U[sel], buf.A[sel]
    else:
        check_routing_bit_exact(g, wl.K, wl.m_tile)
        H, U, A = buf.H[:r.P], buf.U[:r.P], buf.A[:r.P]
    rep["H"] = oracle.compare("H", dev_to_f64(H), cache["h"])
    rep["U"] = oracle.compare("U", dev_to_f64(U), cache["u"])
    rep["A"] = oracle.compare("A", dev_to_f64(A), cache["a"])
    if wl.bias == "zipf":
        assert (r.counts == 0).any(), "the skewed prior should leave some experts empty"
    print(wl.name, {k: (round(v["max"], 5), round(v["mean"], 6)) for k, v in rep.items()})


def test_e4m3_fullsize_c2(ctx):
    """The c2 shape at full size (the configuration the benchmark's e4m3 line times), on sampled tokens:
    every expert contribution of a token depends only on its own row and the experts' weights."""
    wl = synth.WORKLOADS["c2"]
    dev = {name: bits_to_dev(make(wl)) for name, make in (
        ("X", synth.make_x), ("W_r", synth.make_router), ("W_gate", synth.make_w_gate), ("W_up", synth.make_w_up),
        ("W_down", synth.make_w_down))}
    dev["bias"] = None
    buf, w8 = _run(ctx, wl, dev)
    try:
        g = gpu_routing(buf)
        r = check_routing_bit_exact(g, wl.K, 0)
        rng = np.random.default_rng(77)
        toks = np.unique(np.concatenate([[0, wl.T - 1], rng.choice(wl.T, 6, replace=False)])).astype(np.int64)
        X = synth.make_x(wl, rows=toks)
        xq, xs = mo.quantize_rows_e4m3(X)
        tsel = torch.from_numpy(toks).cuda()
        np.testing.assert_array_equal(buf.xq[tsel].cpu().numpy(), xq)
        np.testing.assert_array_equal(buf.xs[tsel].cpu().numpy(), xs)
        Xd = mo.dequantize_rows_e4m3(xq, xs)
        L = mo.router_logits(X, synth.make_router(wl), None)
        w = mo.combine_weights(L, r.topk_ids[toks])
        O = np.zeros((len(toks), wl.d))
        member = r.member[toks]
        for e in sorted(set(np.nonzero(member)[1].tolist())):
            rows = np.nonzero(member[:, e])[0]
            gq, gs = mo.quantize_rows_e4m3(synth.make_w_gate(wl, [e])[0])
            uq, us = mo.quantize_rows_e4m3(synth.make_w_up(wl, [e])[0])
            np.testing.assert_array_equal(w8.Wg_q[e].cpu().numpy(), gq)
            np.testing.assert_array_equal(w8.wu_scale[e].cpu().numpy(), us)
            h = Xd[rows] @ mo.dequantize_rows_e4m3(gq, gs).T
            u = Xd[rows] @ mo.dequantize_rows_e4m3(uq, us).T
            y = (mo.silu(h) * u) @ mo.bf16_bits_to_f64(synth.make_w_down(wl, [e])[0]).T
            O[rows] += w[rows, e][:, None] * y
        rep = oracle.compare("O (sampled tokens)", dev_to_f64(buf.O[tsel]), O)
        print("c2 e4m3", len(toks), "tokens", (rep["max"], rep["mean"]))
    finally:
        del buf, dev, w8
        gc.collect()
        torch.cuda.empty_cache()


def test_e4m3_forward_only(ctx):
    """cache=False with the e4m3 down projection: the same O bit for bit, H and U left untouched."""
    import varlen_grouped_gemm_gb300 as vgg
    wl = synth.scaled(synth.WORKLOADS["c2"], name="c2_small_n256", T=512, d=256, E=16, n=256, K=4)
    inp = Inputs(wl, with_grad=False)
    dv = inp.dev
    buf = vgg.Buffers.allocate(wl.T, wl.d, wl.E, wl.n, wl.K, backward=False, e4m3=True)
    w8 = vgg.E4m3Weights.quantize(ctx, dv["W_gate"], dv["W_up"], dv["W_down"])
    vgg.forward_e4m3(ctx, dv["X"], dv["W_r"], dv["bias"], w8, None, buf)
    O_cached = buf.O.clone()
    buf.H.fill_(7.0)
    buf.U.fill_(7.0)
    buf.O.zero_()
    vgg.forward_e4m3(ctx, dv["X"], dv["W_r"], dv["bias"], w8, None, buf, cache=False)
    rc, code = vgg.moe_get_error(ctx)
    assert rc == vgg.MOE_OK and code == 0, (rc, code)
    assert torch.equal(buf.O, O_cached)
    assert bool((buf.H == 7.0).all()) and bool((buf.U == 7.0).all())


BWD8_CASES = [
    synth.scaled(synth.WORKLOADS["c2"], name="c2_small", T=512, d=256, E=16, n=192, K=4),
    synth.scaled(synth.WORKLOADS["c4"], name="c4_small_d320", T=640, d=320, E=32, n=320, K=4),
    synth.scaled(synth.WORKLOADS["c5"], name="c5_small_tr", T=2048, d=256, E=32, n=128, K=8, m_tile=64),
]


@pytest.mark.parametrize("dx,dact", [(True, False), (False, True), (True, True)], ids=["dx", "dact", "dx_dact"])
@pytest.mark.parametrize("wl", BWD8_CASES, ids=lambda w: w.name)
def test_e4m3_backward_matches_oracle(ctx, wl, dx, dact):
    """moe_backward_e4m3 against the oracle's e4m3 backward:
    * the weight codes ([W_gate; W_up]^T and W_down^T per row) bit for bit;
    * the dSwiGLU GEMM's dO codes bit for bit (they are decided on the exact bf16 dO);
    * the dX GEMM's [dH | dU] codes against the oracle's quantization of its own bf16 [dH | dU]: the decision
      is taken on values that differ by bf16 rounding, so a code may sit on the other side of an e4m3
      rounding boundary: at most 1% of them, each by one e4m3 step;
    * dX against the oracle's sum of the device's [dH | dU] codes times the B codes (plus the router part),
      within the usual tolerance: the GEMM and the per-token reduction exactly;
    * dX against the oracle's own e4m3 backward: mean within the usual tolerance, max within 0.15 (one e4m3
      step of a code is up to 12.5% of that element) -- the variant's own tolerance;
    * the weight gradients (operands dH, dU, A' rounded once to bf16) within that rounding's bound of the oracle's
      e4m3 backward (``check_dw_single_bf16``);
    * every other gradient within the usual tolerance of the oracle's e4m3 backward."""
    import varlen_grouped_gemm_gb300 as vgg
    import oracle
    from _helpers import compare_layer
    inp = Inputs(wl)
    dv = inp.dev
    E, n, d = wl.E, wl.n, wl.d
    buf = vgg.Buffers.allocate(wl.T, d, E, n, wl.K, wl.m_tile, backward=True, dW_dtype=torch.float32, e4m3=True)
    w8 = vgg.E4m3Weights.quantize(ctx, dv["W_gate"], dv["W_up"], dv["W_down"], backward=True)
    vgg.forward(ctx, dv["X"], dv["W_r"], dv["bias"], dv["W_gate"], dv["W_up"], dv["W_down"], buf)
    vgg.backward_e4m3(ctx, dv["dO"], dv["X"], dv["W_r"], dv["W_gate"], dv["W_up"], dv["W_down"], w8, buf, dx=dx,
                      dact=dact)
    rc, code = vgg.moe_get_error(ctx)
    assert rc == vgg.MOE_OK and code == 0, (rc, code)
    Wg, Wu = mo.bf16_bits_to_f64(inp.W_gate), mo.bf16_bits_to_f64(inp.W_up)
    Wd = mo.bf16_bits_to_f64(inp.W_down)
    B = np.concatenate([Wg, Wu], axis=1).transpose(0, 2, 1).reshape(E * d, 2 * n)  # [E*d, 2n]
    bq, bs = mo.quantize_rows_e4m3(B.astype(np.float32))
    np.testing.assert_array_equal(w8.Wgu_q.cpu().numpy().reshape(E * d, 2 * n), bq)
    np.testing.assert_array_equal(w8.wgu_scale.cpu().numpy().reshape(-1), bs)
    Bd = mo.dequantize_rows_e4m3(bq, bs).reshape(E, d, 2 * n)
    tq, ts = mo.quantize_rows_e4m3(Wd.transpose(0, 2, 1).reshape(E * n, d).astype(np.float32))
    np.testing.assert_array_equal(w8.Wdt_q.cpu().numpy().reshape(E * n, d), tq)
    np.testing.assert_array_equal(w8.wdt_scale.cpu().numpy().reshape(-1), ts)
    Wdt = mo.dequantize_rows_e4m3(tq, ts).reshape(E, n, d)

    g = gpu_routing(buf)
    O_ref, cache = mo.moe_forward(inp.X, inp.W_r, inp.bias, inp.W_gate, inp.W_up, inp.W_down, wl.K, wl.m_tile,
                                  logits_for_routing=g["logits"], scores_for_routing=g["scores"])
    grads = mo.moe_backward(inp.X, inp.W_r, inp.bias, inp.W_gate, inp.W_up, inp.W_down, inp.dO, cache,
                            fp8_dx=dx, fp8_dact=dact)
    r = cache["routing"]
    X64, dO64 = mo.bf16_bits_to_f64(inp.X), mo.bf16_bits_to_f64(inp.dO)
    if dact:  # dO codes of every sorted pair, bit for bit
        oq, os_ = mo.quantize_rows_e4m3(inp.dO[r.sorted_tok])
        np.testing.assert_array_equal(buf.doq[:r.P].cpu().numpy(), oq)
        np.testing.assert_array_equal(buf.dos[:r.P].cpu().numpy(), os_)
    if dact and buf.sorted_tok.numel() >= wl.T:  # dO quantized per token and gathered: empty rows zero, scale 1
        assert not buf.doq[r.P:].any().item() and bool((buf.dos[r.P:] == 1).all().item())
    flips = 0
    blocks = {}
    for e in range(E):
        lo, hi = r.offsets[e], r.offsets[e + 1]
        if hi == lo:
            continue
        rows = r.sorted_tok[lo:hi]
        dap = None
        if dact:
            dq, ds_ = mo.quantize_rows_e4m3(inp.dO[rows])
            dap = mo.dequantize_rows_e4m3(dq, ds_) @ Wdt[e].T
        blk = mo.expert_block_backward(X64[rows], dO64[rows], cache["w_full"][rows, e], inp.W_gate[e], inp.W_up[e],
                                       inp.W_down[e], dap=dap)
        blocks[e] = (blk["dh"], blk["du"], blk["a"])
    if dx:
        huq = buf.huq[:r.P].cpu().numpy()
        hus = buf.hus[:r.P].cpu().numpy()
        dX_codes = grads["dlogits"] @ mo.bf16_bits_to_f64(inp.W_r).T
        for e in range(E):
            lo, hi = r.offsets[e], r.offsets[e + 1]
            if hi == lo:
                continue
            rows = r.sorted_tok[lo:hi]
            dh, du, _ = blocks[e]
            hq, _ = mo.quantize_rows_e4m3(mo.round_bf16(np.concatenate([dh, du], axis=1)).astype(np.float32))
            diff = huq[lo:hi] != hq
            flips += int(diff.sum())
            if diff.any():  # a differing code is a neighbour on the e4m3 grid
                a, b = huq[lo:hi][diff].astype(np.int64), hq[diff].astype(np.int64)
                assert np.all((a & 0x80) == (b & 0x80)) and np.all(np.abs((a & 0x7F) - (b & 0x7F)) <= 1)
            np.add.at(dX_codes, rows, mo.dequantize_rows_e4m3(huq[lo:hi], hus[lo:hi]) @ Bd[e].T)
        assert flips <= 0.01 * huq.size, flips
        # the e4m3 GEMM and the token reduction on the device's own codes: the usual bf16 tolerance
        oracle.compare("dX (from the device's codes)", dev_to_f64(buf.dX), dX_codes)
    rep = compare_layer(buf, inp, O_ref, cache, grads,
                        skip=(("dX",) if dx else ()) + ("dW_gate", "dW_up", "dW_down"))
    # the weight gradients take dH, dU, A' rounded once to bf16: that rounding's bound
    rep["dW bound"] = {"max": check_dw_single_bf16(buf, blocks, X64, dO64, r, cache["w_full"]), "mean": 0.0}
    # against the oracle's own e4m3 backward: the variant's tolerance (one e4m3 step of a code is up to 12.5%
    # of that element), both floors
    end = oracle.compare("dX (e4m3 variant)", dev_to_f64(buf.dX), grads["dX"], max_rel=0.15)
    print(wl.name, "dx", dx, "dact", dact, "code flips", flips, "dX vs oracle e4m3",
          (round(end["max"], 4), round(end["mean"], 6)), {k: (round(v["max"], 5), round(v["mean"], 6)) for k, v in rep.items()})


@pytest.mark.parametrize("dx", [False, True], ids=["dact", "dx_dact"])
def test_e4m3_backward_capacity_layout(ctx, dx):
    """The e4m3 dSwiGLU GEMM on the capacity layout ([E, C] slots) with fewer slots than tokens: dO is then
    quantized on its sorted rows rather than once per token.  The slots' dO codes and scales bit for bit (empty
    slots: zero codes, scale 1); every gradient against the oracle's e4m3 backward on the same kept pairs
    (dX with the variant's own tolerance when the dX GEMM is e4m3 too, else the usual one)."""
    import varlen_grouped_gemm_gb300 as vgg
    import oracle
    wl = synth.scaled(synth.WORKLOADS["c2_cap"], name="cap_e4m3", T=512, d=256, E=16, n=192, K=2,
                      capacity_factor=0.25)
    inp = Inputs(wl)
    dv = inp.dev
    buf = vgg.Buffers.allocate(wl.T, wl.d, wl.E, wl.n, wl.K, wl.m_tile, backward=True, dW_dtype=torch.float32,
                               capacity_factor=wl.capacity_factor, drop_policy=wl.drop_policy, e4m3=True)
    assert buf.sorted_tok.numel() < wl.T
    w8 = vgg.E4m3Weights.quantize(ctx, dv["W_gate"], dv["W_up"], dv["W_down"], backward=True)
    vgg.forward(ctx, dv["X"], dv["W_r"], dv["bias"], dv["W_gate"], dv["W_up"], dv["W_down"], buf)
    vgg.backward_e4m3(ctx, dv["dO"], dv["X"], dv["W_r"], dv["W_gate"], dv["W_up"], dv["W_down"], w8, buf, dx=dx,
                      dact=True)
    rc, code = vgg.moe_get_error(ctx)
    assert rc == vgg.MOE_OK and code == 0, (rc, code)
    C = mo.expert_capacity(wl.T, wl.E, wl.K, wl.capacity_factor)
    O_ref, cache = mo.moe_forward(inp.X, inp.W_r, inp.bias, inp.W_gate, inp.W_up, inp.W_down, wl.K,
                                  logits_for_routing=buf.logits.cpu().numpy(), capacity=C, policy=wl.drop_policy,
                                  drop_keys=buf.topk_w.cpu().numpy())
    r = cache["routing"]
    assert r.P < wl.T * wl.K
    st = buf.sorted_tok.cpu().numpy()
    kept = st >= 0
    q, sc = mo.quantize_rows_e4m3(inp.dO[st[kept]])
    doq, dos = buf.doq.cpu().numpy(), buf.dos.cpu().numpy()
    np.testing.assert_array_equal(doq[kept], q)
    np.testing.assert_array_equal(dos[kept], sc)
    assert not doq[~kept].any() and np.all(dos[~kept] == 1)
    g = mo.moe_backward(inp.X, inp.W_r, inp.bias, inp.W_gate, inp.W_up, inp.W_down, inp.dO, cache, fp8_dx=dx,
                        fp8_dact=True)
    oracle.compare("O", dev_to_f64(buf.O), O_ref)
    dX = dev_to_f64(buf.dX)
    if dx:
        oracle.compare("dX (e4m3 variant)", dX, g["dX"], max_rel=0.15)
    else:
        oracle.compare("dX", dX, g["dX"])
    # the weight gradients on operands rounded once to bf16: that rounding's bound
    Wd = mo.bf16_bits_to_f64(inp.W_down)
    tq, ts = mo.quantize_rows_e4m3(Wd.transpose(0, 2, 1).reshape(wl.E * wl.n, wl.d).astype(np.float32))
    Wdt = mo.dequantize_rows_e4m3(tq, ts).reshape(wl.E, wl.n, wl.d)
    X64, dO64 = mo.bf16_bits_to_f64(inp.X), mo.bf16_bits_to_f64(inp.dO)
    blocks = {}
    for e in range(wl.E):
        rows = r.rows_of(e)
        if len(rows) == 0:
            continue
        dq, ds_ = mo.quantize_rows_e4m3(inp.dO[rows])
        blk = mo.expert_block_backward(X64[rows], dO64[rows], cache["w_full"][rows, e], inp.W_gate[e], inp.W_up[e],
                                       inp.W_down[e], dap=mo.dequantize_rows_e4m3(dq, ds_) @ Wdt[e].T)
        blocks[e] = (blk["dh"], blk["du"], blk["a"])
        for name, key in (("dW_gate", "dWg"), ("dW_up", "dWu"), ("dW_down", "dWd")):
            np.testing.assert_allclose(blk[key], g[name][e], rtol=1e-12, atol=1e-15)
    check_dw_single_bf16(buf, blocks, X64, dO64, r, cache["w_full"])
    slot_of = np.concatenate([e * C + np.arange(r.counts[e]) for e in range(wl.E)]).astype(np.int64)
    oracle.compare("dS", dev_to_f64(buf.dS)[slot_of], g["dw"][r.sorted_tok, r.sorted_exp])
    oracle.compare("dlogits", dev_to_f64(buf.dlogits), g["dlogits"])
    oracle.compare("dW_r", dev_to_f64(buf.dW_r), g["dW_r"])
