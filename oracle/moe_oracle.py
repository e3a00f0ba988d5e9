"""Plain fp64 oracle of the MoE expert layer, forward and backward.

TEST INFRASTRUCTURE: imported only by tests, the smoke check and the bench's
CPU baseline.  It is the loop-over-experts shape of the naive training forward
(gather each expert's tokens, three small GEMMs, scatter back), with no
blocking, fusion or reordering beyond what the definitions below state.

Sources (page title, then the section a function follows):

[GG]  "DeepSeek 계열 MoE 학습 가속: Python expert loop → grouped GEMM"
[EP]  "EP: Expert를 나누고 토큰 보내기"
[SM]  "SonicMoE: IO·타일 인식 최적화로 MoE 학습 가속하기"
[DEP] "Deep EP"
[DEP] "Drop/Padding 방식" (same page): the capacity-based dispatch variant

Readings where the pages are silent (listed again in the design notes):
* top-K order: descending logit, ties to the lower expert index;
* sort by expert is stable: within an expert, pairs keep ascending token order;
* combine weights are the softmax renormalised over the top-K experts;
* token rounding: r_e = M * floor((c_e + M/2) / M) capped at M * floor(T/M);
  priority of a token for expert e is (score s[t,e] descending, token ascending);
  padding adds the highest-priority unrouted tokens, dropping removes the
  lowest-priority routed ones; every final pair (t,e) has weight
  s[t,e] / sum_{j in TopK(t)} s[t,j] (the same denominator as top-K);
* the router bias is added to the logits and is not trained;
* capacity dispatch: C = ceil(cf * T * K / E); the "position" policy keeps an
  expert's first C routed tokens in token order, the "probs" policy the C with
  the largest routing probability (the top-K renormalised weight), ties to the
  lower token; kept pairs keep their top-K weight (no re-normalisation).

All floating point here is fp64; bf16 inputs are widened exactly.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits (uint16) to float64."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _f64(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return bf16_bits_to_f64(a)
    return a.astype(np.float64)


# ---------------------------------------------------------------- router


def router_logits(X, W_r, bias=None) -> np.ndarray:
    """l[t,e] = sum_i X[t,i] W_r[i,e] + b[e].

    [DEP] "1) Router": the router looks at the BN x H input token-wise and
    scores every expert ("gate weight score").
    """
    L = _f64(X) @ _f64(W_r)
    if bias is not None:
        L = L + _f64(bias)[None, :]
    return L


def topk_experts(logits, K: int) -> np.ndarray:
    """Indices of the K largest logits per token, largest first, ties to the lower expert.

    [DEP] "1) Router": top-k expert indices per token ([BN, k]).  The comparison
    happens in the dtype of ``logits`` (fp32 logits from a device give the
    device's decision; fp64 logits the exact one).
    """
    logits = np.asarray(logits)
    order = np.argsort(-logits, axis=1, kind="stable")
    return order[:, :K].astype(np.int64)


def softmax(logits) -> np.ndarray:
    """Full softmax over the experts, s[t,e] (fp64)."""
    L = _f64(logits)
    z = np.exp(L - L.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def combine_weights(logits, topk_ids) -> np.ndarray:
    """Weights of every expert relative to the token's top-K set, w[t,e] (fp64, [T,E]).

    w[t,e] = exp(l[t,e]) / sum_{j in TopK(t)} exp(l[t,j]); on the top-K set these
    sum to 1.  [EP] "여러 Expert의 결과도 같은 토큰으로 돌아오기": the weights used to
    combine (0.7 / 0.3 in the example) are kept apart from the selection.
    """
    L = _f64(logits)
    T = L.shape[0]
    rows = np.arange(T)[:, None]
    m = L[rows, topk_ids].max(axis=1, keepdims=True)
    denom = np.exp(L[rows, topk_ids] - m).sum(axis=1, keepdims=True)
    return np.exp(L - m) / denom


def group_by_expert(topk_ids, E: int):
    """Flatten the (token, slot) pairs and sort them by expert, stably.

    [GG] "적용 — fused MoE training forward", steps (1)-(3): topk_ids is
    flattened to 1-D and sorted by expert id, so each expert's tokens form one
    contiguous slice; bincount gives the per-expert token counts.
    [DEP] table "Ragged vs Padding": the ragged layout needs offset metadata.

    Returns counts[E], offsets[E+1], perm[P] (pair p = t*K + k at sorted
    position j is perm[j]) and sorted_tok[P].
    """
    topk_ids = np.asarray(topk_ids)
    K = topk_ids.shape[1]
    flat = topk_ids.reshape(-1)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    perm = np.argsort(flat, kind="stable").astype(np.int64)
    return counts, offsets, perm, perm // K


def token_rounding(scores, topk_ids, m_tile: int):
    """Round every expert's token count to the nearest multiple of m_tile.

    [SM] "5 기여 ③ Token Rounding 라우팅": first plain top-K token choice; then,
    per expert, sort by score and round the received count to the nearest
    multiple of M_tile — pad with the highest-scoring tokens when short, drop
    the lowest-scoring ones when over.

    ``scores`` are the full-softmax scores s[T,E] (compared in their own
    dtype).  Returns member[T,E] (the final pair set) and r[E].
    """
    scores = np.asarray(scores)
    T, E = scores.shape
    routed = np.zeros((T, E), dtype=bool)
    routed[np.arange(T)[:, None], topk_ids] = True
    counts = routed.sum(axis=0)
    r = m_tile * ((counts + m_tile // 2) // m_tile)
    r = np.minimum(r, m_tile * (T // m_tile))
    member = np.zeros((T, E), dtype=bool)
    tokens = np.arange(T)
    for e in range(E):
        # priority order: score descending, then token ascending
        order = np.lexsort((tokens, -scores[:, e]))
        routed_first = order[routed[order, e]]
        unrouted_first = order[~routed[order, e]]
        if r[e] <= counts[e]:
            keep = routed_first[: r[e]]
        else:
            keep = np.concatenate([routed_first, unrouted_first[: r[e] - counts[e]]])
        member[keep, e] = True
    return member, r.astype(np.int64)


def expert_capacity(T: int, E: int, K: int, capacity_factor: float) -> int:
    """Capacity C of every expert: the capacity factor times the mean load T*K/E, rounded up.

    [DEP] "Drop/Padding 방식": the [BN, H] tokens are rearranged per expert into [E, C, H],
    C being the most tokens one expert can hold; the pages give no formula for C, the
    capacity factor is named for the variant's switch.
    """
    return int(math.ceil(capacity_factor * T * K / E))


def capacity_drop(topk_ids, keys, E: int, C: int, policy: str = "position") -> np.ndarray:
    """The pairs an expert keeps under capacity C: member[T,E].

    [DEP] "Drop/Padding 방식": line up each expert's tokens, cut at C and drop the rest;
    tokens over capacity go by the "position" policy (the first C in token order stay)
    or the "probs" policy (the C with the largest routing probability stay, ties to the
    lower token).  ``keys[T,K]`` are the routing probabilities of the top-K pairs (the
    combine weights), compared in their own dtype.
    """
    topk_ids = np.asarray(topk_ids)
    keys = np.asarray(keys)
    T, K = topk_ids.shape
    member = np.zeros((T, E), dtype=bool)
    for e in range(E):
        tt, kk = np.nonzero(topk_ids == e)  # tokens ascending
        if policy == "position":
            keep = tt[:C]
        elif policy == "probs":
            order = np.lexsort((tt, -keys[tt, kk]))
            keep = tt[order][:C]
        else:
            raise ValueError(policy)
        member[keep, e] = True
    return member


@dataclass
class Routing:
    """Discrete routing state: which (token, expert) pairs exist and in which order.

    topk_ids[T,K]  the top-K selection (TopK(t), largest first)
    member[T,E]    the final pair set F(t) (= TopK(t) without token rounding)
    counts[E], offsets[E+1]
    sorted_tok[P], sorted_exp[P]   pairs grouped by expert, ascending token inside
    tok_ptr[T+1], tok_pairs[P]     per token, its sorted positions in ascending expert
    """

    topk_ids: np.ndarray
    member: np.ndarray
    counts: np.ndarray
    offsets: np.ndarray
    sorted_tok: np.ndarray
    sorted_exp: np.ndarray
    tok_ptr: np.ndarray
    tok_pairs: np.ndarray

    @property
    def P(self) -> int:
        return int(self.offsets[-1])

    def rows_of(self, e: int) -> np.ndarray:
        return self.sorted_tok[self.offsets[e]:self.offsets[e + 1]]


def route_discrete(logits, K: int, m_tile: int = 0, scores=None, capacity: int = 0, policy: str = "position",
                   drop_keys=None) -> Routing:
    """The discrete stage of routing from a given set of logits (and scores for rounding).

    With ``capacity`` > 0 the pairs over an expert's capacity are dropped (``capacity_drop``);
    ``drop_keys[T,K]`` are the routing probabilities the "probs" policy compares (default:
    the oracle's own combine weights of the top-K pairs).

    Builds the expert-grouped order ([GG] steps (1)-(3)) and the per-token
    return map ([EP] "토큰을 Expert로 보내고 원래 위치로 돌려받기": each result has to
    be tracked back to its token).
    """
    logits = np.asarray(logits)
    T, E = logits.shape
    topk = topk_experts(logits, K)
    if m_tile:
        if scores is None:
            scores = softmax(logits)
        member, _ = token_rounding(scores, topk, m_tile)
    elif capacity:
        if drop_keys is None:
            drop_keys = np.take_along_axis(combine_weights(logits, topk), topk, axis=1)
        member = capacity_drop(topk, drop_keys, E, capacity, policy)
    else:
        member = np.zeros((T, E), dtype=bool)
        member[np.arange(T)[:, None], topk] = True
    counts = member.sum(axis=0).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    # expert-major, token-ascending order of the pairs
    e_idx, t_idx = np.nonzero(member.T)
    sorted_exp, sorted_tok = e_idx.astype(np.int64), t_idx.astype(np.int64)
    if not m_tile and not capacity:
        # cross-check with the flatten + stable-sort description
        c2, o2, _, st2 = group_by_expert(topk, E)
        assert np.array_equal(c2, counts) and np.array_equal(st2, sorted_tok)
    P = len(sorted_tok)
    j_of = np.full((T, E), -1, dtype=np.int64)
    j_of[sorted_tok, sorted_exp] = np.arange(P)
    tok_cnt = member.sum(axis=1)
    tok_ptr = np.concatenate([[0], np.cumsum(tok_cnt)]).astype(np.int64)
    tt, ee = np.nonzero(member)  # token-major, expert ascending
    tok_pairs = j_of[tt, ee]
    return Routing(topk, member, counts, offsets, sorted_tok, sorted_exp, tok_ptr, tok_pairs)


# ---------------------------------------------------------------- experts


def silu(z):
    return z / (1.0 + np.exp(-z))


def expert_ffn(x, Wg, Wu, Wd):
    """One expert's SwiGLU MLP on the rows routed to it.

    [GG] "(6) 세 번의 gg.gmm": gate, up and down projections with the stacked
    (out, in) weights; [SM] "4.2 Epilogue 융합": SwiGLU, a = silu(x Wg^T) * (x Wu^T).
    Returns h, u, a, y (all fp64).
    """
    x, Wg, Wu, Wd = _f64(x), _f64(Wg), _f64(Wu), _f64(Wd)
    h = x @ Wg.T
    u = x @ Wu.T
    a = silu(h) * u
    y = a @ Wd.T
    return h, u, a, y


def combine(y_sorted, routing: Routing, w_full, T: int) -> np.ndarray:
    """Weighted sum of every token's expert outputs back in original token order.

    [EP] "여러 Expert의 결과도 같은 토큰으로 돌아오기": y(A2) = 0.7 u0 + 0.3 u2, placed
    back in A2's own slot; [DEP] "3) Combine": weighted sum of the k expert outputs.
    ``y_sorted`` holds one row per pair in expert-grouped order.
    """
    y_sorted = _f64(y_sorted)
    O = np.zeros((T, y_sorted.shape[1]))
    w = w_full[routing.sorted_tok, routing.sorted_exp]
    np.add.at(O, routing.sorted_tok, w[:, None] * y_sorted)
    return O


def moe_forward(X, W_r, bias, W_gate, W_up, W_down, K: int, m_tile: int = 0, logits_for_routing=None,
                scores_for_routing=None, capacity: int = 0, policy: str = "position", drop_keys=None):
    """Forward of the layer.  Returns (O[T,d], cache).

    ``capacity`` > 0 selects the capacity (drop/pad) dispatch of ``route_discrete``.

    The selection comes from ``logits_for_routing`` (and ``scores_for_routing``
    under token rounding) when given — e.g. a device's fp32 logits, so that the
    discrete decisions match — else from the oracle's own fp64 logits.  The
    combine weights always come from the oracle's fp64 logits.
    """
    X = _f64(X)
    T, d = X.shape
    L = router_logits(X, W_r, bias)
    sel = L if logits_for_routing is None else logits_for_routing
    routing = route_discrete(sel, K, m_tile, scores=scores_for_routing, capacity=capacity, policy=policy,
                             drop_keys=drop_keys)
    w_full = combine_weights(L, routing.topk_ids)
    E = L.shape[1]
    y_sorted = np.zeros((routing.P, d))
    for e in range(E):
        lo, hi = routing.offsets[e], routing.offsets[e + 1]
        if hi == lo:
            continue
        rows = routing.sorted_tok[lo:hi]
        _, _, _, y = expert_ffn(X[rows], W_gate[e], W_up[e], W_down[e])
        y_sorted[lo:hi] = y
    O = combine(y_sorted, routing, w_full, T)
    return O, dict(logits=L, routing=routing, w_full=w_full, y_sorted=y_sorted)


def expert_block_backward(x, dO, w, Wg, Wu, Wd, dap=None):
    """Backward of one expert on the rows routed to it, by the chain rule on its definition.

    O_t = sum_e w[t,e] y_e(x_t), y = a Wd^T, a = silu(h) * u, h = x Wg^T, u = x Wu^T.
    Returns dict with y, dw (= <dO_t, y_t>), dx contribution, dWg, dWu, dWd.
    ``dap`` replaces dA' = dO Wd (the unweighted gradient of a) when given (the e4m3 dSwiGLU GEMM);
    dw is then <dA', a>, the identity the fused epilogue uses.
    """
    x, dO, w = _f64(x), _f64(dO), _f64(w)
    Wg, Wu, Wd = _f64(Wg), _f64(Wu), _f64(Wd)
    h, u, a, y = expert_ffn(x, Wg, Wu, Wd)
    dy = w[:, None] * dO
    if dap is None:
        dw = np.sum(dO * y, axis=1)
        da = dy @ Wd
    else:
        dw = np.sum(dap * a, axis=1)
        da = w[:, None] * dap
    sig = 1.0 / (1.0 + np.exp(-h))
    du = da * (h * sig)
    dh = da * u * (sig * (1.0 + h * (1.0 - sig)))
    return dict(y=y, a=a, h=h, u=u, dw=dw, dh=dh, du=du,
                dx=dh @ Wg + du @ Wu,
                dWg=dh.T @ x, dWu=du.T @ x, dWd=dy.T @ a)


def router_grad_rows(member, topk_ids, w_full, dw_full):
    """d loss / d logits for the rows given.

    w[t,i] = exp(l_i) / sum_{j in TopK(t)} exp(l_j) for every final pair i in F(t), so
    dL[t,k] = [k in F(t)] w_k dw_k - [k in TopK(t)] w_k * sum_{i in F(t)} w_i dw_i.
    """
    T, E = member.shape
    topk_mask = np.zeros((T, E), dtype=bool)
    topk_mask[np.arange(T)[:, None], topk_ids] = True
    G = np.sum(np.where(member, w_full * dw_full, 0.0), axis=1, keepdims=True)
    return np.where(member, w_full * dw_full, 0.0) - np.where(topk_mask, w_full * G, 0.0)


def moe_backward(X, W_r, bias, W_gate, W_up, W_down, dO, cache, experts=None, fp8_dx: bool = False,
                 fp8_dact: bool = False, mx_dx: bool = False, mx_dact: bool = False, mx_dw: bool = False):
    """Backward of the layer given the forward cache.

    Returns dX, dW_gate, dW_up, dW_down (fp64, all experts or the listed ones),
    dw[T,E] (d loss / d combine weight, zero off the pair set), dlogits[T,E], dW_r[d,E].

    With ``fp8_dx`` the expert part of dX takes e4m3 operands: each pair's row [dH | dU] (bf16, the
    dSwiGLU epilogue's output type, ``round_bf16``) quantized per row, and [W_gate; W_up]^T (d rows of
    2n) quantized per row (per input channel of the layer), ``quantize_rows_e4m3``.
    With ``fp8_dact`` the dSwiGLU GEMM dA' = dO W_down takes e4m3 operands: dO per token (row) and
    W_down^T (n rows of d) per row; dS = <dA', A> then comes from that dA' (the epilogue's identity).
    ``mx_dx`` and ``mx_dact`` are the same two GEMMs with block-scaled operands (``quantize_blocks_mx``):
    [dH | dU] quantized from its exact value (blocks along 2n) against [W_gate; W_up]^T (blocks along 2n),
    and dO per token against W_down^T (blocks along d).
    ``mx_dw``: the weight gradients with block-scaled operands whose blocks run along the expert's tokens
    (``dequantize_token_blocks_mx``): dW_gate = dq(dH)^T dq(X), dW_up = dq(dU)^T dq(X) and
    dW_down = dq(dO)^T dq(A') with A' = w a, every operand quantized from its exact value.
    """
    X, dO = _f64(X), _f64(dO)
    T, d = X.shape
    routing: Routing = cache["routing"]
    w_full = cache["w_full"]
    E = w_full.shape[1]
    n = W_gate.shape[1]
    dX = np.zeros((T, d))
    dw_full = np.zeros((T, E))
    keep = range(E) if experts is None else list(experts)
    dWg = {e: np.zeros((n, d)) for e in keep}
    dWu = {e: np.zeros((n, d)) for e in keep}
    dWd = {e: np.zeros((d, n)) for e in keep}
    for e in range(E):
        rows = routing.rows_of(e)
        if len(rows) == 0:
            continue
        dap = None
        if mx_dact:
            oq, oe = quantize_blocks_mx(dO[rows])
            wq, we = quantize_blocks_mx(_f64(W_down[e]).T)  # [n, d]
            dap = dequantize_blocks_mx(oq, oe) @ dequantize_blocks_mx(wq, we).T
        elif fp8_dact:
            oq, os_ = quantize_rows_e4m3(dO[rows].astype(np.float32))
            wq, ws_ = quantize_rows_e4m3(_f64(W_down[e]).T.astype(np.float32))  # [n, d]
            dap = dequantize_rows_e4m3(oq, os_) @ dequantize_rows_e4m3(wq, ws_).T
        g = expert_block_backward(X[rows], dO[rows], w_full[rows, e], W_gate[e], W_up[e], W_down[e], dap=dap)
        dw_full[rows, e] = g["dw"]
        if mx_dx:
            hq, he = quantize_blocks_mx(np.concatenate([g["dh"], g["du"]], axis=1))
            B = np.concatenate([_f64(W_gate[e]), _f64(W_up[e])], axis=0).T  # [d, 2n]
            bq, be = quantize_blocks_mx(B)
            np.add.at(dX, rows, dequantize_blocks_mx(hq, he) @ dequantize_blocks_mx(bq, be).T)
        elif fp8_dx:
            hq, hs = quantize_rows_e4m3(round_bf16(np.concatenate([g["dh"], g["du"]], axis=1)).astype(np.float32))
            B = np.concatenate([_f64(W_gate[e]), _f64(W_up[e])], axis=0).T  # [d, 2n]
            bq, bs = quantize_rows_e4m3(B.astype(np.float32))
            np.add.at(dX, rows, dequantize_rows_e4m3(hq, hs) @ dequantize_rows_e4m3(bq, bs).T)
        else:
            np.add.at(dX, rows, g["dx"])
        if e in dWg and mx_dw:
            xt = dequantize_token_blocks_mx(X[rows])
            dWg[e] = dequantize_token_blocks_mx(g["dh"]).T @ xt
            dWu[e] = dequantize_token_blocks_mx(g["du"]).T @ xt
            dWd[e] = dequantize_token_blocks_mx(dO[rows]).T @ dequantize_token_blocks_mx(w_full[rows, e][:, None] * g["a"])
        elif e in dWg:
            dWg[e], dWu[e], dWd[e] = g["dWg"], g["dWu"], g["dWd"]
    dL = router_grad_rows(routing.member, routing.topk_ids, w_full, dw_full)
    Wr = _f64(W_r)
    dX += dL @ Wr.T
    dWr = X.T @ dL
    return dict(dX=dX, dW_gate=dWg, dW_up=dWu, dW_down=dWd, dw=dw_full, dlogits=dL, dW_r=dWr)


# ---------------------------------------------------------------- FP8 variant of the gate/up GEMM
#
# [GG] "FP8" (DeepGEMM is named for FP8 grouped GEMMs): the variant computes the gate/up
# projections from e4m3 operands.  The pages give no scaling recipe; reading: one fp32 scale per
# row of X (per token) and per row of W_gate / W_up (per output channel), s = amax / 448 computed in
# fp32, codes e4m3(x / s) with x / s in fp32, round to nearest even, saturating at +-448.  The
# product of two dequantized rows is then exact in fp64.

E4M3_MAX = 448.0


def e4m3_round(v) -> np.ndarray:
    """Nearest e4m3 value of each element (ties to even), saturating at +-448, as fp64.

    e4m3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; normal values 2^(e-7) (1 + m/8) for
    e = 1..15 (all but e = 15, m = 7, which is NaN), subnormals 2^-6 m/8.  The spacing of the values
    in [2^k, 2^(k+1)) is 2^(k-3) for k >= -6, and 2^-9 below 2^-6.
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    k = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    step = np.where(a >= 2.0 ** -6, 2.0 ** (k - 3), 2.0 ** -9)
    q = np.round(a / step) * step  # np.round: half to even; a / step is exact (power-of-two step)
    q = np.minimum(q, E4M3_MAX)
    return np.copysign(q, v)


def e4m3_encode(v) -> np.ndarray:
    """The e4m3 bit patterns (uint8) of values already on the e4m3 grid."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    sign = (np.signbit(v)).astype(np.uint8) << 7
    k = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    normal = a >= 2.0 ** -6
    e = np.where(normal, k + 7, 0).astype(np.int64)
    m = np.where(normal, a / 2.0 ** k - 1.0, a / 2.0 ** -6) * 8
    code = (e << 3) | np.round(m).astype(np.int64)
    return (sign | np.where(a > 0, code, 0).astype(np.uint8)).astype(np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    """fp64 values of e4m3 bit patterns (uint8; NaN patterns are not produced here)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e > 0, 2.0 ** (e - 7) * (1.0 + m / 8.0), 2.0 ** -6 * (m / 8.0))
    return s * mag


def quantize_rows_e4m3(M):
    """Per-row e4m3 quantization: (codes uint8 [R, C], scales fp32 [R]); row r dequantizes to
    e4m3_decode(codes[r]) * scales[r].  The scale and the divided values are computed in fp32."""
    A = np.asarray(M)
    if A.dtype == np.uint16:
        A = bf16_bits_to_f64(A).astype(np.float32)
    A = A.astype(np.float32)
    amax = np.max(np.abs(A), axis=-1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    y = (A / scale[..., None]).astype(np.float32)
    return e4m3_encode(e4m3_round(y)), scale


def dequantize_rows_e4m3(codes, scales) -> np.ndarray:
    return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[..., None]


def round_bf16(v) -> np.ndarray:
    """Nearest bf16 value (8 significant bits, ties to even) of each element, as fp64 (normal range)."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)  # v = m 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.round(m * 256.0) / 256.0, e)


def moe_forward_fp8(X, W_r, bias, W_gate, W_up, W_down, K: int, m_tile: int = 0, logits_for_routing=None,
                    scores_for_routing=None, capacity: int = 0, policy: str = "position", drop_keys=None,
                    fp8_down: bool = False):
    """Forward of the layer with the gate/up projections from e4m3 operands (per-token scales on X,
    per-output-channel scales on W_gate and W_up, ``quantize_rows_e4m3``); routing (with the same
    token rounding / capacity options), SwiGLU, the down projection and the combine as in
    ``moe_forward``.  With ``fp8_down`` the down projection takes e4m3 operands as well: the
    activation rows A (the bf16 operand of the down projection, ``round_bf16``) quantized per row and
    W_down per output channel.  Returns (O, cache) with the cache's ``h``, ``u``, ``a`` per sorted
    pair (fp64) and the quantized operands."""
    X64 = _f64(X)
    T, d = X64.shape
    E, n, _ = np.shape(W_gate)
    xq, xs = quantize_rows_e4m3(X)
    Xd = dequantize_rows_e4m3(xq, xs)
    gq, gs = quantize_rows_e4m3(np.asarray(W_gate).reshape(E * n, d))
    uq, us = quantize_rows_e4m3(np.asarray(W_up).reshape(E * n, d))
    Wg_d = dequantize_rows_e4m3(gq, gs).reshape(E, n, d)
    Wu_d = dequantize_rows_e4m3(uq, us).reshape(E, n, d)
    L = router_logits(X64, W_r, bias)
    sel = L if logits_for_routing is None else logits_for_routing
    routing = route_discrete(sel, K, m_tile, scores=scores_for_routing, capacity=capacity, policy=policy,
                             drop_keys=drop_keys)
    w_full = combine_weights(L, routing.topk_ids)
    P = routing.P
    h = np.zeros((P, n))
    u = np.zeros((P, n))
    for e in range(E):
        lo, hi = routing.offsets[e], routing.offsets[e + 1]
        if hi == lo:
            continue
        rows = routing.sorted_tok[lo:hi]
        h[lo:hi] = Xd[rows] @ Wg_d[e].T
        u[lo:hi] = Xd[rows] @ Wu_d[e].T
    a = silu(h) * u
    extra = {}
    if fp8_down:
        aq, as_ = quantize_rows_e4m3(round_bf16(a).astype(np.float32))
        dq, ds = quantize_rows_e4m3(np.asarray(W_down).reshape(E * d, n))
        a_op = dequantize_rows_e4m3(aq, as_)
        Wd_op = dequantize_rows_e4m3(dq, ds).reshape(E, d, n)
        extra = dict(aq=aq, as_=as_, dq=dq, ds=ds)
    else:
        a_op, Wd_op = a, None
    y_sorted = np.zeros((P, d))
    for e in range(E):
        lo, hi = routing.offsets[e], routing.offsets[e + 1]
        if hi == lo:
            continue
        y_sorted[lo:hi] = a_op[lo:hi] @ (Wd_op[e] if fp8_down else _f64(W_down[e])).T
    O = combine(y_sorted, routing, w_full, T)
    return O, dict(logits=L, routing=routing, w_full=w_full, h=h, u=u, a=a, y_sorted=y_sorted,
                   xq=xq, xs=xs, gq=gq, gs=gs, uq=uq, us=us, **extra)


# ---------------------------------------------------------------- block-scaled (1 x 32) e4m3 variant
#
# [GG] "한계": the further 2x credited to DeepSeek's *fine-grained* FP8 grouped GEMM.  The pages give no
# scaling recipe; reading: every operand row is cut into blocks of 32 consecutive elements along the
# reduction dimension, each block has a power-of-two scale 2^e (one UE8M0 byte, e + 127) with e the
# smallest integer such that the block's largest magnitude is at most 448 2^e (clamped to [-127, 127];
# an all-zero block takes e = 0), and its codes are e4m3(x 2^-e) rounded to nearest even.  The scaling
# by 2^-e is exact, and no code saturates.  A GEMM of two such operands sums, per 32-element block,
# the code products times both blocks' scales.

MX_BLOCK = 32


def mx_block_exponents(amax) -> np.ndarray:
    """The block exponent e of each block maximum: smallest e with amax <= 448 2^e, in [-127, 127];
    0 for an all-zero block."""
    a = np.asarray(amax, dtype=np.float64)
    _, E = np.frexp(np.where(a > 0, a, 1.0))  # a = f 2^E, 0.5 <= f < 1: floor(log2 a) = E - 1
    e = (E - 1) - 8  # a 2^-e in [256, 512)
    e = np.where(np.ldexp(a, -e) > E4M3_MAX, e + 1, e)
    e = np.clip(e, -127, 127)
    return np.where(a > 0, e, 0).astype(np.int64)


def quantize_blocks_mx(M):
    """1 x 32 block quantization along the last axis: (codes uint8 [..., C], exponents int64 [..., C/32]).

    Element j of a row dequantizes to e4m3_decode(code) 2^e[j // 32]."""
    A = _f64(M)
    C = A.shape[-1]
    if C % MX_BLOCK:
        raise ValueError("the blocked axis must be a multiple of 32")
    blocks = A.reshape(A.shape[:-1] + (C // MX_BLOCK, MX_BLOCK))
    e = mx_block_exponents(np.max(np.abs(blocks), axis=-1))
    y = np.ldexp(blocks, -e[..., None])  # exact
    codes = e4m3_encode(e4m3_round(y)).reshape(A.shape)
    return codes, e


def dequantize_blocks_mx(codes, exps) -> np.ndarray:
    c = np.asarray(codes)
    C = c.shape[-1]
    v = e4m3_decode(c).reshape(c.shape[:-1] + (C // MX_BLOCK, MX_BLOCK))
    return np.ldexp(v, np.asarray(exps, dtype=np.int64)[..., None]).reshape(c.shape)


def dequantize_token_blocks_mx(M) -> np.ndarray:
    """Block-scaled values of an expert's [rows, C] operand with the blocks along the rows (tokens): rows
    32 b .. 32 b + 31 of one column form block b, the last block holding the rows left (its largest magnitude
    over those rows alone; zero rows appended to make whole blocks change no block's maximum).  The reduction
    of a weight gradient runs over an expert's tokens, so its 1 x 32 blocks are these."""
    A = _f64(M)
    R, C = A.shape
    Rp = -(-R // MX_BLOCK) * MX_BLOCK
    padded = np.zeros((Rp, C))
    padded[:R] = A
    q, e = quantize_blocks_mx(padded.T)  # [C, Rp]: blocks along the tokens
    return dequantize_blocks_mx(q, e).T[:R]


def moe_forward_mx(X, W_r, bias, W_gate, W_up, W_down, K: int, m_tile: int = 0, logits_for_routing=None,
                   scores_for_routing=None, capacity: int = 0, policy: str = "position", drop_keys=None,
                   mx_down: bool = True):
    """Forward of the layer with block-scaled e4m3 operands (``quantize_blocks_mx``): X per token and
    W_gate / W_up per output channel, blocks along d, for the gate/up projections; with ``mx_down`` the
    down projection takes the activation rows A = silu(h) u (quantized from their exact value, blocks along
    n) and W_down per output channel (blocks along n).  Routing, SwiGLU and the combine as in
    ``moe_forward``.  Returns (O, cache) with h, u, a per sorted pair (fp64) and the codes and exponents."""
    X64 = _f64(X)
    T, d = X64.shape
    E, n, _ = np.shape(W_gate)
    xq, xe = quantize_blocks_mx(X64)
    gq, ge = quantize_blocks_mx(_f64(W_gate).reshape(E * n, d))
    uq, ue = quantize_blocks_mx(_f64(W_up).reshape(E * n, d))
    Xd = dequantize_blocks_mx(xq, xe)
    Wg_d = dequantize_blocks_mx(gq, ge).reshape(E, n, d)
    Wu_d = dequantize_blocks_mx(uq, ue).reshape(E, n, d)
    L = router_logits(X64, W_r, bias)
    sel = L if logits_for_routing is None else logits_for_routing
    routing = route_discrete(sel, K, m_tile, scores=scores_for_routing, capacity=capacity, policy=policy,
                             drop_keys=drop_keys)
    w_full = combine_weights(L, routing.topk_ids)
    P = routing.P
    h = np.zeros((P, n))
    u = np.zeros((P, n))
    for e in range(E):
        lo, hi = routing.offsets[e], routing.offsets[e + 1]
        if hi == lo:
            continue
        rows = routing.sorted_tok[lo:hi]
        h[lo:hi] = Xd[rows] @ Wg_d[e].T
        u[lo:hi] = Xd[rows] @ Wu_d[e].T
    a = silu(h) * u
    extra = {}
    if mx_down:
        aq, ae = quantize_blocks_mx(a)
        dq, de = quantize_blocks_mx(_f64(W_down).reshape(E * d, n))
        a_op = dequantize_blocks_mx(aq, ae)
        Wd_op = dequantize_blocks_mx(dq, de).reshape(E, d, n)
        extra = dict(aq=aq, ae=ae, dq=dq, de=de)
    else:
        a_op, Wd_op = a, _f64(W_down)
    y_sorted = np.zeros((P, d))
    for e in range(E):
        lo, hi = routing.offsets[e], routing.offsets[e + 1]
        if hi == lo:
            continue
        y_sorted[lo:hi] = a_op[lo:hi] @ Wd_op[e].T
    O = combine(y_sorted, routing, w_full, T)
    return O, dict(logits=L, routing=routing, w_full=w_full, h=h, u=u, a=a, y_sorted=y_sorted,
                   xq=xq, xe=xe, gq=gq, ge=ge, uq=uq, ue=ue, **extra)
