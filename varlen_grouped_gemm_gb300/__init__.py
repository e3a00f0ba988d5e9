"""GB300 (sm_103a) MoE expert-layer hot path — Python binding of the C ABI in ``include/moe.h``.

Argument marshalling only: every step of the path (routing, grouping, grouped
GEMMs, combine, backward) runs in the CUDA library ``lib/libvgg_moe.so``.
PyTorch supplies device memory and streams.  There is no CPU fallback: when
the library is missing, every call raises.

The functions carry the C names (``moe_route``, ``moe_permute``,
``moe_grouped_gemm_fwd``, ``moe_combine``, ``moe_backward``); sizes are taken
from the tensors' shapes.  ``Buffers`` allocates every tensor the path needs
for one configuration, and ``forward_backward`` runs the whole path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libvgg_moe.so")

# The symbols declared in include/moe.h.
EXPORTS = (
    "moe_create", "moe_destroy", "moe_status_str", "moe_get_error", "moe_set_wait_timeout", "moe_set_cta_pairs",
    "moe_pair_capacity", "moe_workspace_bytes", "moe_route", "moe_permute", "moe_grouped_gemm_fwd",
    "moe_combine", "moe_backward", "moe_profile_enable", "moe_profile_read", "moe_test_gemm_varlen_m",
    "moe_test_gemm_varlen_k", "moe_test_wait_timeout", "moe_permute_noalloc", "moe_permute_capacity",
    "moe_capacity_workspace_bytes", "moe_quantize_rows_e4m3", "moe_grouped_gemm_fwd_e4m3",
    "moe_quantize_dx_weights_e4m3", "moe_quantize_dact_weights_e4m3", "moe_backward_e4m3",
    "moe_expert_capacity", "moe_test_gemm_varlen_k_dual", "moe_test_gemm_varlen_m_dual",
    "moe_mx_sf_cols", "moe_mx_weight_sf_bytes", "moe_mx_act_sf_bytes", "moe_quantize_rows_mx",
    "moe_quantize_weights_mx", "moe_grouped_gemm_fwd_mx", "moe_quantize_bwd_weights_mx", "moe_backward_mx",
    "moe_mx_dw_ws_bytes",
)

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_DEVICE, MOE_ERR_DEVICE_TIMEOUT = range(6)
DEV_OK, DEV_BAD_EXPERT, DEV_DUP_EXPERT, DEV_BAD_OFFSETS, DEV_TIMEOUT, DEV_CAPACITY = range(6)

_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_LL = ctypes.c_longlong
_SZ = ctypes.c_size_t


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                               "(run varlen_grouped_gemm_gb300/build.py or __graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        L.moe_create.argtypes = [ctypes.POINTER(_P), _I]
        L.moe_destroy.argtypes = [_P]
        L.moe_status_str.argtypes = [_I]
        L.moe_status_str.restype = ctypes.c_char_p
        L.moe_get_error.argtypes = [_P, ctypes.POINTER(_I)]
        L.moe_set_wait_timeout.argtypes = [_P, ctypes.c_ulonglong]
        L.moe_set_cta_pairs.argtypes = [_P, _I, _I]
        L.moe_pair_capacity.argtypes = [_I, _I, _I, _I]
        L.moe_pair_capacity.restype = _LL
        L.moe_workspace_bytes.argtypes = [_I, _I, _I, _I, _I, _I]
        L.moe_workspace_bytes.restype = _SZ
        L.moe_route.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]
        L.moe_permute.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _LL, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
        L.moe_grouped_gemm_fwd.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _LL, _P, _P, _P, _P, _P, _P, _P,
                                           _P, _SZ, _P]
        L.moe_combine.argtypes = [_P, _P, _P, _P, _I, _I, _LL, _P, _P]
        L.moe_backward.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _LL, _P, _P, _P, _P, _P,
                                   _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _SZ, _P]
        L.moe_test_gemm_varlen_m.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _LL, _P, _P, _P]
        L.moe_test_gemm_varlen_k.argtypes = [_P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _LL, _P, _P, _P]
        L.moe_test_wait_timeout.argtypes = [_P, ctypes.c_ulonglong, _P]
        L.moe_expert_capacity.argtypes = [_I, _I, _I, ctypes.c_double]
        L.moe_expert_capacity.restype = _LL
        L.moe_test_gemm_varlen_k_dual.argtypes = [_P, _P, _P, _I, _P, _I, _I, _I, _I, _LL, _P, _P, _I, _P, _P]
        L.moe_test_gemm_varlen_m_dual.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _LL, _P, _P, _P]
        L.moe_permute_noalloc.argtypes = [_P, _P, _P, _I, _I, _I, _LL, _P, _P, _P, _P, _P, _P, _P, _P]
        L.moe_permute_capacity.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _LL, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                           _P]
        L.moe_capacity_workspace_bytes.argtypes = [_I, _I, _I, _I, _I, _I]
        L.moe_capacity_workspace_bytes.restype = _SZ
        L.moe_quantize_rows_e4m3.argtypes = [_P, _P, _LL, _I, _P, _P, _P]
        L.moe_grouped_gemm_fwd_e4m3.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _LL, _P,
                                                _P, _P, _P, _P, _P, _P, _P, _P, _P]
        L.moe_quantize_dx_weights_e4m3.argtypes = [_P, _P, _P, _I, _I, _I, _P, _P, _P, _P]
        L.moe_quantize_dact_weights_e4m3.argtypes = [_P, _P, _I, _I, _I, _P, _P, _P, _P]
        L.moe_backward_e4m3.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _LL,
                                        _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I,
                                        _P, _P, _P, _P, _SZ, _P]
        L.moe_mx_sf_cols.argtypes = [_I]
        L.moe_mx_sf_cols.restype = _LL
        L.moe_mx_weight_sf_bytes.argtypes = [_I, _I, _I, _I]
        L.moe_mx_weight_sf_bytes.restype = _LL
        L.moe_mx_act_sf_bytes.argtypes = [_LL, _I, _I]
        L.moe_mx_act_sf_bytes.restype = _LL
        L.moe_mx_dw_ws_bytes.argtypes = [_I, _I, _I, _LL]
        L.moe_mx_dw_ws_bytes.restype = _SZ
        L.moe_quantize_rows_mx.argtypes = [_P, _P, _LL, _I, _P, _P, _P]
        L.moe_quantize_weights_mx.argtypes = [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P]
        L.moe_grouped_gemm_fwd_mx.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _LL, _P, _P, _P, _P,
                                              _P, _P, _P, _P, _P, _P]
        L.moe_quantize_bwd_weights_mx.argtypes = [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P]
        L.moe_backward_mx.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _LL, _P, _P,
                                      _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P,
                                      _SZ, _P, _SZ, _P]
        L.moe_profile_enable.argtypes = [_P, _I]
        L.moe_profile_read.argtypes = [_P, _I, ctypes.c_char_p, ctypes.POINTER(ctypes.c_double),
                                       ctypes.POINTER(_LL), ctypes.POINTER(_I)]
        _lib = L
    return _lib


def status_str(code: int) -> str:
    return lib().moe_status_str(code).decode()


def _check(name: str, rc: int):
    if rc != MOE_OK:
        raise RuntimeError(f"{name} failed: {status_str(rc)} (status {rc})")


def _ptr(t: torch.Tensor | None, dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class Context:
    """A library context on one device (owns the device error word)."""

    def __init__(self, device: int = 0):
        self.device = device
        h = _P()
        _check("moe_create", lib().moe_create(ctypes.byref(h), device))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            lib().moe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_wait_timeout(self, ns: int):
        _check("moe_set_wait_timeout", lib().moe_set_wait_timeout(self.handle, int(ns)))

    def set_cta_pairs(self, varlen_m: bool, varlen_k: bool):
        """CTA pairs (two CTAs per 256-row tile) for the tiled varlen-M and the weight-gradient GEMMs."""
        _check("moe_set_cta_pairs", lib().moe_set_cta_pairs(self.handle, int(varlen_m), int(varlen_k)))


def moe_profile_enable(ctx: Context, enable: bool = True):
    _check("moe_profile_enable", lib().moe_profile_enable(ctx.handle, 1 if enable else 0))


def moe_profile_read(ctx: Context) -> dict[str, tuple[float, int]]:
    """{kernel label: (total ms, launches)} since the last read (waits for the recorded events)."""
    nmax = 64
    names = ctypes.create_string_buffer(32 * nmax)
    ms = (ctypes.c_double * nmax)()
    cnt = (_LL * nmax)()
    n = _I(0)
    _check("moe_profile_read", lib().moe_profile_read(ctx.handle, nmax, names, ms, cnt, ctypes.byref(n)))
    out = {}
    for i in range(min(n.value, nmax)):
        label = names.raw[32 * i:32 * i + 32].split(b"\0", 1)[0].decode()
        out[label] = (ms[i], int(cnt[i]))
    return out


def moe_get_error(ctx: Context) -> tuple[int, int]:
    """(status, device error code); synchronizes the device and clears the code."""
    code = _I(0)
    rc = lib().moe_get_error(ctx.handle, ctypes.byref(code))
    return rc, code.value


def moe_pair_capacity(T: int, E: int, K: int, m_tile: int = 0) -> int:
    return int(lib().moe_pair_capacity(T, E, K, m_tile))


def moe_workspace_bytes(T: int, d: int, E: int, n: int, K: int, m_tile: int = 0) -> int:
    return int(lib().moe_workspace_bytes(T, d, E, n, K, m_tile))


def _ws(ws):
    return (None, 0) if ws is None else (ws.data_ptr(), ws.numel() * ws.element_size())


def moe_route(ctx, X, W_r, bias, K, logits, scores, topk_ids, topk_w, ws=None, stream=None):
    T, d = X.shape
    E = W_r.shape[1]
    wp, wb = _ws(ws)
    _check("moe_route", lib().moe_route(
        ctx.handle, _ptr(X, torch.bfloat16, "X"), _ptr(W_r, torch.bfloat16, "W_r"),
        _ptr(bias, torch.float32, "bias"), T, d, E, K, _ptr(logits, torch.float32, "logits"),
        _ptr(scores, torch.float32, "scores"), _ptr(topk_ids, torch.int32, "topk_ids"),
        _ptr(topk_w, torch.float32, "topk_w"), wp, wb, _stream(stream)))


def moe_permute(ctx, topk_ids, topk_w, logits, scores, E, m_tile, counts, offsets, sorted_tok, sorted_w,
                tok_ptr, tok_pairs, P_out, ws, stream=None):
    T, K = topk_ids.shape
    cap = sorted_tok.numel()
    wp, wb = _ws(ws)
    _check("moe_permute", lib().moe_permute(
        ctx.handle, _ptr(topk_ids, torch.int32), _ptr(topk_w, torch.float32), _ptr(logits, torch.float32),
        _ptr(scores, torch.float32), T, E, K, m_tile, cap, _ptr(counts, torch.int32),
        _ptr(offsets, torch.int32), _ptr(sorted_tok, torch.int32), _ptr(sorted_w, torch.float32),
        _ptr(tok_ptr, torch.int32), _ptr(tok_pairs, torch.int32), _ptr(P_out, torch.int32), wp, wb,
        _stream(stream)))


def moe_permute_noalloc(ctx, topk_ids, topk_w, E, counts, offsets, sorted_tok, sorted_w, tok_ptr, tok_pairs, P_out,
                        stream=None):
    """moe_permute (plain top-K) with its scratch in a fixed array inside the library: for callers
    that cannot allocate device memory.  At most 32768 tokens and 512 experts."""
    T, K = topk_ids.shape
    _check("moe_permute_noalloc", lib().moe_permute_noalloc(
        ctx.handle, _ptr(topk_ids, torch.int32), _ptr(topk_w, torch.float32), T, E, K, sorted_tok.numel(),
        _ptr(counts, torch.int32), _ptr(offsets, torch.int32), _ptr(sorted_tok, torch.int32),
        _ptr(sorted_w, torch.float32), _ptr(tok_ptr, torch.int32), _ptr(tok_pairs, torch.int32),
        _ptr(P_out, torch.int32), _stream(stream)))


POLICIES = {"position": 0, "probs": 1}


def expert_capacity(T: int, E: int, K: int, capacity_factor: float) -> int:
    """Slots per expert of the capacity dispatch (the library's moe_expert_capacity)."""
    C = int(lib().moe_expert_capacity(T, E, K, float(capacity_factor)))
    if C < 1:
        raise ValueError(f"moe_expert_capacity: invalid arguments T={T} E={E} K={K} cf={capacity_factor}")
    return C


def moe_permute_capacity(ctx, topk_ids, topk_w, E, C, policy, counts, offsets, sorted_tok, sorted_w, tok_ptr,
                         tok_pairs, P_out, ws, stream=None):
    """Capacity (drop/pad) dispatch: expert e keeps at most C pairs in slots [e C, (e+1) C)."""
    T, K = topk_ids.shape
    wp, wb = _ws(ws)
    _check("moe_permute_capacity", lib().moe_permute_capacity(
        ctx.handle, _ptr(topk_ids, torch.int32), _ptr(topk_w, torch.float32), T, E, K, C, POLICIES[policy],
        sorted_tok.numel(), _ptr(counts, torch.int32), _ptr(offsets, torch.int32), _ptr(sorted_tok, torch.int32),
        _ptr(sorted_w, torch.float32), _ptr(tok_ptr, torch.int32), _ptr(tok_pairs, torch.int32),
        _ptr(P_out, torch.int32), wp, wb, _stream(stream)))


def moe_capacity_workspace_bytes(T: int, d: int, E: int, n: int, K: int, C: int) -> int:
    return int(lib().moe_capacity_workspace_bytes(T, d, E, n, K, C))


def moe_grouped_gemm_fwd(ctx, X, W_gate, W_up, W_down, offsets, sorted_tok, sorted_w, H, U, A, Yw, ws=None,
                         stream=None):
    T, d = X.shape
    E, n, _ = W_gate.shape
    cap = sorted_tok.numel()
    wp, wb = _ws(ws)
    bf = torch.bfloat16
    _check("moe_grouped_gemm_fwd", lib().moe_grouped_gemm_fwd(
        ctx.handle, _ptr(X, bf), _ptr(W_gate, bf), _ptr(W_up, bf), _ptr(W_down, bf), T, d, E, n, cap,
        _ptr(offsets, torch.int32), _ptr(sorted_tok, torch.int32), _ptr(sorted_w, torch.float32),
        _ptr(H, torch.float32), _ptr(U, torch.float32), _ptr(A, bf), _ptr(Yw, bf), wp, wb, _stream(stream)))


def moe_quantize_rows_e4m3(ctx, M, q, scales, stream=None):
    """Per-row e4m3 codes (uint8, shaped like M) and fp32 scales (one per row of M's last axis)."""
    cols = M.shape[-1]
    rows = M.numel() // cols
    if q.shape != M.shape or scales.numel() != rows:
        raise ValueError("q must be shaped like M and scales hold one value per row")
    _check("moe_quantize_rows_e4m3", lib().moe_quantize_rows_e4m3(
        ctx.handle, _ptr(M, torch.bfloat16), rows, cols, _ptr(q, torch.uint8), _ptr(scales, torch.float32),
        _stream(stream)))


def moe_grouped_gemm_fwd_e4m3(ctx, Xq, x_scale, Wg_q, wg_scale, Wu_q, wu_scale, W_down, offsets, sorted_tok,
                              sorted_w, H, U, A, Yw, Wd_q=None, wd_scale=None, Aq=None, a_scale=None, stream=None):
    """e4m3 gate/up; the down projection in bf16 (W_down) or, given Wd_q / wd_scale and the Aq / a_scale
    buffers, in e4m3."""
    T, d = Xq.shape
    E, n, _ = Wg_q.shape
    cap = sorted_tok.numel()
    u8, f32 = torch.uint8, torch.float32
    _check("moe_grouped_gemm_fwd_e4m3", lib().moe_grouped_gemm_fwd_e4m3(
        ctx.handle, _ptr(Xq, u8), _ptr(x_scale, f32), _ptr(Wg_q, u8), _ptr(wg_scale, f32), _ptr(Wu_q, u8),
        _ptr(wu_scale, f32), _ptr(W_down, torch.bfloat16), _ptr(Wd_q, u8), _ptr(wd_scale, f32), T, d, E, n, cap,
        _ptr(offsets, torch.int32), _ptr(sorted_tok, torch.int32), _ptr(sorted_w, f32), _ptr(H, f32), _ptr(U, f32),
        _ptr(A, torch.bfloat16), _ptr(Aq, u8), _ptr(a_scale, f32), _ptr(Yw, torch.bfloat16), _stream(stream)))


def mx_sf_cols(cols: int) -> int:
    """Bytes per row of a row-major block-scale array (the library's moe_mx_sf_cols)."""
    return int(lib().moe_mx_sf_cols(cols))


def mx_weight_sf_bytes(E: int, d: int, n: int, which: int) -> int:
    """Bytes of the weight scale blocks: which = 0 the W_gate / W_up pair, 1 W_down."""
    b = int(lib().moe_mx_weight_sf_bytes(E, d, n, which))
    if b <= 0:
        raise ValueError(f"moe_mx_weight_sf_bytes: invalid arguments E={E} d={d} n={n} which={which}")
    return b


def mx_dw_ws_bytes(d: int, E: int, n: int, cap: int) -> int:
    """Bytes of the block-scaled weight gradients' workspace (``moe_mx_dw_ws_bytes``)."""
    b = int(lib().moe_mx_dw_ws_bytes(d, E, n, cap))
    if b <= 0:
        raise ValueError(f"moe_mx_dw_ws_bytes: invalid arguments d={d} E={E} n={n} cap={cap}")
    return b


def mx_act_sf_bytes(cap: int, E: int, n: int) -> int:
    """Bytes of the activation scale blocks of the block-scaled down projection."""
    b = int(lib().moe_mx_act_sf_bytes(cap, E, n))
    if b <= 0:
        raise ValueError(f"moe_mx_act_sf_bytes: invalid arguments cap={cap} E={E} n={n}")
    return b


def moe_quantize_rows_mx(ctx, M, q, sf, stream=None):
    """Block-scaled codes (uint8, shaped like M) and row-major scale bytes [rows, mx_sf_cols(cols)]."""
    cols = M.shape[-1]
    rows = M.numel() // cols
    if q.shape != M.shape or sf.numel() != rows * mx_sf_cols(cols):
        raise ValueError("q must be shaped like M and sf hold mx_sf_cols(cols) bytes per row")
    _check("moe_quantize_rows_mx", lib().moe_quantize_rows_mx(
        ctx.handle, _ptr(M, torch.bfloat16), rows, cols, _ptr(q, torch.uint8), _ptr(sf, torch.uint8),
        _stream(stream)))


def moe_quantize_weights_mx(ctx, W_gate, W_up, W_down, Wg_q, Wu_q, gu_sf, Wd_q, dn_sf, stream=None):
    E, n, d = W_gate.shape
    bf, u8 = torch.bfloat16, torch.uint8
    _check("moe_quantize_weights_mx", lib().moe_quantize_weights_mx(
        ctx.handle, _ptr(W_gate, bf), _ptr(W_up, bf), _ptr(W_down, bf), E, d, n, _ptr(Wg_q, u8), _ptr(Wu_q, u8),
        _ptr(gu_sf, u8), _ptr(Wd_q, u8), _ptr(dn_sf, u8), _stream(stream)))


def moe_grouped_gemm_fwd_mx(ctx, Xq, x_sf, w, offsets, sorted_tok, sorted_w, H, U, x_sf_tiles, Aq, a_sf, Yw,
                            stream=None):
    """Block-scaled gate/up (+ SwiGLU, A quantized in the epilogue) and down projection; ``w`` is MxWeights,
    ``x_sf_tiles`` scratch of mx_act_sf_bytes(cap, E, d) bytes."""
    T, d = Xq.shape
    E, n, _ = w.Wg_q.shape
    cap = sorted_tok.numel()
    u8, f32 = torch.uint8, torch.float32
    _check("moe_grouped_gemm_fwd_mx", lib().moe_grouped_gemm_fwd_mx(
        ctx.handle, _ptr(Xq, u8), _ptr(x_sf, u8), _ptr(w.Wg_q, u8), _ptr(w.Wu_q, u8), _ptr(w.gu_sf, u8),
        _ptr(w.Wd_q, u8), _ptr(w.dn_sf, u8), T, d, E, n, cap, _ptr(offsets, torch.int32),
        _ptr(sorted_tok, torch.int32), _ptr(sorted_w, f32), _ptr(H, f32), _ptr(U, f32), _ptr(x_sf_tiles, u8),
        _ptr(Aq, u8), _ptr(a_sf, u8), _ptr(Yw, torch.bfloat16), _stream(stream)))


def moe_combine(ctx, Yw, tok_ptr, tok_pairs, O, stream=None):
    T, d = O.shape
    _check("moe_combine", lib().moe_combine(
        ctx.handle, _ptr(Yw, torch.bfloat16), _ptr(tok_ptr, torch.int32), _ptr(tok_pairs, torch.int32), T, d,
        tok_pairs.numel(), _ptr(O, torch.bfloat16), _stream(stream)))


def moe_backward(ctx, dO, X, W_r, W_gate, W_up, W_down, K, m_tile, topk_ids, topk_w, offsets, sorted_tok,
                 sorted_w, tok_ptr, tok_pairs, H, U, dX, dW_gate, dW_up, dW_down, dS, dlogits, dW_r, ws,
                 stream=None):
    T, d = X.shape
    E, n, _ = W_gate.shape
    cap = sorted_tok.numel()
    wp, wb = _ws(ws)
    bf = torch.bfloat16
    dw_fp32 = 1 if dW_gate.dtype == torch.float32 else 0
    _check("moe_backward", lib().moe_backward(
        ctx.handle, _ptr(dO, bf), _ptr(X, bf), _ptr(W_r, bf), _ptr(W_gate, bf), _ptr(W_up, bf), _ptr(W_down, bf),
        T, d, E, n, K, m_tile, cap, _ptr(topk_ids, torch.int32), _ptr(topk_w, torch.float32),
        _ptr(offsets, torch.int32), _ptr(sorted_tok, torch.int32), _ptr(sorted_w, torch.float32),
        _ptr(tok_ptr, torch.int32), _ptr(tok_pairs, torch.int32), _ptr(H, torch.float32), _ptr(U, torch.float32),
        _ptr(dX, bf),
        _ptr(dW_gate), _ptr(dW_up), _ptr(dW_down), dw_fp32, _ptr(dS, torch.float32),
        _ptr(dlogits, torch.float32), _ptr(dW_r, torch.float32), wp, wb, _stream(stream)))


def moe_quantize_dx_weights_e4m3(ctx, W_gate, W_up, Wgu_q, wgu_scale, stream=None):
    """[W_gate; W_up]^T per expert ([E, d, 2n]) as e4m3 codes with one scale per row (the dX GEMM's B)."""
    E, n, d = W_gate.shape
    tmp = torch.empty((E, d, 2 * n), dtype=torch.bfloat16, device=W_gate.device)
    _check("moe_quantize_dx_weights_e4m3", lib().moe_quantize_dx_weights_e4m3(
        ctx.handle, _ptr(W_gate, torch.bfloat16), _ptr(W_up, torch.bfloat16), E, n, d, _ptr(tmp, torch.bfloat16),
        _ptr(Wgu_q, torch.uint8), _ptr(wgu_scale, torch.float32), _stream(stream)))
    return tmp  # the caller keeps it alive until the stream has run the call


def moe_quantize_dact_weights_e4m3(ctx, W_down, Wdt_q, wdt_scale, stream=None):
    """W_down^T per expert ([E, n, d]) as e4m3 codes with one scale per row (the dSwiGLU GEMM's B)."""
    E, d, n = W_down.shape
    tmp = torch.empty((E, n, d), dtype=torch.bfloat16, device=W_down.device)
    _check("moe_quantize_dact_weights_e4m3", lib().moe_quantize_dact_weights_e4m3(
        ctx.handle, _ptr(W_down, torch.bfloat16), E, n, d, _ptr(tmp, torch.bfloat16), _ptr(Wdt_q, torch.uint8),
        _ptr(wdt_scale, torch.float32), _stream(stream)))
    return tmp  # the caller keeps it alive until the stream has run the call


def moe_backward_e4m3(ctx, dO, X, W_r, W_gate, W_up, W_down, Wgu_q, wgu_scale, Wdt_q, wdt_scale, K, m_tile, topk_ids,
                      topk_w, offsets, sorted_tok, sorted_w, tok_ptr, tok_pairs, H, U, HUq, hu_scale, dOq, do_scale,
                      dX, dW_gate, dW_up, dW_down, dS, dlogits, dW_r, ws, stream=None):
    T, d = X.shape
    E, n, _ = W_gate.shape
    cap = sorted_tok.numel()
    wp, wb = _ws(ws)
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    dw_fp32 = 1 if dW_gate.dtype == torch.float32 else 0
    _check("moe_backward_e4m3", lib().moe_backward_e4m3(
        ctx.handle, _ptr(dO, bf), _ptr(X, bf), _ptr(W_r, bf), _ptr(W_gate, bf), _ptr(W_up, bf), _ptr(W_down, bf),
        _ptr(Wgu_q, torch.uint8), _ptr(wgu_scale, f32), _ptr(Wdt_q, torch.uint8), _ptr(wdt_scale, f32), T, d, E, n,
        K, m_tile, cap, _ptr(topk_ids, i32), _ptr(topk_w, f32), _ptr(offsets, i32), _ptr(sorted_tok, i32),
        _ptr(sorted_w, f32), _ptr(tok_ptr, i32), _ptr(tok_pairs, i32), _ptr(H, f32), _ptr(U, f32),
        _ptr(HUq, torch.uint8), _ptr(hu_scale, f32), _ptr(dOq, torch.uint8), _ptr(do_scale, f32), _ptr(dX, bf),
        _ptr(dW_gate), _ptr(dW_up), _ptr(dW_down), dw_fp32, _ptr(dS, f32), _ptr(dlogits, f32), _ptr(dW_r, f32), wp,
        wb, _stream(stream)))


def moe_test_gemm_varlen_m(ctx, A, idx, B, b_kmajor, offsets, D, stream=None):
    G = B.shape[0]
    K = A.shape[1]
    N = B.shape[1] if b_kmajor else B.shape[2]
    _check("moe_test_gemm_varlen_m", lib().moe_test_gemm_varlen_m(
        ctx.handle, _ptr(A, torch.bfloat16), _ptr(idx, torch.int32), _ptr(B, torch.bfloat16), int(b_kmajor), G,
        A.shape[0], K, N, D.shape[0], _ptr(offsets, torch.int32), _ptr(D, torch.float32), _stream(stream)))


def moe_test_gemm_varlen_k(ctx, A, idx_a, B, idx_b, offsets, D, cap, stream=None):
    G, M, N = D.shape
    _check("moe_test_gemm_varlen_k", lib().moe_test_gemm_varlen_k(
        ctx.handle, _ptr(A, torch.bfloat16), _ptr(idx_a, torch.int32), A.shape[0], _ptr(B, torch.bfloat16),
        _ptr(idx_b, torch.int32), B.shape[0], G, M, N, cap, _ptr(offsets, torch.int32), _ptr(D, torch.float32),
        _stream(stream)))


def moe_test_gemm_varlen_m_dual(ctx, A_hi, A_lo, B, offsets, D, stream=None):
    """Test export: per group and sorted row, (A_hi + A_lo) B[e]^T (B is [G, N, K]); D is [cap, N] fp32."""
    G, N, K = B.shape
    _check("moe_test_gemm_varlen_m_dual", lib().moe_test_gemm_varlen_m_dual(
        ctx.handle, _ptr(A_hi, torch.bfloat16), _ptr(A_lo, torch.bfloat16), _ptr(B, torch.bfloat16), G,
        A_hi.shape[0], K, N, D.shape[0], _ptr(offsets, torch.int32), _ptr(D, torch.float32), _stream(stream)))


def moe_test_gemm_varlen_k_dual(ctx, A_hi, A_lo, B, offsets, D, cap, trans=False, b_offsets=None, stream=None):
    """Test export: per group, (A_hi + A_lo)^T B over the group's rows (D [G, M, N], or [G, N, M] with trans);
    b_offsets: B's rows in the padded layout (groups rounded up to 16 rows, zero rows in between)."""
    G = D.shape[0]
    M = A_hi.shape[1]
    N = B.shape[1]
    _check("moe_test_gemm_varlen_k_dual", lib().moe_test_gemm_varlen_k_dual(
        ctx.handle, _ptr(A_hi, torch.bfloat16), _ptr(A_lo, torch.bfloat16), A_hi.shape[0], _ptr(B, torch.bfloat16),
        B.shape[0], G, M, N, cap, _ptr(offsets, torch.int32), _ptr(b_offsets, torch.int32), int(bool(trans)),
        _ptr(D, torch.float32), _stream(stream)))


def moe_test_wait_timeout(ctx, timeout_ns: int, stream=None):
    _check("moe_test_wait_timeout", lib().moe_test_wait_timeout(ctx.handle, int(timeout_ns), _stream(stream)))


# ------------------------------------------------------------------ buffers and the whole path


@dataclass
class Buffers:
    """Every device tensor of one forward + backward for sizes (T, d, E, n, K, m_tile)."""

    T: int
    d: int
    E: int
    n: int
    K: int
    m_tile: int
    cap: int
    logits: torch.Tensor
    scores: torch.Tensor | None
    topk_ids: torch.Tensor
    topk_w: torch.Tensor
    counts: torch.Tensor
    offsets: torch.Tensor
    sorted_tok: torch.Tensor
    sorted_w: torch.Tensor
    tok_ptr: torch.Tensor
    tok_pairs: torch.Tensor
    P: torch.Tensor
    H: torch.Tensor
    U: torch.Tensor
    A: torch.Tensor
    Yw: torch.Tensor
    O: torch.Tensor
    dX: torch.Tensor | None
    dW_gate: torch.Tensor | None
    dW_up: torch.Tensor | None
    dW_down: torch.Tensor | None
    dS: torch.Tensor | None
    dlogits: torch.Tensor | None
    dW_r: torch.Tensor | None
    ws: torch.Tensor
    capacity: int = 0          # capacity dispatch: slots per expert (0 = ragged)
    drop_policy: str = "position"
    xq: torch.Tensor | None = None  # e4m3 forward: X's codes [T, d] and per-token scales [T]
    xs: torch.Tensor | None = None
    aq: torch.Tensor | None = None  # e4m3 down projection: A's codes [cap, n] and per-row scales [cap]
    as_: torch.Tensor | None = None
    huq: torch.Tensor | None = None  # e4m3 dX GEMM: [dH | dU] codes [cap, 2n] and per-row scales [cap]
    hus: torch.Tensor | None = None
    doq: torch.Tensor | None = None  # e4m3 dSwiGLU GEMM: sorted dO codes [cap, d] and per-row scales [cap]
    dos: torch.Tensor | None = None
    mxq: torch.Tensor | None = None  # block-scaled forward: X's codes [T, d] and scales [T, mx_sf_cols(d)]
    mxsf: torch.Tensor | None = None
    maq: torch.Tensor | None = None  # block-scaled down projection: A's codes [cap, n] and scale blocks
    masf: torch.Tensor | None = None
    mxsft: torch.Tensor | None = None  # block-scaled gate/up: the gathered X rows' scales per sorted row tile
    mdoq: torch.Tensor | None = None  # block-scaled backward: sorted dO codes [cap, d], their scales per row tile,
    mdosft: torch.Tensor | None = None  # [dH | dU] codes [cap, 2n] and their scale blocks
    mhuq: torch.Tensor | None = None
    mhusf: torch.Tensor | None = None
    mdw: torch.Tensor | None = None  # block-scaled weight gradients' workspace (moe_mx_dw_ws_bytes), on first use

    @staticmethod
    def allocate(T, d, E, n, K, m_tile=0, backward=True, dW_dtype=torch.bfloat16, device="cuda", capacity=0,
                 drop_policy="position", capacity_factor=0.0, e4m3=False, mx=False):
        """Buffers for one configuration; capacity > 0 (or capacity_factor > 0, giving
        ceil(capacity_factor * T * K / E)) selects the capacity (drop/pad) dispatch with that many slots per
        expert (pair-indexed arrays sized E * capacity)."""
        if capacity_factor and not capacity:
            capacity = expert_capacity(T, E, K, capacity_factor)
        if capacity and m_tile:
            raise ValueError("token rounding and the capacity dispatch are exclusive")
        cap = E * capacity if capacity else moe_pair_capacity(T, E, K, m_tile)
        f32, i32, bf = torch.float32, torch.int32, torch.bfloat16

        def z(shape, dt):
            return torch.zeros(shape, dtype=dt, device=device)

        ws_bytes = moe_capacity_workspace_bytes(T, d, E, n, K, capacity) if capacity else \
            moe_workspace_bytes(T, d, E, n, K, m_tile)
        if ws_bytes == 0:
            raise ValueError(f"unsupported sizes T={T} d={d} E={E} n={n} K={K}")
        return Buffers(
            T, d, E, n, K, m_tile, cap,
            logits=z((T, E), f32), scores=z((T, E), f32) if m_tile else None,
            topk_ids=z((T, K), i32), topk_w=z((T, K), f32), counts=z((E,), i32), offsets=z((E + 1,), i32),
            sorted_tok=z((cap,), i32), sorted_w=z((cap,), f32), tok_ptr=z((T + 1,), i32),
            tok_pairs=z((cap,), i32), P=z((1,), i32),
            H=z((cap, n), f32), U=z((cap, n), f32), A=z((cap, n), bf), Yw=z((cap, d), bf), O=z((T, d), bf),
            dX=z((T, d), bf) if backward else None,
            dW_gate=z((E, n, d), dW_dtype) if backward else None,
            dW_up=z((E, n, d), dW_dtype) if backward else None,
            dW_down=z((E, d, n), dW_dtype) if backward else None,
            dS=z((cap,), f32) if backward else None, dlogits=z((T, E), f32) if backward else None,
            dW_r=z((d, E), f32) if backward else None,
            ws=torch.empty(ws_bytes, dtype=torch.uint8, device=device), capacity=capacity, drop_policy=drop_policy,
            xq=z((T, d), torch.uint8) if e4m3 else None, xs=z((T,), f32) if e4m3 else None,
            aq=z((cap, n), torch.uint8) if e4m3 else None, as_=z((cap,), f32) if e4m3 else None,
            huq=z((cap, 2 * n), torch.uint8) if (e4m3 and backward) else None,
            hus=z((cap,), f32) if (e4m3 and backward) else None,
            doq=z((cap, d), torch.uint8) if (e4m3 and backward) else None,
            dos=z((cap,), f32) if (e4m3 and backward) else None,
            mxq=z((T, d), torch.uint8) if mx else None, mxsf=z((T, mx_sf_cols(d)), torch.uint8) if mx else None,
            maq=z((cap, n), torch.uint8) if mx else None,
            masf=z((mx_act_sf_bytes(cap, E, n),), torch.uint8) if mx else None,
            mxsft=z((mx_act_sf_bytes(cap, E, d),), torch.uint8) if mx else None,
            mdoq=z((cap, d), torch.uint8) if (mx and backward) else None,
            mdosft=z((mx_act_sf_bytes(cap, E, d),), torch.uint8) if (mx and backward) else None,
            mhuq=z((cap, 2 * n), torch.uint8) if (mx and backward) else None,
            mhusf=z((mx_act_sf_bytes(cap, E, 2 * n),), torch.uint8) if (mx and backward) else None)


def forward(ctx, X, W_r, bias, W_gate, W_up, W_down, buf: Buffers, stream=None, cache=True):
    """Routing, grouping, grouped GEMMs and combine; the output is ``buf.O``.  ``cache=False``: forward only,
    the pre-activations H, U the backward needs are not written."""
    moe_route(ctx, X, W_r, bias, buf.K, buf.logits, buf.scores, buf.topk_ids, buf.topk_w, buf.ws, stream)
    if buf.capacity:
        moe_permute_capacity(ctx, buf.topk_ids, buf.topk_w, buf.E, buf.capacity, buf.drop_policy, buf.counts,
                             buf.offsets, buf.sorted_tok, buf.sorted_w, buf.tok_ptr, buf.tok_pairs, buf.P, buf.ws,
                             stream)
    else:
        moe_permute(ctx, buf.topk_ids, buf.topk_w, buf.logits, buf.scores, buf.E, buf.m_tile, buf.counts,
                    buf.offsets, buf.sorted_tok, buf.sorted_w, buf.tok_ptr, buf.tok_pairs, buf.P, buf.ws, stream)
    moe_grouped_gemm_fwd(ctx, X, W_gate, W_up, W_down, buf.offsets, buf.sorted_tok, buf.sorted_w,
                         buf.H if cache else None, buf.U if cache else None, buf.A, buf.Yw, buf.ws, stream)
    moe_combine(ctx, buf.Yw, buf.tok_ptr, buf.tok_pairs, buf.O, stream)


@dataclass
class MxWeights:
    """The expert weights as block-scaled e4m3 (1 x 32 blocks along each row, power-of-two scales): codes
    Wg_q, Wu_q [E, n, d], Wd_q [E, d, n] (uint8) and the scale blocks the GEMMs read (gu_sf, dn_sf)."""

    Wg_q: torch.Tensor
    Wu_q: torch.Tensor
    gu_sf: torch.Tensor
    Wd_q: torch.Tensor
    dn_sf: torch.Tensor
    Wdt_q: torch.Tensor | None = None  # the backward: W_down^T codes [E, n, d] and scale blocks
    wdt_sf: torch.Tensor | None = None
    Wgu_q: torch.Tensor | None = None  # [W_gate; W_up]^T codes [E, d, 2n] and scale blocks
    wgu_sf: torch.Tensor | None = None

    @staticmethod
    def quantize(ctx, W_gate, W_up, W_down, stream=None, backward=False) -> "MxWeights":
        """The forward's codes and scale blocks; with ``backward`` also the two backward operands."""
        E, n, d = W_gate.shape
        dev = W_gate.device
        u8 = torch.uint8
        w = MxWeights(torch.empty((E, n, d), dtype=u8, device=dev), torch.empty((E, n, d), dtype=u8, device=dev),
                      torch.empty(mx_weight_sf_bytes(E, d, n, 0), dtype=u8, device=dev),
                      torch.empty((E, d, n), dtype=u8, device=dev),
                      torch.empty(mx_weight_sf_bytes(E, d, n, 1), dtype=u8, device=dev))
        moe_quantize_weights_mx(ctx, W_gate, W_up, W_down, w.Wg_q, w.Wu_q, w.gu_sf, w.Wd_q, w.dn_sf, stream)
        if backward:
            w.Wdt_q = torch.empty((E, n, d), dtype=u8, device=dev)
            w.wdt_sf = torch.empty(mx_weight_sf_bytes(E, d, n, 2), dtype=u8, device=dev)
            w.Wgu_q = torch.empty((E, d, 2 * n), dtype=u8, device=dev)
            w.wgu_sf = torch.empty(mx_weight_sf_bytes(E, d, n, 3), dtype=u8, device=dev)
            tmp = torch.empty((E, d, 2 * n), dtype=torch.bfloat16, device=dev)
            _check("moe_quantize_bwd_weights_mx", lib().moe_quantize_bwd_weights_mx(
                ctx.handle, _ptr(W_gate, torch.bfloat16), _ptr(W_up, torch.bfloat16), _ptr(W_down, torch.bfloat16),
                E, d, n, _ptr(tmp), _ptr(w.Wdt_q, u8), _ptr(w.wdt_sf, u8), _ptr(w.Wgu_q, u8), _ptr(w.wgu_sf, u8),
                _stream(stream)))
            torch.cuda.synchronize(dev)  # the scratch copy may go once the call has run
            del tmp
        return w


@dataclass
class E4m3Weights:
    """W_gate and W_up as e4m3 codes [E, n, d] (uint8) with one fp32 scale per output channel [E, n]; with
    W_down given, W_down as codes [E, d, n] with scales [E, d] too (the e4m3 down projection)."""

    Wg_q: torch.Tensor
    wg_scale: torch.Tensor
    Wu_q: torch.Tensor
    wu_scale: torch.Tensor
    Wd_q: torch.Tensor | None = None
    wd_scale: torch.Tensor | None = None
    Wgu_q: torch.Tensor | None = None  # the e4m3 dX GEMM: [W_gate; W_up]^T codes [E, d, 2n], scales [E, d]
    wgu_scale: torch.Tensor | None = None
    Wdt_q: torch.Tensor | None = None  # the e4m3 dSwiGLU GEMM: W_down^T codes [E, n, d], scales [E, n]
    wdt_scale: torch.Tensor | None = None

    @staticmethod
    def quantize(ctx, W_gate, W_up, W_down=None, stream=None, backward=False) -> "E4m3Weights":
        """The forward's codes (W_down's too when given); with ``backward`` also the two backward copies
        ([W_gate; W_up]^T for the dX GEMM, W_down^T for the dSwiGLU GEMM; W_down required)."""
        E, n, d = W_gate.shape
        dev = W_gate.device
        w = E4m3Weights(torch.empty((E, n, d), dtype=torch.uint8, device=dev),
                        torch.empty((E, n), dtype=torch.float32, device=dev),
                        torch.empty((E, n, d), dtype=torch.uint8, device=dev),
                        torch.empty((E, n), dtype=torch.float32, device=dev))
        moe_quantize_rows_e4m3(ctx, W_gate, w.Wg_q, w.wg_scale, stream)
        moe_quantize_rows_e4m3(ctx, W_up, w.Wu_q, w.wu_scale, stream)
        if W_down is not None:
            w.Wd_q = torch.empty((E, d, n), dtype=torch.uint8, device=dev)
            w.wd_scale = torch.empty((E, d), dtype=torch.float32, device=dev)
            moe_quantize_rows_e4m3(ctx, W_down, w.Wd_q, w.wd_scale, stream)
        if backward:
            if W_down is None:
                raise ValueError("the backward codes need W_down")
            w.Wgu_q = torch.empty((E, d, 2 * n), dtype=torch.uint8, device=dev)
            w.wgu_scale = torch.empty((E, d), dtype=torch.float32, device=dev)
            tmp = moe_quantize_dx_weights_e4m3(ctx, W_gate, W_up, w.Wgu_q, w.wgu_scale, stream)
            w.Wdt_q = torch.empty((E, n, d), dtype=torch.uint8, device=dev)
            w.wdt_scale = torch.empty((E, n), dtype=torch.float32, device=dev)
            tmp2 = moe_quantize_dact_weights_e4m3(ctx, W_down, w.Wdt_q, w.wdt_scale, stream)
            torch.cuda.synchronize(dev)  # the scratch copies may go once the calls have run
            del tmp, tmp2
        return w


def forward_e4m3(ctx, X, W_r, bias, w8: E4m3Weights, W_down, buf: Buffers, stream=None, cache=True):
    """The forward with the gate/up GEMM on e4m3 operands (``buf`` allocated with ``e4m3=True``): routing and
    grouping as ``forward``, X quantized per token, then the e4m3 grouped GEMMs and the combine.  When ``w8``
    holds W_down's codes the down projection runs on e4m3 operands too (``W_down`` may then be None).
    ``cache=False``: forward only (H, U not written)."""
    if buf.xq is None:
        raise ValueError("buffers were allocated without e4m3=True")
    moe_route(ctx, X, W_r, bias, buf.K, buf.logits, buf.scores, buf.topk_ids, buf.topk_w, buf.ws, stream)
    if buf.capacity:
        moe_permute_capacity(ctx, buf.topk_ids, buf.topk_w, buf.E, buf.capacity, buf.drop_policy, buf.counts,
                             buf.offsets, buf.sorted_tok, buf.sorted_w, buf.tok_ptr, buf.tok_pairs, buf.P, buf.ws,
                             stream)
    else:
        moe_permute(ctx, buf.topk_ids, buf.topk_w, buf.logits, buf.scores, buf.E, buf.m_tile, buf.counts,
                    buf.offsets, buf.sorted_tok, buf.sorted_w, buf.tok_ptr, buf.tok_pairs, buf.P, buf.ws, stream)
    moe_quantize_rows_e4m3(ctx, X, buf.xq, buf.xs, stream)
    moe_grouped_gemm_fwd_e4m3(ctx, buf.xq, buf.xs, w8.Wg_q, w8.wg_scale, w8.Wu_q, w8.wu_scale,
                              None if w8.Wd_q is not None else W_down, buf.offsets, buf.sorted_tok, buf.sorted_w,
                              buf.H if cache else None, buf.U if cache else None, buf.A, buf.Yw, Wd_q=w8.Wd_q,
                              wd_scale=w8.wd_scale,
                              Aq=buf.aq if w8.Wd_q is not None else None,
                              a_scale=buf.as_ if w8.Wd_q is not None else None, stream=stream)
    moe_combine(ctx, buf.Yw, buf.tok_ptr, buf.tok_pairs, buf.O, stream)


def forward_mx(ctx, X, W_r, bias, wmx: MxWeights, buf: Buffers, stream=None, cache=True):
    """The forward on block-scaled e4m3 operands (``buf`` allocated with ``mx=True``): routing and grouping as
    ``forward``, X quantized in 1 x 32 blocks, the gate/up GEMM (whose epilogue quantizes A), the down
    projection and the combine.  ``cache=False``: forward only (H, U not written)."""
    if buf.mxq is None:
        raise ValueError("buffers were allocated without mx=True")
    moe_route(ctx, X, W_r, bias, buf.K, buf.logits, buf.scores, buf.topk_ids, buf.topk_w, buf.ws, stream)
    if buf.capacity:
        moe_permute_capacity(ctx, buf.topk_ids, buf.topk_w, buf.E, buf.capacity, buf.drop_policy, buf.counts,
                             buf.offsets, buf.sorted_tok, buf.sorted_w, buf.tok_ptr, buf.tok_pairs, buf.P, buf.ws,
                             stream)
    else:
        moe_permute(ctx, buf.topk_ids, buf.topk_w, buf.logits, buf.scores, buf.E, buf.m_tile, buf.counts,
                    buf.offsets, buf.sorted_tok, buf.sorted_w, buf.tok_ptr, buf.tok_pairs, buf.P, buf.ws, stream)
    moe_quantize_rows_mx(ctx, X, buf.mxq, buf.mxsf, stream)
    moe_grouped_gemm_fwd_mx(ctx, buf.mxq, buf.mxsf, wmx, buf.offsets, buf.sorted_tok, buf.sorted_w,
                            buf.H if cache else None, buf.U if cache else None, buf.mxsft, buf.maq, buf.masf, buf.Yw,
                            stream)
    moe_combine(ctx, buf.Yw, buf.tok_ptr, buf.tok_pairs, buf.O, stream)


def backward_mx(ctx, dO, X, W_r, W_gate, W_up, W_down, wmx: MxWeights, buf: Buffers, stream=None, dw=False):
    """The backward with the dSwiGLU and dX GEMMs on block-scaled operands (``wmx`` quantized with
    ``backward=True``, ``buf`` allocated with ``mx=True``); with ``dw`` the weight gradients too (blocks of 32
    tokens of one expert), else they stay bf16 on dH, dU, A' rounded once to bf16.  The block-scaled weight
    gradients are slower on one GB300 (c2 step 1.20 against 0.94 ms): with short per-expert reductions the
    GEMMs are bound by per-tile work, not by the tensor cores, and their operands take a transposing
    quantization pass."""
    if wmx.Wdt_q is None or buf.mhuq is None:
        raise ValueError("block-scaled backward needs MxWeights.quantize(..., backward=True) and Buffers(mx=True)")
    T, d = X.shape
    E, n, _ = W_gate.shape
    cap = buf.sorted_tok.numel()
    wp, wb = _ws(buf.ws)
    bf, u8, f32, i32 = torch.bfloat16, torch.uint8, torch.float32, torch.int32
    dw_fp32 = 1 if buf.dW_gate.dtype == f32 else 0
    if dw and buf.mdw is None:
        buf.mdw = torch.empty(mx_dw_ws_bytes(d, E, n, cap), dtype=u8, device=dO.device)
    _check("moe_backward_mx", lib().moe_backward_mx(
        ctx.handle, _ptr(dO, bf), _ptr(X, bf), _ptr(W_r, bf), _ptr(W_gate, bf), _ptr(W_up, bf), _ptr(W_down, bf),
        _ptr(wmx.Wdt_q, u8), _ptr(wmx.wdt_sf, u8), _ptr(wmx.Wgu_q, u8), _ptr(wmx.wgu_sf, u8), T, d, E, n, buf.K,
        buf.m_tile, cap, _ptr(buf.topk_ids, i32), _ptr(buf.topk_w, f32), _ptr(buf.offsets, i32),
        _ptr(buf.sorted_tok, i32), _ptr(buf.sorted_w, f32), _ptr(buf.tok_ptr, i32), _ptr(buf.tok_pairs, i32),
        _ptr(buf.H, f32), _ptr(buf.U, f32), _ptr(buf.mdoq, u8), _ptr(buf.mdosft, u8), _ptr(buf.mhuq, u8),
        _ptr(buf.mhusf, u8), _ptr(buf.dX, bf), _ptr(buf.dW_gate), _ptr(buf.dW_up), _ptr(buf.dW_down), dw_fp32,
        _ptr(buf.dS, f32), _ptr(buf.dlogits, f32), _ptr(buf.dW_r, f32), wp, wb,
        _ptr(buf.mdw, u8) if dw else None, buf.mdw.numel() if dw else 0, _stream(stream)))


def backward_e4m3(ctx, dO, X, W_r, W_gate, W_up, W_down, w8: E4m3Weights, buf: Buffers, stream=None, dx=True,
                  dact=True):
    """The backward with the dX GEMM (``dx``) and the dSwiGLU GEMM (``dact``) on e4m3 operands (``w8`` quantized
    with ``backward=True``, ``buf`` allocated with ``e4m3=True``); the weight gradients stay bf16, on dH, dU and
    A' rounded once to bf16.  Measured on one GB300, the e4m3 training step is faster than bf16 by 1.55x at
    d = 7168, n = 2048, 1.23x at d = 2048, n = 512 and 1.07x at d = 1536, n = 256 (where the per-row
    quantization passes take most of what the shorter GEMMs save)."""
    if w8.Wgu_q is None or buf.huq is None:
        raise ValueError("e4m3 backward needs E4m3Weights.quantize(..., backward=True) and Buffers(e4m3=True)")
    moe_backward_e4m3(ctx, dO, X, W_r, W_gate, W_up, W_down, w8.Wgu_q if dx else None, w8.wgu_scale if dx else None,
                      w8.Wdt_q if dact else None, w8.wdt_scale if dact else None, buf.K, buf.m_tile, buf.topk_ids,
                      buf.topk_w, buf.offsets, buf.sorted_tok, buf.sorted_w, buf.tok_ptr, buf.tok_pairs, buf.H, buf.U,
                      buf.huq if dx else None, buf.hus if dx else None, buf.doq if dact else None,
                      buf.dos if dact else None, buf.dX, buf.dW_gate, buf.dW_up, buf.dW_down, buf.dS, buf.dlogits,
                      buf.dW_r, buf.ws, stream)


def backward(ctx, dO, X, W_r, W_gate, W_up, W_down, buf: Buffers, stream=None):
    moe_backward(ctx, dO, X, W_r, W_gate, W_up, W_down, buf.K, buf.m_tile, buf.topk_ids, buf.topk_w, buf.offsets,
                 buf.sorted_tok, buf.sorted_w, buf.tok_ptr, buf.tok_pairs, buf.H, buf.U, buf.dX, buf.dW_gate,
                 buf.dW_up, buf.dW_down, buf.dS, buf.dlogits, buf.dW_r, buf.ws, stream)


class StepGraph:
    """One forward + backward (``backward=False``: the forward) captured as a CUDA graph for fixed tensors and
    buffers.  The library's host work (argument checks, tensor-map encoding, launch configuration) runs once, at
    capture; ``replay()`` launches the whole step at once on the current stream.  New inputs are copied into the
    captured tensors (same addresses) before a replay; outputs land in ``buf`` as with the eager calls."""

    def __init__(self, ctx, X, W_r, bias, W_gate, W_up, W_down, dO, buf: Buffers, backward=True):
        def run():
            if backward:
                forward_backward(ctx, X, W_r, bias, W_gate, W_up, W_down, dO, buf)
            else:
                forward(ctx, X, W_r, bias, W_gate, W_up, W_down, buf)
        side = torch.cuda.Stream(device=X.device)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):  # one eager pass outside the capture (first-use configuration)
            run()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize(X.device)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            run()
        torch.cuda.synchronize(X.device)

    def replay(self):
        self.graph.replay()


def forward_backward(ctx, X, W_r, bias, W_gate, W_up, W_down, dO, buf: Buffers, stream=None):
    forward(ctx, X, W_r, bias, W_gate, W_up, W_down, buf, stream)
    backward(ctx, dO, X, W_r, W_gate, W_up, W_down, buf, stream)
