"""The C-ABI library builds for sm_103a, loads, and exports every symbol include/moe.h declares (CPU only)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s*]*?\b(moe_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def libpath():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from varlen_grouped_gemm_gb300 import build
    return build.build()


def test_header_declares_the_five_entry_points():
    names = _declared()
    for n in ("moe_route", "moe_permute", "moe_grouped_gemm_fwd", "moe_combine", "moe_backward"):
        assert n in names


def test_library_exports_every_declared_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing
    import varlen_grouped_gemm_gb300 as vgg
    assert set(vgg.EXPORTS) == set(_declared())


def test_host_only_queries(libpath):
    import varlen_grouped_gemm_gb300 as vgg
    assert vgg.moe_pair_capacity(4096, 128, 8, 0) == 4096 * 8
    assert vgg.moe_pair_capacity(32768, 512, 8, 128) == 32768 * 8 + 512 * 64
    assert vgg.moe_workspace_bytes(4096, 2048, 128, 512, 8, 0) > 0
    assert vgg.moe_workspace_bytes(4096, 2000, 128, 512, 8, 0) == 0  # d not a multiple of 64
    assert vgg.status_str(vgg.MOE_ERR_INVALID_ARG) == "invalid argument"


def test_block_scale_size_queries(libpath):
    """The block-scaled form's scale layouts, by their stated shapes: 4 bytes per 128 columns of a row-major
    array; pairs of 512-byte blocks per 192-row tile (96 + 96 rows for the gate/up pair) and 128 columns of the
    reduction for the weights; one block per 128-row tile (at most cap / 128 + E tiles) and 128 columns for
    the activations."""
    import varlen_grouped_gemm_gb300 as vgg
    L = vgg.lib()
    assert [L.moe_mx_sf_cols(c) for c in (64, 128, 2048, 2880, 0)] == [4, 4, 64, 92, 0]
    E, d, n = 128, 2048, 512
    assert L.moe_mx_weight_sf_bytes(E, d, n, 0) == 1024 * E * 6 * 16       # ceil(512 / 96) tiles, 2048 / 128 stages
    assert L.moe_mx_weight_sf_bytes(E, d, n, 1) == 1024 * E * 11 * 4       # ceil(2048 / 192) tiles, 512 / 128
    assert L.moe_mx_weight_sf_bytes(E, d, n, 2) == 1024 * E * 3 * 16       # W_down^T: ceil(512 / 192), 2048 / 128
    assert L.moe_mx_weight_sf_bytes(E, d, n, 3) == 1024 * E * 11 * 8       # [W_gate; W_up]^T: 1024 / 128 stages
    assert L.moe_mx_weight_sf_bytes(E, 2000, n, 0) == 0 and L.moe_mx_weight_sf_bytes(E, d, n, 4) == 0
    assert L.moe_mx_act_sf_bytes(32768, 128, 512) == 512 * (256 + 128) * 4
    assert L.moe_mx_act_sf_bytes(100, 3, 2880) == 512 * (1 + 3) * 23
    assert L.moe_mx_act_sf_bytes(0, 3, 64) == 0


def test_block_scaled_weight_gradient_workspace_size(libpath):
    """moe_mx_dw_ws_bytes by the stated layout: the stage offsets, the four K-major code matrices over the
    padded reduction (cap + 127 E tokens rounded up to 128) and their scale blocks, each region 256-aligned."""
    import varlen_grouped_gemm_gb300 as vgg
    L = vgg.lib()
    al = lambda x: (x + 255) // 256 * 256

    def want(d, E, n, cap, bn_gu, bn_dn):
        kq = -(-(cap + 127 * E) // 128) * 128
        kst = kq // 128
        codes = al(2 * n * kq) + al(d * kq) + al(d * kq) + al(n * kq)
        blocks = (al(512 * kst * -(-2 * n // 128)) + al(512 * kst * -(-d // bn_gu) * -(-bn_gu // 128)) +
                  al(512 * kst * -(-d // 128)) + al(512 * kst * -(-n // bn_dn) * -(-bn_dn // 128)))
        return al(4 * (E + 1)) + codes + blocks

    assert L.moe_mx_dw_ws_bytes(2048, 128, 512, 32768) == want(2048, 128, 512, 32768, 192, 192)
    assert L.moe_mx_dw_ws_bytes(1536, 512, 256, 32768 * 8 + 512 * 64) == want(1536, 512, 256, 294912, 192, 128)
    assert L.moe_mx_dw_ws_bytes(2880, 128, 2880, 32768) == want(2880, 128, 2880, 32768, 192, 192)
    for bad in ((2000, 8, 64, 100), (64, 0, 64, 100), (64, 8, 64, 0), (64, 2000, 64, 100)):
        assert L.moe_mx_dw_ws_bytes(*bad) == 0, bad


def test_expert_capacity_matches_the_oracle(libpath):
    """The capacity dispatch's slot count C = ceil(cf T K / E) comes from the library (the binding does no
    arithmetic); it equals the oracle's reading on a grid that includes exact multiples and fractions."""
    import varlen_grouped_gemm_gb300 as vgg
    from oracle import moe_oracle as mo
    for T in (1, 5, 10, 4096, 8192, 65536):
        for E in (3, 4, 8, 128, 512):
            for K in (1, 2, 8):
                for cf in (0.5, 1.0, 1.25, 2.0, 1.0 / 3.0, 0.1):
                    assert vgg.expert_capacity(T, E, K, cf) == mo.expert_capacity(T, E, K, cf), (T, E, K, cf)
    assert vgg.lib().moe_expert_capacity(4096, 128, 8, 1.0) == 256
    for bad in ((0, 8, 2, 1.0), (16, 0, 2, 1.0), (16, 8, 0, 1.0), (16, 8, 2, 0.0), (16, 8, 2, -1.0),
                (16, 8, 2, float("nan"))):
        assert vgg.lib().moe_expert_capacity(*bad) == 0, bad


def test_argument_errors_are_reported_without_a_device(libpath):
    lib = ctypes.CDLL(libpath)
    lib.moe_route.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 4 + [ctypes.c_void_p] * 5 + \
        [ctypes.c_size_t, ctypes.c_void_p]
    assert lib.moe_route(None, None, None, None, 1, 64, 8, 2, None, None, None, None, None, 0, None) == 1


# Every entry point that takes a context checks its arguments before any device work: a NULL context (all
# other arguments zero) is MOE_ERR_INVALID_ARG, with or without a GPU.
_CTX_ENTRIES = ["moe_route", "moe_permute", "moe_grouped_gemm_fwd", "moe_combine", "moe_backward",
                "moe_permute_noalloc", "moe_permute_capacity", "moe_quantize_rows_e4m3", "moe_grouped_gemm_fwd_e4m3",
                "moe_quantize_dx_weights_e4m3", "moe_quantize_dact_weights_e4m3", "moe_backward_e4m3",
                "moe_test_gemm_varlen_m", "moe_test_gemm_varlen_k", "moe_test_gemm_varlen_k_dual",
                "moe_test_gemm_varlen_m_dual", "moe_quantize_rows_mx", "moe_quantize_weights_mx",
                "moe_grouped_gemm_fwd_mx", "moe_quantize_bwd_weights_mx", "moe_backward_mx"]


@pytest.mark.parametrize("name", _CTX_ENTRIES)
def test_null_context_is_an_argument_error(libpath, name):
    import varlen_grouped_gemm_gb300 as vgg
    fn = getattr(vgg.lib(), name)
    args = [None if t in (ctypes.c_void_p, ctypes.c_char_p) else 0 for t in fn.argtypes]
    assert fn.argtypes[0] is ctypes.c_void_p
    assert fn(*args) == vgg.MOE_ERR_INVALID_ARG
