"""Grouped-GEMM main loops on integer-valued bf16 operands: every product and partial sum is an
integer below 2^24, so fp32 accumulation is exact in any order and the device result must equal the
int64 reference bit for bit.  This pins the gather, the varlen bookkeeping (empty, one-row and
ragged groups, ragged N), both operand layouts (K-major and MN-major), the two-part A operand and
transposed store of the weight-gradient GEMMs, the CTA-pair form of the tiled GEMMs (two CTAs per
256-row tile, M = 256 UMMAs), and the bounded wait."""
import contextlib

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import varlen_grouped_gemm_gb300 as vgg
    return vgg.Context(0)


def _ints(shape, lo, hi, seed):
    return np.random.default_rng(seed).integers(lo, hi + 1, size=shape).astype(np.int64)


def _bf(a):
    return torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).cuda()


@contextlib.contextmanager
def _cta_pairs(ctx, on):
    """CTA pairs for both GEMM families while the block runs (off is the default)."""
    ctx.set_cta_pairs(on, on)
    try:
        yield
    finally:
        ctx.set_cta_pairs(False, False)


@pytest.mark.parametrize("gathered,pairs", [(True, False), (False, False), (False, True)])
@pytest.mark.parametrize("b_kmajor", [True, False])
@pytest.mark.parametrize("sizes,K,N", [([0, 1, 130, 257, 64], 192, 200), ([300], 64, 136), ([5, 0, 0, 129], 128, 264)])
def test_varlen_m_exact(ctx, gathered, pairs, b_kmajor, sizes, K, N):
    """pairs: CTA pairs on 256 x 256 tiles; a group's odd CTA may hold rows past the group (or no rows at
    all), which it must neither store nor let into the even CTA's rows."""
    import varlen_grouped_gemm_gb300 as vgg
    G = len(sizes)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    P = int(offsets[-1])
    cap = P + 7
    rows_a = P + 40 if gathered else cap
    A = _ints((rows_a, K), -2, 2, 1)
    idx = np.random.default_rng(2).permutation(rows_a)[:cap].astype(np.int32) if gathered else None
    if not b_kmajor:
        N -= N % 64  # the MN-major operand is read in 64-column chunks
    Bk = _ints((G, N, K), -1, 1, 3)  # [G, N, K]
    B = Bk if b_kmajor else np.ascontiguousarray(Bk.transpose(0, 2, 1))
    D = torch.full((cap, N), -7.0, device="cuda")
    with _cta_pairs(ctx, pairs):
        vgg.moe_test_gemm_varlen_m(ctx, _bf(A), None if idx is None else torch.from_numpy(idx).cuda(), _bf(B),
                                   b_kmajor, torch.from_numpy(offsets).cuda(), D)
    rc, code = vgg.moe_get_error(ctx)
    assert rc == 0 and code == 0
    got = D.cpu().numpy()
    for e in range(G):
        for j in range(offsets[e], offsets[e + 1]):
            row = idx[j] if gathered else j
            np.testing.assert_array_equal(got[j], (A[row] @ Bk[e].T).astype(np.float32), err_msg=f"e={e} j={j}")
    assert np.all(got[P:] == -7.0), "rows outside every group must stay untouched"


@pytest.mark.parametrize("sizes,M,N", [([0, 5, 64, 200], 192, 192), ([1, 0, 333], 128, 256), ([70], 64, 320)])
@pytest.mark.parametrize("gathered", ["a", "b", "none"])
def test_varlen_k_exact(ctx, sizes, M, N, gathered):
    """D[e] = sum over the group's rows j of A[rowa(j)]^T B[rowb(j)]; one operand is gathered through an
    index (zero past the group's end), the other is read by sorted position (it runs into the next
    group's rows, which the zero-filled gathered rows cancel)."""
    import varlen_grouped_gemm_gb300 as vgg
    G = len(sizes)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    P = int(offsets[-1])
    cap = P + 3
    Tsrc = P + 17
    idx = np.random.default_rng(6).integers(0, Tsrc, size=cap).astype(np.int32)
    if gathered == "a":
        A, B = _ints((Tsrc, M), -2, 2, 4), _ints((cap, N), -2, 2, 5)
        idx_a, idx_b = torch.from_numpy(idx).cuda(), None
    elif gathered == "b":
        A, B = _ints((cap, M), -2, 2, 4), _ints((Tsrc, N), -2, 2, 5)
        idx_a, idx_b = None, torch.from_numpy(idx).cuda()
    else:
        A, B = _ints((cap, M), -2, 2, 4), _ints((cap, N), -2, 2, 5)
        idx_a, idx_b = None, None
    D = torch.full((G, M, N), 3.0, device="cuda")
    vgg.moe_test_gemm_varlen_k(ctx, _bf(A), idx_a, _bf(B), idx_b, torch.from_numpy(offsets).cuda(), D, cap)
    rc, code = vgg.moe_get_error(ctx)
    assert rc == 0 and code == 0
    got = D.cpu().numpy()
    for e in range(G):
        rows = np.arange(offsets[e], offsets[e + 1])
        ra = idx[rows] if gathered == "a" else rows
        rb = idx[rows] if gathered == "b" else rows
        np.testing.assert_array_equal(got[e], (A[ra].T @ B[rb]).astype(np.float32), err_msg=f"group {e}")


@pytest.mark.parametrize("pairs", [False, True])
@pytest.mark.parametrize("sizes,K,N", [([0, 1, 130, 257, 64], 192, 200), ([300], 64, 512), ([5, 0, 0, 129], 128, 264)])
def test_varlen_m_dual_exact(ctx, pairs, sizes, K, N):
    """The down projection's form: per sorted row, (A_hi + A_lo) B[e]^T with two UMMAs per K step into one
    accumulator; A_lo holds small integers times 2^-8 so that a dropped or misplaced low-part product shows."""
    import varlen_grouped_gemm_gb300 as vgg
    G = len(sizes)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    P = int(offsets[-1])
    cap = P + 7
    A_hi = _ints((cap, K), -2, 2, 11).astype(np.float64)
    A_lo = _ints((cap, K), -3, 3, 12).astype(np.float64) / 256.0
    B = _ints((G, N, K), -1, 1, 13).astype(np.float64)
    D = torch.full((cap, N), -7.0, device="cuda")
    with _cta_pairs(ctx, pairs):
        vgg.moe_test_gemm_varlen_m_dual(ctx, _bf(A_hi), _bf(A_lo), _bf(B), torch.from_numpy(offsets).cuda(), D)
    rc, code = vgg.moe_get_error(ctx)
    assert rc == 0 and code == 0
    got = D.cpu().numpy()
    for e in range(G):
        lo, hi = offsets[e], offsets[e + 1]
        ref = ((A_hi[lo:hi] + A_lo[lo:hi]) @ B[e].T).astype(np.float32)
        np.testing.assert_array_equal(got[lo:hi], ref, err_msg=f"group {e}")
    assert np.all(got[P:] == -7.0), "rows outside every group must stay untouched"


@pytest.mark.parametrize("sizes,M,N", [([0, 5, 64, 200], 192, 192), ([1, 0, 333], 128, 256), ([70], 64, 320),
                                         ([17] * 9 + [0, 130], 320, 512), ([300, 0, 17], 128, 4096)])
@pytest.mark.parametrize("trans", [False, True])
@pytest.mark.parametrize("padded,pairs", [(False, False), (True, False), (True, True)])
def test_varlen_k_dual_exact(ctx, sizes, M, N, trans, padded, pairs):
    """The weight-gradient form: per group, (A_hi + A_lo)^T B over the group's rows, two UMMAs per K step into
    one accumulator; B's rows past a group's end are cleared in shared memory.  A_lo holds small integers
    times 2^-8 (exact in bf16) so that a dropped or misplaced low-part product changes the result.  With
    trans the tile leaves through transposed 32 x 32 blocks: D[e] is the transpose.  padded: B in the layout of
    the backward's sorted copies, every group followed by zero rows up to a multiple of 16 (no clearing)."""
    import varlen_grouped_gemm_gb300 as vgg
    G = len(sizes)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    P = int(offsets[-1])
    cap = P + 3
    A_hi = _ints((cap, M), -2, 2, 7).astype(np.float64)
    A_lo = _ints((cap, M), -3, 3, 8).astype(np.float64) / 256.0
    B = _ints((cap, N), -2, 2, 9).astype(np.float64)
    shape = (G, N, M) if trans else (G, M, N)
    D = torch.full(shape, 3.0, device="cuda")
    b_off = None
    Bdev = B
    if padded:
        poff = np.concatenate([[0], np.cumsum((np.array(sizes) + 15) // 16 * 16)]).astype(np.int32)
        Bdev = np.zeros((int(poff[-1]) + 64, N))  # a few rows past the last group stay zero too
        for e in range(G):
            Bdev[poff[e]:poff[e] + sizes[e]] = B[offsets[e]:offsets[e + 1]]
        b_off = torch.from_numpy(poff).cuda()
    with _cta_pairs(ctx, pairs):
        vgg.moe_test_gemm_varlen_k_dual(ctx, _bf(A_hi), _bf(A_lo), _bf(Bdev), torch.from_numpy(offsets).cuda(), D,
                                        cap, trans=trans, b_offsets=b_off)
    rc, code = vgg.moe_get_error(ctx)
    assert rc == 0 and code == 0
    got = D.cpu().numpy()
    for e in range(G):
        rows = np.arange(offsets[e], offsets[e + 1])
        ref = ((A_hi[rows] + A_lo[rows]).T @ B[rows]).astype(np.float32)  # multiples of 2^-8 below 2^15: exact
        np.testing.assert_array_equal(got[e], ref.T if trans else ref, err_msg=f"group {e}")


def test_bounded_wait_times_out_and_context_survives(ctx):
    import varlen_grouped_gemm_gb300 as vgg
    vgg.moe_test_wait_timeout(ctx, 2_000_000)  # 2 ms
    rc, code = vgg.moe_get_error(ctx)
    assert rc == vgg.MOE_ERR_DEVICE_TIMEOUT and code == vgg.DEV_TIMEOUT
    # the context keeps working afterwards
    offsets = torch.tensor([0, 3], dtype=torch.int32, device="cuda")
    A = _bf(np.ones((3, 64)))
    B = _bf(np.ones((1, 8, 64)))
    D = torch.zeros((3, 8), device="cuda")
    vgg.moe_test_gemm_varlen_m(ctx, A, None, B, True, offsets, D)
    assert vgg.moe_get_error(ctx) == (0, 0)
    assert torch.all(D == 64.0)


def test_corrupt_offsets_are_reported_not_trapped(ctx):
    import varlen_grouped_gemm_gb300 as vgg
    offsets = torch.tensor([0, 5, 2], dtype=torch.int32, device="cuda")  # not monotone
    A = _bf(np.ones((8, 64)))
    B = _bf(np.ones((2, 8, 64)))
    D = torch.zeros((8, 8), device="cuda")
    vgg.moe_test_gemm_varlen_m(ctx, A, None, B, True, offsets, D)
    rc, code = vgg.moe_get_error(ctx)
    assert rc == vgg.MOE_ERR_DEVICE and code == vgg.DEV_BAD_OFFSETS
    assert torch.all(D == 0)
