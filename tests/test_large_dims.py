"""Large dimensions: a million rows, a million columns, a million-deep K.

Index arithmetic that is right at test sizes can overflow or wrap at these
(row x pitch products, tile counts past 2^16, K-tile counters, TMA
coordinates).  Operands are small integers, so every partial sum is exact in
fp32 and each sampled element must equal the oracle's bit for bit; the
samples include the first and last rows and columns and every tile edge near
the end of each dimension."""
import numpy as np
import pytest
import torch

import dense_gemm_blackwell_tcgen05_gb300 as g
import gemm_inputs as gi
import oracle
from tests import parity as P

pytestmark = pytest.mark.gpu


def _ints(rows, cols, seed, lo=-2, hi=3):
    gen = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi, (rows, cols), generator=gen, dtype=torch.int8)


def _positions(M, N, seed, n=2000):
    rng = np.random.default_rng(seed)
    rows = list(rng.integers(0, M, n))
    cols = list(rng.integers(0, N, n))
    for r in (0, 1, M - 257, M - 256, M - 129, M - 128, M - 2, M - 1):
        if 0 <= r < M:
            for c in (0, N - 1, int(rng.integers(0, N))):
                rows.append(r)
                cols.append(c)
    for c in (0, N - 257, N - 256, N - 129, N - 128, N - 2, N - 1):
        if 0 <= c < N:
            for r in (0, M - 1, int(rng.integers(0, M))):
                rows.append(r)
                cols.append(c)
    return np.array(rows, np.int64), np.array(cols, np.int64)


def _check(D, A_codes, B_codes, K, seed, what):
    M, N = D.shape
    rows, cols = _positions(M, N, seed)
    D_ref, _ = oracle.gemm_bf16_entries(A_codes, B_codes, rows, cols, K)
    got = gi.bf16_codes(D[torch.from_numpy(rows), torch.from_numpy(cols)].contiguous())
    want = oracle.f64_to_bf16_rne(D_ref)
    bad = np.flatnonzero(got != want)
    assert len(bad) == 0, f"{what}: {len(bad)} of {len(rows)} sampled elements differ, " \
                          f"first at ({rows[bad[0]]}, {cols[bad[0]]})"


@pytest.mark.parametrize("v", [g.VARIANT_AUTO, g.VARIANT_1CTA, g.VARIANT_2CTA | g.VARIANT_DIRECT_STORE])
@pytest.mark.parametrize("shape", [(1 << 20 | 1, 40, 64), (24, 1 << 20 | 3, 64), (128, 136, 1 << 20)],
                         ids=["million_rows", "million_cols", "million_k"])
def test_bf16_large_dims(v, shape):
    M, N, K = shape
    A = _ints(M, K, 1).to(torch.bfloat16)
    B = _ints(N, K, 2).to(torch.bfloat16)
    Ad, Bd = A.cuda(), B.cuda()
    ldd = N + 8
    Dbuf = torch.full((M, ldd), float("nan"), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_bf16_variant(v, Ad.data_ptr(), Bd.data_ptr(), Dbuf.data_ptr(), M, N, K, K, K, ldd, s)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    assert g.gemm_last_status(s) == g.GEMM_OK
    Dall = Dbuf.cpu()
    assert torch.isnan(Dall[:, N:].float()).all(), "pitch padding written"
    _check(Dall[:, :N], gi.bf16_codes(A), gi.bf16_codes(B), K, M + N, f"bf16 {shape} v{v}")


def test_smallk_million_rows():
    M, N, K = 1 << 22, 24, 8
    A = _ints(M, K, 3).to(torch.bfloat16)
    B = _ints(N, K, 4).to(torch.bfloat16)
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_bf16_variant(g.VARIANT_AUTO, Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K,
                             K, K, N, s)
    assert rc == g.GEMM_OK and g.gemm_last_status(s) == g.GEMM_OK
    _check(D.cpu(), gi.bf16_codes(A), gi.bf16_codes(B), K, 7, "small K, 4M rows")


@pytest.mark.parametrize("tiled", [False, True], ids=["row_major_scales", "tiled_scales"])
@pytest.mark.parametrize("shape", [(1 << 20 | 1, 40, 128), (136, 136, 1 << 19)],
                         ids=["million_rows", "half_million_k"])
def test_mxfp8_large_dims(tiled, shape):
    """Integer E4M3 values in [-2, 2] with scale byte 127 (2^0): exact sums."""
    M, N, K = shape
    A8 = _ints(M, K, 5)
    B8 = _ints(N, K, 6)
    A = P.e4m3_from_ints(A8.numpy().astype(np.int64))
    B = P.e4m3_from_ints(B8.numpy().astype(np.int64))
    pitch = gi.sf_pitch(K)
    SFA = torch.full((M, pitch), 127, dtype=torch.uint8)
    SFB = torch.full((N, pitch), 127, dtype=torch.uint8)
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    Ad, Bd = A.cuda(), B.cuda()
    if tiled:
        SAd, SBd = gi.tile_scales(SFA, M, K).cuda(), gi.tile_scales(SFB, N, K).cuda()
        rc = g.gemm_mxfp8_tiled(g.VARIANT_AUTO, Ad.data_ptr(), Bd.data_ptr(), SAd.data_ptr(),
                                SBd.data_ptr(), D.data_ptr(), M, N, K, K, K, N, s)
    else:
        SAd, SBd = SFA.cuda(), SFB.cuda()
        rc = g.gemm_mxfp8_variant(g.VARIANT_AUTO, Ad.data_ptr(), Bd.data_ptr(), SAd.data_ptr(),
                                  SBd.data_ptr(), D.data_ptr(), M, N, K, K, K, pitch, pitch, N, s)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    assert g.gemm_last_status(s) == g.GEMM_OK
    rows, cols = _positions(M, N, K)
    D_ref, _ = oracle.gemm_mxfp8_entries(A.numpy(), B.numpy(), SFA.numpy(), SFB.numpy(), rows, cols, K)
    got = gi.bf16_codes(D.cpu()[torch.from_numpy(rows), torch.from_numpy(cols)].contiguous())
    want = oracle.f64_to_bf16_rne(D_ref)
    bad = np.flatnonzero(got != want)
    assert len(bad) == 0, f"mxfp8 {shape} tiled={tiled}: {len(bad)} sampled elements differ"
