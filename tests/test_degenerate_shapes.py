"""Degenerate shapes on every kernel variant: a single row or column of D, a
1x1 output, K = 1 and K far below one K-tile.  Operands are small integers
(and power-of-two scales for MXFP8) so that every partial sum is exact in
fp32 and the result must match the oracle bit for bit.  The output pitch is
wider than N and pre-filled with NaN, and one extra row below D too: neither
may be written."""
import numpy as np
import pytest
import torch

import dense_gemm_blackwell_tcgen05_gb300 as g
import gemm_inputs as gi
import oracle
from tests import parity as P
from tests.test_gemm_mxfp8 import int_operands

pytestmark = pytest.mark.gpu

BF16_VARIANTS = {
    "1cta": g.VARIANT_1CTA,
    "2cta": g.VARIANT_2CTA,
    "sync": g.VARIANT_SYNC,
    "1cta_direct": g.VARIANT_1CTA | g.VARIANT_DIRECT_STORE,
    "2cta_direct": g.VARIANT_2CTA | g.VARIANT_DIRECT_STORE,
    "smallk": g.VARIANT_SMALLK,
    "smallk_tc": g.VARIANT_SMALLK_TC,
    "auto": g.VARIANT_AUTO,
}
MX_VARIANTS = {
    "1cta": g.VARIANT_1CTA,
    "1cta_direct": g.VARIANT_1CTA | g.VARIANT_DIRECT_STORE,
    "2cta": g.VARIANT_2CTA,
    "auto": g.VARIANT_AUTO,
}
BF16_SHAPES = [(1, 300, 200), (300, 1, 200), (1, 1, 1), (2, 3, 70), (1, 257, 4096), (257, 1, 1),
               (1, 1, 4096), (130, 2, 16)]
MX_SHAPES = [(1, 300, 256), (300, 1, 96), (1, 1, 32), (3, 2, 1), (1, 257, 4096), (130, 2, 40)]


def _guarded_output(M, N):
    """D with pitch N + 8 and one extra row, all NaN; returns (buffer, ldd)."""
    ldd = N + 8
    return torch.full((M + 1, ldd), float("nan"), dtype=torch.bfloat16, device="cuda"), ldd


def _check(Dbuf, M, N, D_ref):
    got_all = Dbuf.cpu()
    got = gi.bf16_codes(got_all[:M, :N].contiguous())
    want = oracle.f64_to_bf16_rne(D_ref)
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        raise AssertionError(f"{len(bad)} mismatches; first at {tuple(bad[0])}")
    assert torch.isnan(got_all[:M, N:].float()).all(), "pitch padding written"
    assert torch.isnan(got_all[M].float()).all(), "row below D written"


@pytest.mark.parametrize("v", list(BF16_VARIANTS))
@pytest.mark.parametrize("shape", BF16_SHAPES)
def test_bf16_degenerate(v, shape):
    M, N, K = shape
    if v in ("smallk", "smallk_tc") and K > 16:
        pytest.skip("the small-K kernel takes K <= 16")
    lda = (K + 7) // 8 * 8          # a 16-byte row pitch
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    A = torch.zeros(M, lda, dtype=torch.bfloat16)
    B = torch.zeros(N, lda, dtype=torch.bfloat16)
    A[:, :K] = P.bf16_from_ints(rng.integers(-2, 3, size=(M, K)))
    B[:, :K] = P.bf16_from_ints(rng.integers(-2, 3, size=(N, K)))
    Dbuf, ldd = _guarded_output(M, N)
    Ad, Bd = A.cuda(), B.cuda()
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_bf16_variant(BF16_VARIANTS[v], Ad.data_ptr(), Bd.data_ptr(), Dbuf.data_ptr(), M, N,
                             K, lda, lda, ldd, s)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    assert g.gemm_last_status(s) == g.GEMM_OK
    D_ref, _ = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B), K)
    _check(Dbuf, M, N, D_ref)


@pytest.mark.parametrize("v", list(MX_VARIANTS))
@pytest.mark.parametrize("shape", MX_SHAPES)
def test_mxfp8_degenerate(v, shape):
    M, N, K = shape
    lda = (K + 15) // 16 * 16       # a 16-byte row pitch
    A, SFA, B, SFB = int_operands(M, N, K, seed=M * 5 + N + K, lda=lda)
    Dbuf, ldd = _guarded_output(M, N)
    Ad, Bd, SAd, SBd = (t.cuda() for t in (A, B, SFA, SFB))
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_mxfp8_variant(MX_VARIANTS[v], Ad.data_ptr(), Bd.data_ptr(), SAd.data_ptr(),
                              SBd.data_ptr(), Dbuf.data_ptr(), M, N, K, lda, lda, SFA.shape[1],
                              SFB.shape[1], ldd, s)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    assert g.gemm_last_status(s) == g.GEMM_OK
    D_ref, _ = oracle.gemm_mxfp8(A.numpy(), B.numpy(), SFA.numpy(), SFB.numpy(), K)
    _check(Dbuf, M, N, D_ref)


TILED_VARIANTS = {
    "auto": g.VARIANT_AUTO,
    "1cta": g.VARIANT_1CTA,
    "2cta": g.VARIANT_2CTA,
    "2cta_direct": g.VARIANT_2CTA | g.VARIANT_DIRECT_STORE,
}


@pytest.mark.parametrize("v", list(TILED_VARIANTS))
@pytest.mark.parametrize("shape", MX_SHAPES)
def test_mxfp8_tiled_degenerate(v, shape):
    """The same shapes through gemm_mxfp8_tiled: scales rearranged into the
    tiled layout (zero-padded to whole 128-row blocks and 4-block groups)."""
    M, N, K = shape
    lda = (K + 15) // 16 * 16
    A, SFA, B, SFB = int_operands(M, N, K, seed=M * 5 + N + K, lda=lda)
    Dbuf, ldd = _guarded_output(M, N)
    Ad, Bd = A.cuda(), B.cuda()
    SAt, SBt = gi.tile_scales(SFA, M, K).cuda(), gi.tile_scales(SFB, N, K).cuda()
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_mxfp8_tiled(TILED_VARIANTS[v], Ad.data_ptr(), Bd.data_ptr(), SAt.data_ptr(),
                            SBt.data_ptr(), Dbuf.data_ptr(), M, N, K, lda, lda, ldd, s)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    assert g.gemm_last_status(s) == g.GEMM_OK
    D_ref, _ = oracle.gemm_mxfp8(A.numpy(), B.numpy(), SFA.numpy(), SFB.numpy(), K)
    _check(Dbuf, M, N, D_ref)
