"""Seeded random shapes through every schedule path: whole tiles, the tail
split, the edge-last deal, the one-CTA MMA cut at the right edge, small K,
odd pitches, one CTA and the pair, TMA and masked stores, the tiled-scale
MXFP8 kernels, and the general build's stream-K split and fused epilogue.
Operands are small integers (and, for MXFP8, power-of-two scales), so every
fp32 partial sum is exact and D must equal the oracle's result bit for bit
everywhere; the pitch padding (pre-filled with NaN) must be left untouched."""
import numpy as np
import pytest
import torch

import dense_gemm_blackwell_tcgen05_gb300 as g
import gemm_inputs as gi
import oracle
from tests import parity as P
from tests.test_gemm_mxfp8 import int_operands

pytestmark = pytest.mark.gpu

BF16_VARIANTS = [g.VARIANT_AUTO, g.VARIANT_1CTA, g.VARIANT_2CTA,
                 g.VARIANT_1CTA | g.VARIANT_DIRECT_STORE, g.VARIANT_2CTA | g.VARIANT_DIRECT_STORE]


def _dim(rng, hi):
    """Sizes that hit tile edges often: a multiple of 128 or 256 plus a
    small remainder, or any size up to hi."""
    r = rng.random()
    if r < 0.35:
        return int(rng.integers(1, hi // 128 + 1)) * 128 + int(rng.integers(0, 9))
    if r < 0.55:
        return int(rng.integers(1, hi // 256 + 1)) * 256 - int(rng.integers(0, 5))
    return int(rng.integers(1, hi + 1))


def _bf16_cases(n=40, seed=2026):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        M, N = _dim(rng, 2600), _dim(rng, 2600)
        K = int(rng.integers(1, 17)) if i % 8 == 0 else int(rng.integers(1, 320))
        v = BF16_VARIANTS[i % len(BF16_VARIANTS)]
        pad = int(rng.integers(0, 10)) if i % 3 else 0
        cases.append((M, N, K, v, N + pad))
    return cases


def _mx_cases(n=12, seed=2027):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        M, N = _dim(rng, 2000), _dim(rng, 2000)
        K = int(rng.integers(1, 20)) * 16
        v = (g.VARIANT_AUTO, g.VARIANT_1CTA, g.VARIANT_2CTA | g.VARIANT_DIRECT_STORE)[i % 3]
        cases.append((M, N, K, v))
    return cases


def _ids(c):
    return "x".join(str(x) for x in c[:3]) + f"-v{c[3]:#x}" + (f"-ld{c[4]}" if len(c) > 4 else "")


@pytest.mark.parametrize("case", _bf16_cases(), ids=_ids)
def test_bf16_random_shape_is_exact(case):
    M, N, K, v, ldd = case
    lda = (K + 7) // 8 * 8
    rng = np.random.default_rng(M * 31 + N * 7 + K)
    A = torch.zeros(M, lda, dtype=torch.bfloat16)
    B = torch.zeros(N, lda, dtype=torch.bfloat16)
    A[:, :K] = P.bf16_from_ints(rng.integers(-3, 4, size=(M, K)))
    B[:, :K] = P.bf16_from_ints(rng.integers(-3, 4, size=(N, K)))
    D = torch.full((M, ldd), float("nan"), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    Ad, Bd = A.cuda(), B.cuda()   # held until the call has run
    rc = g.gemm_bf16_variant(v, Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K,
                             lda, lda, ldd, s)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    assert g.gemm_last_status(s) == g.GEMM_OK
    sched = g.gemm_last_schedule()
    Dh = D.cpu()
    D_ref, _ = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B), K)
    got = gi.bf16_codes(Dh[:, :N].contiguous())
    bad = np.argwhere(got != oracle.f64_to_bf16_rne(D_ref))
    assert len(bad) == 0, f"{case}: {len(bad)} mismatches, first {tuple(bad[0])}; schedule {sched}"
    if ldd > N:
        assert torch.isnan(Dh[:, N:].float()).all(), f"{case}: pitch padding written"


@pytest.mark.parametrize("case", _mx_cases(), ids=_ids)
def test_mxfp8_tiled_random_shape_is_exact(case):
    M, N, K, v = case
    A, SFA, B, SFB = int_operands(M, N, K, seed=M + 5 * N + K)
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    SAt, SBt = gi.tile_scales(SFA, M, K).cuda(), gi.tile_scales(SFB, N, K).cuda()
    Ad, Bd = A.cuda(), B.cuda()   # held until the call has run
    rc = g.gemm_mxfp8_tiled(v, Ad.data_ptr(), Bd.data_ptr(), SAt.data_ptr(),
                            SBt.data_ptr(), D.data_ptr(), M, N, K, K, K, N, s)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    assert g.gemm_last_status(s) == g.GEMM_OK
    D_ref, _ = oracle.gemm_mxfp8(A.numpy(), B.numpy(), SFA.numpy(), SFB.numpy(), K)
    got = gi.bf16_codes(D.cpu())
    bad = np.argwhere(got != oracle.f64_to_bf16_rne(D_ref))
    assert len(bad) == 0, f"{case}: {len(bad)} mismatches, first {tuple(bad[0])}"


def _general_cases():
    """Random shapes (K > 16, so that the persistent kernel runs) on the one-CTA
    and pair variants with either store path."""
    out = []
    for seed in (300, 301):
        for (M, N, K, v, ldd) in _bf16_cases(n=24, seed=seed):
            if K > 16:
                out.append((M, N, K, v, ldd))
    return out


def _int_pair(M, N, K, seed):
    rng = np.random.default_rng(seed)
    lda = (K + 7) // 8 * 8
    A = torch.zeros(M, lda, dtype=torch.bfloat16)
    B = torch.zeros(N, lda, dtype=torch.bfloat16)
    A[:, :K] = P.bf16_from_ints(rng.integers(-3, 4, size=(M, K)))
    B[:, :K] = P.bf16_from_ints(rng.integers(-3, 4, size=(N, K)))
    return A, B, lda


@pytest.mark.parametrize("case", _general_cases(), ids=_ids)
def test_forced_streamk_random_shape_is_exact(case):
    """Every tile split along K (stream-K forced on), the partial sums added by
    the owner in K order: exact integer sums, so bitwise equal to the oracle."""
    M, N, K, v, ldd = case
    A, B, lda = _int_pair(M, N, K, M + N + K)
    Ad, Bd = A.cuda(), B.cuda()
    s = torch.cuda.current_stream().cuda_stream
    prev = g.gemm_set_streamk_mode(g.STREAMK_ALWAYS)
    try:
        ws = g.streamk_workspace(False, v)
        D = torch.full((M, ldd), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = g.gemm_bf16_streamk(v, Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K, lda, lda,
                                 ldd, ws.data_ptr(), ws.numel(), s)
        assert rc == g.GEMM_OK, g.gemm_status_string(rc)
        sched = g.gemm_last_schedule()
        assert g.gemm_last_status(s) == g.GEMM_OK
    finally:
        g.gemm_set_streamk_mode(prev)
    D_ref, _ = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B), K)
    Dh = D.cpu()
    got = gi.bf16_codes(Dh[:, :N].contiguous())
    bad = np.argwhere(got != oracle.f64_to_bf16_rne(D_ref))
    assert len(bad) == 0, f"{case}: {len(bad)} mismatches, first {tuple(bad[0])}; schedule {sched}"
    if ldd > N:
        assert torch.isnan(Dh[:, N:].float()).all(), f"{case}: pitch padding written"


@pytest.mark.parametrize("case", _general_cases(), ids=_ids)
def test_fused_random_shape_is_exact(case):
    """relu(2 acc - C + bias) with integer C and bias: every step is exact in
    fp32, so D equals the oracle's epilogue of its own sums bit for bit.  C has
    D's pitch, so an aligned pitch brings it in by TMA on the pair."""
    M, N, K, v, ldd = case
    A, B, lda = _int_pair(M, N, K, M + 3 * N + K)
    Ad, Bd = A.cuda(), B.cuda()
    gen = torch.Generator().manual_seed(K)
    bias = torch.randint(-8, 9, (N,), generator=gen).to(torch.float32)
    C = torch.randint(-8, 9, (M, ldd), generator=gen).to(torch.bfloat16)
    Cd, bd = C.cuda(), bias.cuda()
    epi = g.make_epilogue(2.0, -1.0, Cd, bd, "relu", torch.bfloat16)
    D = torch.full((M, ldd), float("nan"), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_bf16_fused(v, Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K, lda, lda, ldd,
                           epi, s)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    assert g.gemm_last_status(s) == g.GEMM_OK
    D_sum, _ = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B), K)
    want = oracle.epilogue(D_sum, 2.0, -1.0, C[:, :N].double().numpy(), bias.double().numpy(), 1)
    Dh = D.cpu()
    got = gi.bf16_codes(Dh[:, :N].contiguous())
    bad = np.argwhere(got != oracle.f64_to_bf16_rne(want))
    assert len(bad) == 0, f"{case}: {len(bad)} mismatches, first {tuple(bad[0])}"
    if ldd > N:
        assert torch.isnan(Dh[:, N:].float()).all(), f"{case}: pitch padding written"
