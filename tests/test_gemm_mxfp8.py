"""Block-scaled MXFP8 GEMM on the GPU through the C ABI against the oracle.
Bitwise for integer E4M3 operands with power-of-two scales varying per
(row, 32-k block) -- every partial sum is then exact in fp32, so a scale
applied to the wrong row or block shows up as a wrong bit -- and within the
bf16-output bound for operands quantised from N(0,1)."""
import numpy as np
import pytest
import torch

import dense_gemm_blackwell_tcgen05_gb300 as g
import gemm_inputs as gi
import oracle
from tests import parity as P

pytestmark = pytest.mark.gpu

VARIANTS = {
    "1cta": g.VARIANT_1CTA,
    "1cta_direct": g.VARIANT_1CTA | g.VARIANT_DIRECT_STORE,
    "2cta": g.VARIANT_2CTA,
    "auto": g.VARIANT_AUTO,
}


def run(A, SFA, B, SFB, variant, K=None, ldd=None):
    """A [M, lda], B [N, ldb] uint8 E4M3 codes; SFA/SFB [rows, pitch] uint8."""
    Ad, Bd, SAd, SBd = (t.cuda() for t in (A, B, SFA, SFB))
    M, lda = A.shape
    N, ldb = B.shape
    K = lda if K is None else K
    ldd = N if ldd is None else ldd
    D = torch.full((M, ldd), float("nan"), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_mxfp8_variant(variant, Ad.data_ptr(), Bd.data_ptr(), SAd.data_ptr(), SBd.data_ptr(),
                              D.data_ptr(), M, N, K, lda, ldb, SFA.shape[1], SFB.shape[1], ldd, s)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    st = g.gemm_last_status(s)
    assert st == g.GEMM_OK, g.gemm_status_string(st)
    return D[:, :N].cpu()


def ref(A, SFA, B, SFB, K=None):
    return oracle.gemm_mxfp8(A.numpy(), B.numpy(), SFA.numpy(), SFB.numpy(), K)


def int_operands(M, N, K, seed, lda=None, imax=None, sf_lo=None, sf_hi=None):
    """Integer E4M3 values in [-imax, imax] and scale bytes in [sf_lo, sf_hi],
    chosen so that every partial sum is exact in fp32: the sum is a multiple
    of 2^(2 sf_lo - 254) and at most imax^2 K 2^(2 sf_hi - 254) in size, so it
    needs fewer than 24 significant bits whatever the summation order."""
    rng = np.random.default_rng(seed)
    lda = K if lda is None else lda
    if imax is None:
        imax, sf_lo, sf_hi = (4, 124, 130) if K <= 256 else (1, 126, 129)
    span = np.log2(imax * imax * K) + 2 * (sf_hi - sf_lo)
    assert span <= 24, "operand ranges would not keep fp32 partial sums exact"
    nblk = (K + 31) // 32
    pitch = gi.sf_pitch(K)
    A = torch.zeros(M, lda, dtype=torch.uint8)
    A[:, :K] = P.e4m3_from_ints(rng.integers(-imax, imax + 1, size=(M, K)))
    B = torch.zeros(N, lda, dtype=torch.uint8)
    B[:, :K] = P.e4m3_from_ints(rng.integers(-imax, imax + 1, size=(N, K)))
    SFA = torch.zeros(M, pitch, dtype=torch.uint8)
    SFB = torch.zeros(N, pitch, dtype=torch.uint8)
    SFA[:, :nblk] = torch.from_numpy(rng.integers(sf_lo, sf_hi + 1, size=(M, nblk)).astype(np.uint8))
    SFB[:, :nblk] = torch.from_numpy(rng.integers(sf_lo, sf_hi + 1, size=(N, nblk)).astype(np.uint8))
    return A, SFA, B, SFB


@pytest.mark.parametrize("v", list(VARIANTS))
@pytest.mark.parametrize("shape", [(128, 256, 128), (300, 520, 256), (129, 300, 160),
                                   (257, 513, 100), (130, 260, 1056)])
def test_exact_integers(v, shape):
    M, N, K = shape
    lda = (K + 15) // 16 * 16
    A, SFA, B, SFB = int_operands(M, N, K, seed=M + 3 * N + K, lda=lda)
    D = run(A, SFA, B, SFB, VARIANTS[v], K=K)
    D_ref, _ = ref(A, SFA, B, SFB, K)
    want = oracle.f64_to_bf16_rne(D_ref)
    got = gi.bf16_codes(D)
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        i, j = bad[0]
        raise AssertionError(f"{len(bad)} mismatches; first at {(i, j)}: got {D[i, j].item()} "
                             f"want {D_ref[i, j]}")


@pytest.mark.parametrize("v", list(VARIANTS))
def test_identity(v):
    K, N = 256, 300
    A = torch.zeros(K, K, dtype=torch.uint8)
    A[torch.arange(K), torch.arange(K)] = 0x38                # E4M3 1.0
    SFA = torch.full((K, gi.sf_pitch(K)), 127, dtype=torch.uint8)
    _, _, B, SFB = int_operands(1, N, K, seed=2)
    D = run(A, SFA, B, SFB, VARIANTS[v])
    D_ref, _ = ref(A, SFA, B, SFB)
    assert np.array_equal(gi.bf16_codes(D), oracle.f64_to_bf16_rne(D_ref))


@pytest.mark.parametrize("v", list(VARIANTS))
@pytest.mark.parametrize("shape", [(300, 520, 384), (128, 256, 4096), (513, 1031, 224)])
def test_quantised_normal_full(v, shape):
    M, N, K = shape
    A, SFA, B, SFB = gi.mxfp8_operands(M, N, K, seed=M + N)
    D = run(A, SFA, B, SFB, VARIANTS[v])
    D_ref, S = ref(A, SFA, B, SFB)
    P.check_within_bound(P.bf16_to_f64(D), D_ref, S, f"mx {shape}/{v}")


def test_wide_scale_pitch():
    M, N, K = 200, 300, 256
    A, SFA, B, SFB = int_operands(M, N, K, seed=4)
    SFA_w = torch.zeros(M, 48, dtype=torch.uint8)
    SFA_w[:, :SFA.shape[1]] = SFA
    D = run(A, SFA_w, B, SFB, g.VARIANT_AUTO)
    D_ref, _ = ref(A, SFA, B, SFB)
    assert np.array_equal(gi.bf16_codes(D), oracle.f64_to_bf16_rne(D_ref))


@pytest.mark.slow
def test_workload_mxfp8_8192():
    w = gi.WORKLOADS["mxfp8_8192"]
    A, SFA, B, SFB = gi.workload_operands("mxfp8_8192")
    D = run(A, SFA, B, SFB, g.VARIANT_AUTO)
    rows, cols = P.sample_positions(w.M, w.N, 3000, seed=w.seed)
    D_ref, S = oracle.gemm_mxfp8_entries(A.numpy(), B.numpy(), SFA.numpy(), SFB.numpy(), rows, cols)
    P.check_within_bound(P.bf16_to_f64(D)[rows, cols], D_ref, S, "mxfp8_8192")


@pytest.mark.parametrize("v", list(VARIANTS))
@pytest.mark.parametrize("K, lda", [(100, 112), (40, 48), (1000, 1008)])
def test_k_tail_reads_nothing_past_k(v, K, lda):
    """Operand padding holds 448 and scale padding holds the NaN scale 0xFF;
    neither may reach the result."""
    M, N = 256, 512
    A = torch.full((M, lda), 0x38, dtype=torch.uint8)          # E4M3 1.0
    B = torch.full((N, lda), 0x38, dtype=torch.uint8)
    A[:, K:] = 0x7E
    B[:, K:] = 0x7E
    nblk = (K + 31) // 32
    SFA = torch.full((M, 48), 0xFF, dtype=torch.uint8)
    SFB = torch.full((N, 48), 0xFF, dtype=torch.uint8)
    SFA[:, :nblk] = 127
    SFB[:, :nblk] = 127
    D = run(A, SFA, B, SFB, VARIANTS[v], K=K)
    D_ref, _ = ref(A, SFA, B, SFB, K)
    assert np.array_equal(gi.bf16_codes(D), oracle.f64_to_bf16_rne(D_ref))
