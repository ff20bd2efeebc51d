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
def test_workload_mxfp8_8192_tiled():
    """The bench's MXFP8 headline configuration: gemm_mxfp8_tiled, automatic
    kernel (the CTA pair, 256x256 tiles), every tile edge sampled."""
    w = gi.WORKLOADS["mxfp8_8192"]
    assert w.sf_layout == "tiled"
    A, SFA, B, SFB = gi.workload_operands("mxfp8_8192")
    D = g.matmul_mxfp8_tiled(A.cuda(), gi.tile_scales(SFA, w.M, w.K).cuda(), B.cuda(),
                             gi.tile_scales(SFB, w.N, w.K).cuda())
    assert g.gemm_last_status(0) == g.GEMM_OK
    rows, cols = P.sample_positions(w.M, w.N, 3000, seed=w.seed, tile_m=128, tile_n=256)
    D_ref, S = oracle.gemm_mxfp8_entries(A.numpy(), B.numpy(), SFA.numpy(), SFB.numpy(), rows, cols)
    P.check_within_bound(P.bf16_to_f64(D.cpu())[rows, cols], D_ref, S, "mxfp8_8192 tiled")


@pytest.mark.slow
def test_workload_mxfp8_8192():
    w = gi.WORKLOADS["mxfp8_8192_rows"]
    A, SFA, B, SFB = gi.workload_operands("mxfp8_8192")
    D = run(A, SFA, B, SFB, g.VARIANT_AUTO)
    # every 224-column tile edge of the MXFP8 kernels and every 128-row edge
    rows, cols = P.sample_positions(w.M, w.N, 3000, seed=w.seed, tile_m=128, tile_n=224)
    assert {223, 224, 8063, 8064} <= set(cols.tolist())
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


# ----------------------------------------------------- non-finite and extreme scales

def assert_matches_oracle(D, D_ref, what):
    """NaN exactly where the oracle has NaN, +-Inf where it has +-Inf, and the
    bf16 RNE of the oracle's value everywhere else, bit for bit (a zero of
    either sign where the oracle's value rounds to zero)."""
    d = P.bf16_to_f64(D)
    nan_ref = np.isnan(D_ref)
    assert np.array_equal(np.isnan(d), nan_ref), f"{what}: NaN pattern differs"
    inf_ref = np.isinf(D_ref)
    assert np.array_equal(d[inf_ref], D_ref[inf_ref]), f"{what}: Inf differs"
    fin = np.isfinite(D_ref)
    want = oracle.bf16_to_f64(oracle.f64_to_bf16_rne(D_ref[fin]))
    if not np.array_equal(d[fin], want):        # -0 == +0 here
        bad = np.flatnonzero(d[fin] != want)
        raise AssertionError(f"{what}: {bad.size} finite mismatches; first got {d[fin][bad[0]]} "
                             f"want {want[bad[0]]}")


MX_VARIANTS = ["1cta", "2cta", "auto"]


@pytest.mark.parametrize("v", MX_VARIANTS)
def test_nan_code_inside_k(v):
    """E4M3 NaN codes (0x7F, 0xFF) inside K: row r of D (from A) and column j
    (from B) are NaN, every other element is exact."""
    M, N, K = 260, 470, 256
    A, SFA, B, SFB = int_operands(M, N, K, seed=31)
    A[5, 100] = 0x7F
    A[200, 0] = 0xFF
    B[300, 255] = 0x7F
    D = run(A, SFA, B, SFB, VARIANTS[v])
    D_ref, _ = ref(A, SFA, B, SFB)
    assert np.isnan(D_ref[5]).all() and np.isnan(D_ref[:, 300]).all()
    assert_matches_oracle(D, D_ref, f"nan code/{v}")


@pytest.mark.parametrize("v", MX_VARIANTS)
def test_nan_scale_on_live_block(v):
    """A UE8M0 NaN scale (0xFF) on a block whose elements are live (inside K,
    nonzero): every product of that block is NaN, so row r of D (scale of A)
    and column j (scale of B) are NaN, the rest exact."""
    M, N, K = 300, 450, 192
    A, SFA, B, SFB = int_operands(M, N, K, seed=32)
    A[7, 64:96] = P.e4m3_from_ints(np.full(32, 3))         # live, nonzero block 2 of row 7
    B[250, 160:192] = P.e4m3_from_ints(np.full(32, -2))    # live block 5 (the last) of row 250
    SFA[7, 2] = 0xFF
    SFB[250, 5] = 0xFF
    D = run(A, SFA, B, SFB, VARIANTS[v])
    D_ref, _ = ref(A, SFA, B, SFB)
    assert np.isnan(D_ref[7]).all() and np.isnan(D_ref[:, 250]).all()
    assert_matches_oracle(D, D_ref, f"nan scale/{v}")


def e4m3_subnormal_codes(rng, shape):
    """Random E4M3 subnormal codes: sign, exponent field 0, mantissa 1..7
    (values +-m 2^-9)."""
    m = rng.integers(1, 8, size=shape)
    sign = rng.integers(0, 2, size=shape) << 7
    return torch.from_numpy((sign | m).astype(np.uint8))


@pytest.mark.parametrize("v", MX_VARIANTS)
def test_zero_scale_byte_is_two_to_minus_127(v):
    """Scale byte 0 means 2^-127, not zero: A holds subnormal E4M3 codes
    (+-m 2^-9) scaled by 2^-127 and B small integers scaled by 2^127 (byte
    254), so every product is +-m v 2^-9 exactly and the sums are exact in
    fp32; then the same with normal codes in A."""
    M, N, K = 200, 300, 256
    rng = np.random.default_rng(33)
    _, _, B, SFB = int_operands(M, N, K, seed=34)
    nblk = K // 32
    SFB[:, :nblk] = 254
    SFA = torch.zeros(M, gi.sf_pitch(K), dtype=torch.uint8)      # byte 0 everywhere
    A = e4m3_subnormal_codes(rng, (M, K))
    D = run(A, SFA, B, SFB, VARIANTS[v])
    D_ref, _ = ref(A, SFA, B, SFB)
    assert np.all(np.abs(D_ref[np.nonzero(D_ref)]) >= 2.0 ** -9)   # far from underflow
    assert_matches_oracle(D, D_ref, f"scale 0 subnormal/{v}")
    A2, _, _, _ = int_operands(M, N, K, seed=35)
    D = run(A2, SFA, B, SFB, VARIANTS[v])
    D_ref, _ = ref(A2, SFA, B, SFB)
    assert_matches_oracle(D, D_ref, f"scale 0 normal/{v}")


@pytest.mark.parametrize("v", MX_VARIANTS)
def test_zero_scales_underflow_to_zero(v):
    """Both scales 2^-127 (byte 0): every product is below 2^-248, far under
    the smallest bf16 (and fp32) subnormal, so the oracle's value rounds to
    zero and D must be zero everywhere."""
    M, N, K = 130, 260, 128
    A, _, B, _ = int_operands(M, N, K, seed=36)
    A[:, :K] = P.e4m3_from_ints(np.random.default_rng(37).integers(1, 5, size=(M, K)))
    SFA = torch.zeros(M, gi.sf_pitch(K), dtype=torch.uint8)
    SFB = torch.zeros(N, gi.sf_pitch(K), dtype=torch.uint8)
    D = run(A, SFA, B, SFB, VARIANTS[v])
    D_ref, _ = ref(A, SFA, B, SFB)
    assert np.all(np.abs(D_ref) < 2.0 ** -240) and np.any(D_ref != 0)
    assert_matches_oracle(D, D_ref, f"underflow/{v}")


# ------------------------------------------- scale matrices in any layout (gathered)

def run_sf_layout(A, SFA_rows, B, SFB_rows, variant, K, ldsf, offset):
    """The scale rows stored at pitch `ldsf` bytes, `offset` bytes into a
    device buffer (so the base may be misaligned)."""
    M, N = A.shape[0], B.shape[0]
    nblk = (K + 31) // 32

    def place(sf_rows):
        R = sf_rows.shape[0]
        buf = torch.full((offset + R * ldsf + 64,), 0xFF, dtype=torch.uint8)   # NaN scales around
        view = buf[offset:offset + R * ldsf].view(R, ldsf)
        view[:, :nblk] = sf_rows[:, :nblk]
        return buf.cuda(), view

    sa_dev, sa = place(SFA_rows)
    sb_dev, sb = place(SFB_rows)
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_mxfp8_variant(variant, Ad.data_ptr(), Bd.data_ptr(), sa_dev.data_ptr() + offset,
                              sb_dev.data_ptr() + offset, D.data_ptr(), M, N, K, A.shape[1],
                              B.shape[1], ldsf, ldsf, N, s)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    st = g.gemm_last_status(s)
    assert st == g.GEMM_OK, g.gemm_status_string(st)
    return D.cpu(), sa, sb


@pytest.mark.parametrize("v", MX_VARIANTS)
@pytest.mark.parametrize("ldsf, offset", [(33, 0), (33, 1), (40, 4), (48, 3)])
def test_dense_scale_layout_k1040(v, ldsf, offset):
    """K = 1040 (33 scale blocks, a partial K-tile) with the scale matrices
    in the dense layout ld = ceil(K/32) = 33, and at other pitches and base
    offsets that TMA cannot read; bytes around the rows hold NaN scales that
    must not be read.  Exact integer operands: bitwise against the oracle."""
    M, N, K = 300, 470, 1040
    A, SFA, B, SFB = int_operands(M, N, K, seed=38, lda=1040)
    D, sa, sb = run_sf_layout(A, SFA, B, SFB, VARIANTS[v], K, ldsf, offset)
    D_ref, _ = ref(A, sa, B, sb, K)
    assert_matches_oracle(D, D_ref, f"dense scales ld={ldsf} off={offset}/{v}")


def test_dense_scale_layout_quantised_normal():
    """Quantised N(0,1) operands, dense scale layout, several waves of tiles."""
    M, N, K = 1100, 1500, 1040
    A, SFA, B, SFB = gi.mxfp8_operands(M, N, K, seed=39)
    D, sa, sb = run_sf_layout(A, SFA, B, SFB, g.VARIANT_AUTO, K, 33, 0)
    D_ref, S = ref(A, sa, B, sb, K)
    P.check_within_bound(P.bf16_to_f64(D), D_ref, S, "dense scales, quantised")


@pytest.mark.parametrize("v", ["1cta", "2cta"])
@pytest.mark.parametrize("M, N, ldd", [(300, 520, 536), (129, 456, 456), (257, 1000, 1008)])
def test_tma_store_epilogue_guard_band(v, M, N, ldd):
    """The 32-column TMA-store epilogue of the MXFP8 kernels (aligned D, N * 2
    a multiple of 16): ragged M and N against the 224-column tiles, exact,
    and the pitch padding never written."""
    K = 256
    A, SFA, B, SFB = int_operands(M, N, K, seed=M + N)
    plan = g.gemm_kernel_plan(True, VARIANTS[v])
    assert plan["tile_n"] == 224
    Ad, Bd, SAd, SBd = (t.cuda() for t in (A, B, SFA, SFB))
    D = torch.full((M, ldd), float("nan"), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_mxfp8_variant(VARIANTS[v], Ad.data_ptr(), Bd.data_ptr(), SAd.data_ptr(),
                              SBd.data_ptr(), D.data_ptr(), M, N, K, K, K, SFA.shape[1],
                              SFB.shape[1], ldd, s)
    assert rc == g.GEMM_OK and g.gemm_last_status(s) == g.GEMM_OK
    D = D.cpu()
    assert torch.isnan(D[:, N:].float()).all(), "padding columns written"
    D_ref, _ = ref(A, SFA, B, SFB)
    assert np.array_equal(gi.bf16_codes(D[:, :N]), oracle.f64_to_bf16_rne(D_ref))


# ------------------------------------ tiled scale layout (gemm_mxfp8_tiled)

TILED_VARIANTS = {
    "auto": g.VARIANT_AUTO,
    "2cta": g.VARIANT_2CTA,
    "2cta_direct": g.VARIANT_2CTA | g.VARIANT_DIRECT_STORE,
    "1cta": g.VARIANT_1CTA,
}


def run_tiled(A, SFA, B, SFB, variant, K=None, ldd=None):
    """The same operands as run(), the row-major scales rearranged into the
    tiled layout on the host (a permutation with zero padding)."""
    M, lda = A.shape
    N, ldb = B.shape
    K = lda if K is None else K
    ldd = N if ldd is None else ldd
    Ad, Bd = A.cuda(), B.cuda()
    SAt, SBt = gi.tile_scales(SFA, M, K).cuda(), gi.tile_scales(SFB, N, K).cuda()
    D = torch.full((M, ldd), float("nan"), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_mxfp8_tiled(variant, Ad.data_ptr(), Bd.data_ptr(), SAt.data_ptr(), SBt.data_ptr(),
                            D.data_ptr(), M, N, K, lda, ldb, ldd, s)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    st = g.gemm_last_status(s)
    assert st == g.GEMM_OK, g.gemm_status_string(st)
    D = D.cpu()
    if ldd > N:
        assert torch.isnan(D[:, N:].float()).all(), "padding columns written"
    return D[:, :N]


def test_tiled_plan():
    for v, cg, tm in (("auto", 2, 256), ("2cta", 2, 256), ("1cta", 1, 128)):
        p = g.gemm_kernel_plan(2, TILED_VARIANTS[v])
        assert (p["cluster"], p["tile_m"], p["tile_n"], p["tmem_cols"]) == (cg, tm, 256, 512)


@pytest.mark.parametrize("v", list(TILED_VARIANTS))
@pytest.mark.parametrize("shape", [(128, 256, 128), (256, 256, 128), (300, 520, 256),
                                   (129, 300, 160), (1000, 900, 1184), (513, 1031, 1056)])
def test_tiled_exact_integers(v, shape):
    """Bitwise against the oracle with scales varying per (row, 32-k block):
    a scale chunk loaded for the wrong row block, K-tile or CTA shows up as a
    wrong bit."""
    M, N, K = shape
    lda = (K + 15) // 16 * 16
    A, SFA, B, SFB = int_operands(M, N, K, seed=M + 5 * N + K, lda=lda)
    D = run_tiled(A, SFA, B, SFB, TILED_VARIANTS[v], K=K)
    D_ref, _ = ref(A, SFA, B, SFB, K)
    assert_matches_oracle(D, D_ref, f"tiled {shape}/{v}")


@pytest.mark.parametrize("v", ["auto", "1cta"])
@pytest.mark.parametrize("shape", [(300, 520, 384), (700, 1100, 2048)])
def test_tiled_quantised_normal(v, shape):
    M, N, K = shape
    A, SFA, B, SFB = gi.mxfp8_operands(M, N, K, seed=M + N + 1)
    D = run_tiled(A, SFA, B, SFB, TILED_VARIANTS[v], ldd=N + 8)
    D_ref, S = ref(A, SFA, B, SFB)
    P.check_within_bound(P.bf16_to_f64(D), D_ref, S, f"tiled mx {shape}/{v}")


@pytest.mark.parametrize("v", ["auto", "1cta"])
def test_tiled_nan_scale_and_code(v):
    M, N, K = 300, 450, 192
    A, SFA, B, SFB = int_operands(M, N, K, seed=41)
    A[7, 64:96] = P.e4m3_from_ints(np.full(32, 3))
    SFA[7, 2] = 0xFF
    B[250, 100] = 0x7F
    D = run_tiled(A, SFA, B, SFB, TILED_VARIANTS[v])
    D_ref, _ = ref(A, SFA, B, SFB)
    assert np.isnan(D_ref[7]).all() and np.isnan(D_ref[:, 250]).all()
    assert_matches_oracle(D, D_ref, f"tiled nan/{v}")


def test_tiled_validation():
    A = torch.zeros(256, 256, dtype=torch.uint8, device="cuda")
    D = torch.empty(256, 256, dtype=torch.bfloat16, device="cuda")
    sf = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    f = lambda sfa, v=g.VARIANT_AUTO: g.gemm_mxfp8_tiled(v, A.data_ptr(), A.data_ptr(), sfa,
                                                         sf.data_ptr(), D.data_ptr(), 256, 256,
                                                         256, 256, 256, 256, 0)
    assert f(sf.data_ptr() + 8) == g.GEMM_ERR_ALIGNMENT
    assert f(0) == g.GEMM_ERR_INVALID_ARG
    assert f(sf.data_ptr(), g.VARIANT_SYNC) == g.GEMM_ERR_INVALID_ARG
    assert f(sf.data_ptr()) == g.GEMM_OK
    assert g.gemm_last_status(0) == g.GEMM_OK
