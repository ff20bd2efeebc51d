"""bf16 GEMM on the GPU through the C ABI, element by element against the
oracle.  Bitwise where every partial sum is exact in fp32 (all-ones,
identity, K=1, small integers); within the bound
|D - D_ref| <= 2^-7 |D_ref| + 1e-3 sum_k |a_ik b_jk| otherwise."""
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
    "2cta": g.VARIANT_2CTA,
    "sync": g.VARIANT_SYNC,
    "1cta_direct": g.VARIANT_1CTA | g.VARIANT_DIRECT_STORE,
    "2cta_direct": g.VARIANT_2CTA | g.VARIANT_DIRECT_STORE,
    "auto": g.VARIANT_AUTO,
}
FAST = ["1cta", "2cta", "auto"]


def run(A_cpu, B_cpu, variant, K=None, ldd=None, stream=None):
    """D = A B^T on the GPU (A [M, lda], B [N, ldb] bf16 CPU tensors)."""
    A = A_cpu.cuda()
    B = B_cpu.cuda()
    M, lda = A.shape
    N, ldb = B.shape
    K = lda if K is None else K
    ldd = N if ldd is None else ldd
    Dfull = torch.full((M, ldd), float("nan"), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream() if stream is None else stream
    rc = g.gemm_bf16_variant(variant, A.data_ptr(), B.data_ptr(), Dfull.data_ptr(), M, N, K, lda,
                             ldb, ldd, s.cuda_stream)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    st = g.gemm_last_status(s.cuda_stream)
    assert st == g.GEMM_OK, g.gemm_status_string(st)
    return Dfull[:, :N].cpu()


def ref(A_cpu, B_cpu, K=None):
    return oracle.gemm_bf16(gi.bf16_codes(A_cpu), gi.bf16_codes(B_cpu), K)


def assert_bitwise(D_gpu, D_ref):
    want = oracle.f64_to_bf16_rne(D_ref)
    got = gi.bf16_codes(D_gpu)
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        i, j = bad[0]
        raise AssertionError(f"{len(bad)} mismatches; first at {(i, j)}: got {D_gpu[i, j].item()} "
                             f"want {D_ref[i, j]}")


# ------------------------------------------------------------ exact pins

@pytest.mark.parametrize("v", list(VARIANTS))
def test_single_tile_workload(v):
    w = gi.WORKLOADS["single_tile"]
    A, B = gi.workload_operands("single_tile")
    D = run(A, B, VARIANTS[v])
    D_ref, S = ref(A, B)
    P.check_within_bound(P.bf16_to_f64(D), D_ref, S, f"single_tile/{v}")
    assert D.shape == (w.M, w.N)


@pytest.mark.parametrize("v", list(VARIANTS))
@pytest.mark.parametrize("K", [8, 64, 1040])
def test_all_ones(v, K):
    M, N = 300, 520
    A = torch.ones(M, K, dtype=torch.bfloat16)
    B = torch.ones(N, K, dtype=torch.bfloat16)
    D = run(A, B, VARIANTS[v])
    assert torch.all(D.float() == K), (D.float().min().item(), D.float().max().item())


@pytest.mark.parametrize("v", list(VARIANTS))
def test_identity(v):
    K, N = 256, 300
    A = torch.eye(K, dtype=torch.bfloat16)
    B = torch.randn(N, K, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    D = run(A, B, VARIANTS[v])
    assert torch.equal(D, B.t().contiguous())


@pytest.mark.parametrize("v", list(VARIANTS))
def test_k1_outer_product(v):
    g_ = torch.Generator().manual_seed(6)
    M, N = 200, 300
    A = torch.zeros(M, 8, dtype=torch.bfloat16)
    B = torch.zeros(N, 8, dtype=torch.bfloat16)
    A[:, 0] = (torch.randn(M, generator=g_) * 3).to(torch.bfloat16)
    B[:, 0] = (torch.randn(N, generator=g_) * 0.5).to(torch.bfloat16)
    D = run(A, B, VARIANTS[v], K=1)
    D_ref, _ = ref(A, B, 1)
    assert_bitwise(D, D_ref)


@pytest.mark.parametrize("v", list(VARIANTS))
@pytest.mark.parametrize("shape", [(300, 520, 64), (129, 257, 40), (257, 300, 1040), (4099, 513, 200)])
def test_small_integers(v, shape):
    M, N, K = shape
    rng = np.random.default_rng(M + N + K)
    A = P.bf16_from_ints(rng.integers(-2, 3, size=(M, K)))
    B = P.bf16_from_ints(rng.integers(-2, 3, size=(N, K)))
    D = run(A, B, VARIANTS[v])
    D_ref, _ = ref(A, B)
    assert_bitwise(D, D_ref)


# ------------------------------------------------------- seeded, tolerance

@pytest.mark.parametrize("v", list(VARIANTS))
@pytest.mark.parametrize("shape", [(300, 520, 200), (128, 256, 4096), (513, 1031, 264), (1, 1, 8)])
def test_random_full(v, shape):
    M, N, K = shape
    A, B = gi.bf16_operands(M, N, K, seed=M * 7 + N)
    D = run(A, B, VARIANTS[v])
    D_ref, S = ref(A, B)
    P.check_within_bound(P.bf16_to_f64(D), D_ref, S, f"{shape}/{v}")


@pytest.mark.parametrize("v", ["1cta", "2cta", "sync"])
def test_pitches_and_guard_bands(v):
    """lda > K, ldb > K, ldd > N (aligned and unaligned): rows read at the
    pitch, and nothing outside D[:, :N] is written."""
    M, N, K = 261, 300, 136
    A_wide, B_wide = gi.bf16_operands(M, N, K + 24, seed=9)    # lda = K + 24
    B_wide = B_wide[:, :K + 8].contiguous()                      # ldb = K + 8
    for ldd in (N + 12, N + 13):                                 # 16-byte rows / odd pitch
        sentinel = torch.tensor(-1234.0).to(torch.bfloat16)
        Dbuf = torch.full((M + 2, ldd), sentinel.item(), dtype=torch.bfloat16, device="cuda")
        D = Dbuf[1:M + 1]
        A = A_wide.cuda()
        B = B_wide.cuda()
        s = torch.cuda.current_stream().cuda_stream
        rc = g.gemm_bf16_variant(VARIANTS[v], A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K,
                                 A.stride(0), B.stride(0), ldd, s)
        assert rc == g.GEMM_OK
        assert g.gemm_last_status(s) == g.GEMM_OK
        host = Dbuf.cpu()
        assert torch.all(host[0] == sentinel) and torch.all(host[M + 1] == sentinel)
        assert torch.all(host[1:M + 1, N:] == sentinel), "write outside D[:, :N]"
        D_ref, S = oracle.gemm_bf16(gi.bf16_codes(A_wide), gi.bf16_codes(B_wide), K)
        P.check_within_bound(P.bf16_to_f64(host[1:M + 1, :N]), D_ref, S, f"ldd={ldd}/{v}")


@pytest.mark.parametrize("v", FAST)
def test_k_zero_writes_zeros(v):
    D = torch.full((37, 45), 7.0, dtype=torch.bfloat16, device="cuda")
    A = torch.zeros(37, 8, dtype=torch.bfloat16, device="cuda")
    rc = g.gemm_bf16_variant(VARIANTS[v], A.data_ptr(), A.data_ptr(), D.data_ptr(), 37, 45, 0, 8, 8,
                             45, 0)
    assert rc == g.GEMM_OK and g.gemm_last_status(0) == g.GEMM_OK
    assert torch.all(D == 0)


def test_empty_m_or_n_is_noop():
    D = torch.full((4, 4), 7.0, dtype=torch.bfloat16, device="cuda")
    assert g.gemm_bf16(0, 0, D.data_ptr(), 0, 4, 16, 16, 16, 4, 0) == g.GEMM_OK
    assert g.gemm_bf16(0, 0, D.data_ptr(), 4, 0, 16, 16, 16, 4, 0) == g.GEMM_OK
    torch.cuda.synchronize()
    assert torch.all(D == 7.0)


def test_host_pointer_rejected():
    A = torch.zeros(4, 16, dtype=torch.bfloat16)            # host memory
    D = torch.zeros(4, 4, dtype=torch.bfloat16, device="cuda")
    Ad = A.cuda()
    assert g.gemm_bf16(A.data_ptr(), Ad.data_ptr(), D.data_ptr(), 4, 4, 16, 16, 16, 4, 0) \
        == g.GEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("v", FAST)
def test_nonfinite_propagation(v):
    M, N, K = 130, 260, 72
    A = torch.ones(M, K, dtype=torch.bfloat16)
    B = torch.ones(N, K, dtype=torch.bfloat16)
    A[5, 3] = float("nan")
    A[129, 0] = float("inf")
    B[257, 0] = 0.0                                          # inf * 0 -> NaN at (129, 257)
    D = run(A, B, VARIANTS[v]).float()
    assert torch.all(torch.isnan(D[5]))
    assert torch.isnan(D[129, 257]) and torch.isinf(D[129, 0]) and D[129, 0] > 0
    mask = torch.ones_like(D, dtype=torch.bool)
    mask[5] = False
    mask[129] = False
    mask[:, 257] = False
    assert torch.all(D[mask] == K)
    rows = [i for i in range(M) if i not in (5, 129)]
    assert torch.all(D[rows, 257] == K - 1)            # the one zero term of column 257


def test_deterministic_and_streams():
    A, B = gi.bf16_operands(700, 900, 520, seed=11)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        D1 = run(A, B, g.VARIANT_AUTO, stream=side)
    D2 = run(A, B, g.VARIANT_AUTO)
    assert torch.equal(D1, D2)


# ----------------------------------------------- the named workloads, full size

def _sampled(name, variant, n_random=3000):
    w = gi.WORKLOADS[name]
    A, B = gi.workload_operands(name)
    D = run(A, B, variant)
    rows, cols = P.sample_positions(w.M, w.N, n_random, seed=w.seed)
    D_ref, S = oracle.gemm_bf16_entries(gi.bf16_codes(A), gi.bf16_codes(B), rows, cols)
    got = P.bf16_to_f64(D)[rows, cols]
    P.check_within_bound(got, D_ref, S, name)
    return A, B, D


def test_workload_ragged_k8_full():
    A, B = gi.workload_operands("ragged_k8")
    for v in (g.VARIANT_AUTO, g.VARIANT_1CTA, g.VARIANT_2CTA):
        D = run(A, B, v)
        D_ref, S = ref(A, B)
        P.check_within_bound(P.bf16_to_f64(D), D_ref, S, f"ragged_k8/{v}")


def test_workload_ragged_k1040():
    A, B, D = _sampled("ragged_k1040", g.VARIANT_AUTO)
    # the last M-block (ragged rows) in full
    r0 = (A.shape[0] // 256) * 256
    D_ref, S = oracle.gemm_bf16(gi.bf16_codes(A[r0:]), gi.bf16_codes(B))
    P.check_within_bound(P.bf16_to_f64(D[r0:]), D_ref, S, "ragged_k1040 tail rows")


def test_workload_square_4096():
    _sampled("square_4096", g.VARIANT_AUTO)


@pytest.mark.slow
def test_workload_square_8192():
    _sampled("square_8192", g.VARIANT_AUTO)


@pytest.mark.parametrize("v", list(VARIANTS))
@pytest.mark.parametrize("K, lda", [(1, 8), (3, 8), (100, 104), (70, 72), (1043, 1048)])
def test_k_tail_reads_nothing_past_k(v, K, lda):
    """The pitch padding [K, lda) holds large values; none may enter the sum."""
    M, N = 256, 512
    A = torch.ones(M, lda, dtype=torch.bfloat16)
    B = torch.ones(N, lda, dtype=torch.bfloat16)
    A[:, K:] = 1000.0
    B[:, K:] = 1000.0
    D = run(A, B, VARIANTS[v], K=K)
    D_ref, _ = ref(A, B, K)
    assert_bitwise(D, D_ref)


@pytest.mark.parametrize("v", ["1cta", "2cta", "auto"])
@pytest.mark.parametrize("N, ldd", [(300, 304), (300, 320), (260, 264), (1000, 1024)])
def test_ragged_n_never_writes_padding(v, N, ldd):
    """D as a column slice of a wider matrix: columns [N, ldd) belong to
    someone else and must keep their contents."""
    M, K = 261, 136
    A, B = gi.bf16_operands(M, N, K, seed=N)
    big = torch.full((M, ldd), -1234.0, dtype=torch.bfloat16, device="cuda")
    D = big[:, :N]
    Ad, Bd = A.cuda(), B.cuda()
    s = torch.cuda.current_stream().cuda_stream
    assert g.gemm_bf16_variant(VARIANTS[v], Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K, K,
                               K, ldd, s) == g.GEMM_OK
    assert g.gemm_last_status(s) == g.GEMM_OK
    host = big.cpu()
    assert torch.all(host[:, N:] == torch.tensor(-1234.0).to(torch.bfloat16))
    D_ref, S = ref(A, B)
    P.check_within_bound(P.bf16_to_f64(host[:, :N]), D_ref, S, f"N={N} ldd={ldd}/{v}")


# --------------------------------------------- small-K CUDA-core kernel (K <= 16)

SMALLK_VARIANTS = {"smallk": g.VARIANT_SMALLK, "smallk_tc": g.VARIANT_SMALLK_TC, "auto": g.VARIANT_AUTO}


@pytest.mark.parametrize("v", list(SMALLK_VARIANTS))
@pytest.mark.parametrize("M, N, K, lda, ldd", [(300, 520, 8, 8, 520), (4099, 2053, 8, 8, 2053),
                                               (129, 257, 1, 8, 264), (257, 300, 16, 16, 301),
                                               (33, 1031, 3, 8, 1031), (1, 1, 5, 8, 1)])
def test_smallk_small_integers_bitwise(v, M, N, K, lda, ldd):
    """Bitwise for both row-store forms: bf16 pairs (4-byte aligned rows) and
    single values (odd pitch: every other row), ragged M and N, padding left
    untouched."""
    variant = SMALLK_VARIANTS[v]
    gen = torch.Generator().manual_seed(M + N + K)
    A = torch.zeros(M, lda, dtype=torch.bfloat16)
    B = torch.zeros(N, lda, dtype=torch.bfloat16)
    A[:, :K] = torch.randint(-4, 5, (M, K), generator=gen).to(torch.bfloat16)
    B[:, :K] = torch.randint(-4, 5, (N, K), generator=gen).to(torch.bfloat16)
    A[:, K:] = float("nan")        # past K: never read
    B[:, K:] = float("nan")
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.full((M, ldd), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc = g.gemm_bf16_variant(variant, Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K, lda,
                             lda, ldd, 0)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    assert g.gemm_last_status(0) == g.GEMM_OK
    D = D.cpu()
    if ldd > N:
        assert torch.isnan(D[:, N:].float()).all()
    D_ref, _ = ref(A, B, K)
    assert_bitwise(D[:, :N], D_ref)


@pytest.mark.parametrize("v", ["smallk", "smallk_tc"])
@pytest.mark.parametrize("M, N, K, ldd, offset", [
    (64, 2053, 8, 2053, 0), (64, 2053, 8, 2053, 3), (40, 257, 5, 261, 1), (40, 255, 8, 255, 7),
    (48, 513, 12, 515, 2), (48, 127, 16, 133, 5), (70000, 40, 4, 41, 1), (300, 1, 8, 1, 1)])
def test_smallk_any_row_alignment(v, M, N, K, ldd, offset):
    """Rows that start at every element offset within a 16-byte line (odd
    pitches, D placed `offset` elements into its buffer), ragged column strips
    and a grid that walks several row tiles per block: bitwise, and nothing
    written before D, between rows or after the last row."""
    gen = torch.Generator().manual_seed(M + N + K + ldd)
    lda = (K + 7) // 8 * 8
    A = torch.zeros(M, lda, dtype=torch.bfloat16)
    B = torch.zeros(N, lda, dtype=torch.bfloat16)
    A[:, :K] = torch.randint(-4, 5, (M, K), generator=gen).to(torch.bfloat16)
    B[:, :K] = torch.randint(-4, 5, (N, K), generator=gen).to(torch.bfloat16)
    Ad, Bd = A.cuda(), B.cuda()
    buf = torch.full((offset + M * ldd + 64,), -1234.0, dtype=torch.bfloat16, device="cuda")
    dptr = buf.data_ptr() + 2 * offset
    rc = g.gemm_bf16_variant(SMALLK_VARIANTS[v], Ad.data_ptr(), Bd.data_ptr(), dptr, M, N, K, lda,
                             lda, ldd, 0)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    assert g.gemm_last_status(0) == g.GEMM_OK
    host = buf.cpu()
    sentinel = torch.tensor(-1234.0).to(torch.bfloat16)
    assert torch.all(host[:offset] == sentinel) and torch.all(host[offset + M * ldd:] == sentinel)
    D = host[offset:offset + M * ldd].view(M, ldd)
    assert torch.all(D[:, N:] == sentinel)
    D_ref, _ = ref(A, B, K)
    assert_bitwise(D[:, :N], D_ref)


@pytest.mark.slow
def test_smallk_auto_large_output():
    """K = 8 with a 52 MB output: the automatic choice takes the tensor-core
    small-K kernel; bitwise on small integers, odd pitch, padding untouched."""
    M, N, K, ldd = 8192, 3199, 8, 3201
    gen = torch.Generator().manual_seed(5)
    A = torch.randint(-4, 5, (M, K), generator=gen).to(torch.bfloat16)
    B = torch.randint(-4, 5, (N, K), generator=gen).to(torch.bfloat16)
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.full((M, ldd), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc = g.gemm_bf16(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K, K, K, ldd, 0)
    assert rc == g.GEMM_OK and g.gemm_last_status(0) == g.GEMM_OK
    D = D.cpu()
    assert torch.isnan(D[:, N:].float()).all()
    D_ref, _ = ref(A, B, K)
    assert_bitwise(D[:, :N], D_ref)


def test_smallk_rejects_an_odd_byte_address():
    A = torch.zeros(8, 8, dtype=torch.bfloat16, device="cuda")
    buf = torch.zeros(100, dtype=torch.uint8, device="cuda")
    rc = g.gemm_bf16_variant(g.VARIANT_SMALLK, A.data_ptr(), A.data_ptr(), buf.data_ptr() + 1, 8,
                             8, 8, 8, 8, 8, 0)
    assert rc == g.GEMM_ERR_ALIGNMENT


@pytest.mark.parametrize("v", ["smallk", "smallk_tc"])
@pytest.mark.parametrize("K", [3, 8, 13, 16])
def test_smallk_random_within_bound(v, K):
    A0, B0 = gi.bf16_operands(1000, 777, K, seed=41 + K)
    lda = (K + 7) // 8 * 8   # a pitch of whole 16-byte lines, NaN past K
    A = torch.full((1000, lda), float("nan"), dtype=torch.bfloat16)
    B = torch.full((777, lda), float("nan"), dtype=torch.bfloat16)
    A[:, :K], B[:, :K] = A0, B0
    D = run(A, B, SMALLK_VARIANTS[v], K=K)
    D_ref, S = ref(A, B, K)
    P.check_within_bound(P.bf16_to_f64(D), D_ref, S, "smallk random")


@pytest.mark.parametrize("v", ["smallk", "smallk_tc"])
def test_smallk_nonfinite(v):
    M, N, K = 64, 300, 8
    A = torch.ones(M, K, dtype=torch.bfloat16)
    B = torch.ones(N, K, dtype=torch.bfloat16)
    A[3, 2] = float("nan")
    A[7, 0] = float("inf")
    B[11, 0] = 0.0                          # inf * 0 = NaN at (7, 11)
    D = run(A, B, SMALLK_VARIANTS[v]).float()
    assert torch.isnan(D[3]).all()
    assert torch.isnan(D[7, 11]) and torch.isinf(D[7, 12]) and D[7, 12] > 0
    others = torch.ones(M, dtype=torch.bool)
    others[[3, 7]] = False
    cols = torch.ones(N, dtype=torch.bool)
    cols[11] = False
    assert torch.all(D[others][:, cols] == 8) and torch.all(D[others][:, 11] == 7)
