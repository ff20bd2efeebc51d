"""GPU MXFP8 quantiser through the C ABI, bit for bit against the oracle's
quantiser (and, at full size, against the independent torch-based input
encoder).  Codes and scale bytes are integers, so the bar is exact."""
import numpy as np
import pytest
import torch

import dense_gemm_blackwell_tcgen05_gb300 as g
import gemm_inputs as gi
import oracle
from tests import parity as P

pytestmark = pytest.mark.gpu


def gpu_quantize(X_cpu: np.ndarray, K=None, ldq_extra=0, ldsf=None):
    """X_cpu float32 [rows, ldx]; returns (Q [rows, K], SF [rows, nblk]) from the GPU."""
    rows, ldx = X_cpu.shape
    K = ldx if K is None else K
    nblk = (K + 31) // 32
    ldq = K + ldq_extra
    ldsf = nblk if ldsf is None else ldsf
    X = torch.from_numpy(np.ascontiguousarray(X_cpu)).cuda()
    Q = torch.full((rows, ldq), 0xAB, dtype=torch.uint8, device="cuda")
    SF = torch.full((rows, ldsf), 0xCD, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_mxfp8_quantize(X.data_ptr(), rows, K, ldx, Q.data_ptr(), ldq, SF.data_ptr(), ldsf, s)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    torch.cuda.synchronize()
    Qh, SFh = Q.cpu().numpy(), SF.cpu().numpy()
    assert np.all(Qh[:, K:] == 0xAB), "wrote past K"
    assert np.all(SFh[:, nblk:] == 0xCD), "wrote past the last scale block"
    return Qh[:, :K], SFh[:, :nblk]


def special_rows(K, seed):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((9, K)).astype(np.float32)
    X[1, :32] = 0.0
    X[2] *= 1e6
    X[3] *= 1e-7
    X[4, 5 % K] = 448.0 * 8
    if K > 40:
        X[4, 40] = np.float32(448.0 * 8 * (1 + 2 ** -20))
    X[5, ::7] = 1e-40                         # float32 subnormals
    X[6] *= 3e38 / max(1.0, float(np.abs(X[6]).max()))   # near the float32 maximum
    X[7, 3 % K] = -1e-30                      # rounds to -0 after scaling
    X[8] = np.float32(2.0 ** -140)            # every element subnormal
    return X


def assert_same(Q, SF, Qr, SFr):
    if not np.array_equal(SF, SFr):
        i, j = np.argwhere(SF != SFr)[0]
        raise AssertionError(f"scale byte ({i},{j}): gpu {SF[i, j]} oracle {SFr[i, j]}")
    if not np.array_equal(Q, Qr):
        i, j = np.argwhere(Q != Qr)[0]
        raise AssertionError(f"code ({i},{j}): gpu {Q[i, j]:#x} oracle {Qr[i, j]:#x}")


@pytest.mark.parametrize("K", [1, 31, 32, 101, 512, 1000, 8192])
def test_matches_oracle(K):
    X = special_rows(K, seed=K)
    Q, SF = gpu_quantize(X)
    assert_same(Q, SF, *oracle.mxfp8_quantize(X))


@pytest.mark.parametrize("extra", [1, 3, 4])
def test_pitches(extra):
    K = 200
    X = special_rows(K + extra, seed=extra)
    Q, SF = gpu_quantize(X, K=K, ldq_extra=extra, ldsf=16)
    assert_same(Q, SF, *oracle.mxfp8_quantize(X, K))


def test_nonfinite():
    X = np.ones((2, 64), np.float32)
    X[0, 3] = np.nan
    X[0, 7] = -np.inf
    X[1, 33] = np.inf
    Q, SF = gpu_quantize(X)
    assert_same(Q, SF, *oracle.mxfp8_quantize(X))


def test_full_size_workload_operands():
    """The MXFP8 workload's float32 operands: GPU codes equal the torch-based
    input encoder's on every element, and the oracle's on sampled rows."""
    w = gi.WORKLOADS["mxfp8_8192"]
    A, _ = gi.float_operands(w.M, w.N, w.K, w.seed, w.dist, w.scale)
    Xd = A.cuda()
    Q, SF = g.quantize_mxfp8(Xd)
    q_ref, sf_ref = gi.mxfp8_quantize(A)
    assert torch.equal(Q.cpu(), q_ref) and torch.equal(SF.cpu(), sf_ref)
    rows = np.random.default_rng(5).integers(0, w.M, 64)
    Qr, SFr = oracle.mxfp8_quantize(A.numpy()[rows])
    assert np.array_equal(Q.cpu().numpy()[rows], Qr)
    assert np.array_equal(SF.cpu().numpy()[rows][:, :SFr.shape[1]], SFr)


def test_quantise_then_gemm():
    """GPU quantiser feeding the GPU block-scaled GEMM agrees with the oracle
    quantiser feeding the oracle GEMM."""
    M, N, K = 300, 520, 384
    A, B = gi.float_operands(M, N, K, seed=31)
    qa, sfa = g.quantize_mxfp8(A.cuda())
    qb, sfb = g.quantize_mxfp8(B.cuda())
    D = g.matmul_mxfp8(qa, sfa, qb, sfb)
    assert g.gemm_last_status(torch.cuda.current_stream().cuda_stream) == g.GEMM_OK
    Qa, SFa = oracle.mxfp8_quantize(A.numpy())
    Qb, SFb = oracle.mxfp8_quantize(B.numpy())
    assert np.array_equal(qa.cpu().numpy(), Qa) and np.array_equal(qb.cpu().numpy(), Qb)
    D_ref, S = oracle.gemm_mxfp8(Qa, Qb, SFa, SFb)
    P.check_within_bound(P.bf16_to_f64(D), D_ref, S, "quantise->gemm")


@pytest.mark.parametrize("rows, K", [(1, 1), (127, 31), (128, 32), (129, 33), (300, 100),
                                     (257, 1040), (64, 4096)])
def test_quantize_tiled_layout(rows, K):
    """The tiled scale output: every byte of the buffer written -- the oracle's
    scales at their tiled positions, zero in the padding -- and the codes as
    in the row-major form."""
    rng = np.random.default_rng(rows + K)
    X_cpu = (rng.standard_normal((rows, K)) * rng.uniform(1e-3, 1e3, (rows, 1))).astype(np.float32)
    X = torch.from_numpy(X_cpu).cuda()
    n = (rows + 127) // 128 * (((K + 31) // 32 + 3) // 4) * 512
    Q = torch.full((rows, K), 0xAB, dtype=torch.uint8, device="cuda")
    SF = torch.full((n,), 0xCD, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_mxfp8_quantize_tiled(X.data_ptr(), rows, K, K, Q.data_ptr(), K, SF.data_ptr(), s)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    torch.cuda.synchronize()
    Qr, SFr = oracle.mxfp8_quantize(X_cpu)
    assert np.array_equal(Q.cpu().numpy(), Qr)
    want = gi.tile_scales(torch.from_numpy(np.ascontiguousarray(SFr)), rows, K).numpy()
    got = SF.cpu().numpy()
    assert got.shape == want.shape
    if not np.array_equal(got, want):
        i = int(np.flatnonzero(got != want)[0])
        raise AssertionError(f"tiled scale byte {i}: gpu {got[i]} want {want[i]}")


def test_quantize_tiled_feeds_the_tiled_gemm():
    """GPU-quantised operands with tiled scales into gemm_mxfp8_tiled, against
    the oracle on the oracle's own quantisation of the same floats."""
    M, N, K = 300, 520, 384
    XA, XB = gi.float_operands(M, N, K, seed=12)
    A, SFA = g.quantize_mxfp8_tiled(XA.cuda())
    B, SFB = g.quantize_mxfp8_tiled(XB.cuda())
    D = g.matmul_mxfp8_tiled(A, SFA, B, SFB)
    assert g.gemm_last_status(0) == g.GEMM_OK
    QA, SA = oracle.mxfp8_quantize(XA.numpy())
    QB, SB = oracle.mxfp8_quantize(XB.numpy())
    D_ref, S = oracle.gemm_mxfp8(QA, QB, SA, SB)
    P.check_within_bound(P.bf16_to_f64(D), D_ref, S, "quantised tiled gemm")
