"""Fused epilogue (gemm_bf16_fused / gemm_mxfp8_fused) on the GPU against the
oracle: D = act(alpha * A B^T + beta * C + bias[col]).

Bitwise where every step is exact in fp32 -- small-integer operands, C and
bias, power-of-two alpha and beta, ReLU or no activation -- so the only
rounding is the final one to the output type, taken the same way on both
sides.  Otherwise (GELU, random data) within the GEMM bound carried through
the epilogue:

    |D - D_ref| <= r |D_ref| + L (|alpha| 1e-3 S + 2^-18 (|alpha P| + |beta C| + |bias|))

with S = sum_k |a b|, P the exact product, L = 1.13 >= max |GELU'| (1 for the
others), and r = 2^-7 for a bf16 output, 2^-20 for fp32.  The 2^-18 term
covers the few fp32 roundings of the epilogue and erf's error."""
import numpy as np
import pytest
import torch

import dense_gemm_blackwell_tcgen05_gb300 as g
import gemm_inputs as gi
import oracle
from tests import parity as P
from tests.test_gemm_mxfp8 import int_operands as mx_int_operands

pytestmark = pytest.mark.gpu

ACT = {"none": 0, "relu": 1, "gelu": 2}
BF16_VARIANTS = {"auto": g.VARIANT_AUTO, "1cta": g.VARIANT_1CTA, "2cta": g.VARIANT_2CTA,
                 "1cta_direct": g.VARIANT_1CTA | g.VARIANT_DIRECT_STORE,
                 "2cta_direct": g.VARIANT_2CTA | g.VARIANT_DIRECT_STORE}
MX_VARIANTS = {"auto": g.VARIANT_AUTO, "1cta_tma": g.VARIANT_1CTA, "2cta": g.VARIANT_2CTA}


def ints(shape, seed, lo=-3, hi=4, dtype=torch.bfloat16):
    gen = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi, shape, generator=gen).to(dtype)


def f64(t):
    return t.double().numpy() if t.dtype != torch.bfloat16 else P.bf16_to_f64(t)


def run(A, B, variant, out_dtype, alpha=1.0, beta=0.0, C=None, bias=None, act="none",
        ldd=None, SFA=None, SFB=None):
    """One fused call; A, B (and C, bias, SFA, SFB) are CPU tensors."""
    M, K = A.shape
    N = B.shape[0]
    ldd = N if ldd is None else ldd
    D = torch.full((M, ldd), float("nan"), dtype=out_dtype, device="cuda")
    Cd = None if C is None else C.cuda()
    bd = None if bias is None else bias.cuda()
    e = g.make_epilogue(alpha, beta, Cd, bd, act, out_dtype)
    s = torch.cuda.current_stream().cuda_stream
    if SFA is None:
        Ad, Bd = A.cuda(), B.cuda()
        rc = g.gemm_bf16_fused(variant, Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K, K, K,
                               ldd, e, s)
    else:
        Ad, Bd, SAd, SBd = A.cuda(), B.cuda(), SFA.cuda(), SFB.cuda()
        rc = g.gemm_mxfp8_fused(variant, Ad.data_ptr(), Bd.data_ptr(), SAd.data_ptr(),
                                SBd.data_ptr(), D.data_ptr(), M, N, K, A.stride(0), B.stride(0),
                                SFA.stride(0), SFB.stride(0), ldd, e, s)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    assert g.gemm_last_status(s) == g.GEMM_OK
    D = D.cpu()
    if ldd > N:
        assert torch.isnan(D[:, N:].float()).all(), "wrote past N"
    return D[:, :N]


def reference(P_, S, alpha, beta, C, bias, act):
    Cf = None if C is None else f64(C)
    bf = None if bias is None else f64(bias)
    D_ref = oracle.epilogue(P_, alpha, beta, Cf, bf, ACT[act])
    scale = np.abs(alpha * P_)
    if Cf is not None:
        scale = scale + np.abs(beta * Cf[:, :P_.shape[1]])
    if bf is not None:
        scale = scale + np.abs(bf[None, :P_.shape[1]])
    return D_ref, S, scale


def assert_bitwise(D, D_ref, what):
    if D.dtype == torch.bfloat16:
        got, want = gi.bf16_codes(D), oracle.f64_to_bf16_rne(D_ref)
    else:
        got, want = D.numpy().view(np.uint32), D_ref.astype(np.float32).view(np.uint32)
    bad = np.argwhere(got != want)
    assert len(bad) == 0, f"{what}: {len(bad)} mismatches, first at {tuple(bad[0])}"


def assert_bound(D, D_ref, S, scale, alpha, act, what):
    r = 2.0 ** -7 if D.dtype == torch.bfloat16 else 2.0 ** -20
    L = 1.13 if act == "gelu" else 1.0
    got = f64(D)
    bound = r * np.abs(D_ref) + L * (abs(alpha) * 1e-3 * S + 2.0 ** -18 * scale) + 1e-30
    err = np.abs(got - D_ref)
    bad = ~(err <= bound)
    assert not bad.any(), (f"{what}: {bad.sum()} outside the bound; worst ratio "
                           f"{np.nanmax(err / bound):.3g}")


# ------------------------------------------------------------ exact cases

EXACT = [  # alpha, beta, C?, bias dtype, act
    (1.0, 0.0, False, None, "relu"),
    (0.5, 1.0, True, torch.bfloat16, "none"),
    (-2.0, -0.25, True, torch.float32, "relu"),
    (1.0, 2.0, True, None, "relu"),
    (0.25, 0.0, False, torch.bfloat16, "none"),
]


@pytest.mark.parametrize("v", list(BF16_VARIANTS))
@pytest.mark.parametrize("out", ["bf16", "f32"])
@pytest.mark.parametrize("case", range(len(EXACT)))
def test_bf16_exact(v, out, case):
    alpha, beta, use_c, bias_dt, act = EXACT[case]
    out_dtype = torch.bfloat16 if out == "bf16" else torch.float32
    M, N, K = 300, 520, 200
    A, B = ints((M, K), 1 + case), ints((N, K), 2 + case)
    C = ints((M, N + 8), 3 + case, -8, 9, out_dtype) if use_c else None
    bias = ints((N,), 4 + case, -8, 9, bias_dt) if bias_dt is not None else None
    D = run(A, B, BF16_VARIANTS[v], out_dtype, alpha, beta, C, bias, act)
    P_, S = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B))
    D_ref, _, _ = reference(P_, S, alpha, beta, C, bias, act)
    assert_bitwise(D, D_ref, f"{v}/{out}/{EXACT[case]}")


@pytest.mark.parametrize("v", list(MX_VARIANTS))
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_mxfp8_exact(v, out):
    out_dtype = torch.bfloat16 if out == "bf16" else torch.float32
    M, N, K = 257, 448, 256
    # integer E4M3 values up to 2 and scales 2^-3 .. 2^3: 22 significant bits
    # at most, so alpha acc - C + bias stays exact in fp32
    A, SFA, B, SFB = mx_int_operands(M, N, K, seed=21, imax=2, sf_lo=124, sf_hi=130)
    C = ints((M, N), 5, -8, 9, out_dtype)
    bias = ints((N,), 6, -8, 9, torch.float32)
    D = run(A, B, MX_VARIANTS[v], out_dtype, 0.5, -1.0, C, bias, "relu", SFA=SFA, SFB=SFB)
    P_, S = oracle.gemm_mxfp8(A.numpy(), B.numpy(), SFA.numpy(), SFB.numpy(), K)
    D_ref, _, _ = reference(P_, S, 0.5, -1.0, C, bias, "relu")
    assert_bitwise(D, D_ref, f"mxfp8 {v}/{out}")


def test_in_place_update():
    """C == D: D <- A B^T + D."""
    M, N, K = 300, 520, 128
    A, B = ints((M, K), 7), ints((N, K), 8)
    D0 = ints((M, N), 9, -8, 9)
    D = D0.cuda()
    e = g.make_epilogue(1.0, 1.0, D, None, "none", torch.bfloat16)
    Ad, Bd = A.cuda(), B.cuda()
    rc = g.gemm_bf16_fused(g.VARIANT_AUTO, Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K, K,
                           K, N, e, 0)
    assert rc == g.GEMM_OK and g.gemm_last_status(0) == g.GEMM_OK
    P_, S = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B))
    D_ref, _, _ = reference(P_, S, 1.0, 1.0, D0, None, "none")
    assert_bitwise(D.cpu(), D_ref, "in place")


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_k_zero(out):
    out_dtype = torch.bfloat16 if out == "bf16" else torch.float32
    M, N = 130, 70
    A = torch.zeros(M, 8, dtype=torch.bfloat16)
    B = torch.zeros(N, 8, dtype=torch.bfloat16)
    C = ints((M, N + 2), 10, -8, 9, out_dtype)
    bias = ints((N,), 11, -8, 9, torch.bfloat16)
    D = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
    Cd, bd = C.cuda(), bias.cuda()
    e = g.make_epilogue(3.0, -0.5, Cd, bd, "relu", out_dtype)
    Ad, Bd = A.cuda(), B.cuda()   # never read with K = 0, but kept alive all the same
    rc = g.gemm_bf16_fused(g.VARIANT_AUTO, Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(),
                           M, N, 0, 8, 8, N, e, 0)
    assert rc == g.GEMM_OK and g.gemm_last_status(0) == g.GEMM_OK
    D_ref = oracle.epilogue(np.zeros((M, N)), 3.0, -0.5, f64(C), f64(bias), 1)
    assert_bitwise(D.cpu(), D_ref, "k=0")


# ------------------------------------------------------ GELU and random data

@pytest.mark.parametrize("v", ["auto", "1cta", "2cta_direct"])
@pytest.mark.parametrize("out", ["bf16", "f32"])
@pytest.mark.parametrize("act", ["gelu", "relu", "none"])
def test_bf16_random_within_bound(v, out, act):
    out_dtype = torch.bfloat16 if out == "bf16" else torch.float32
    M, N, K = 257, 300, 1040
    A, B = gi.bf16_operands(M, N, K, seed=31)
    gen = torch.Generator().manual_seed(32)
    C = torch.randn(M, N + 3, generator=gen).to(out_dtype)
    bias = torch.randn(N, generator=gen)
    D = run(A, B, BF16_VARIANTS[v], out_dtype, 0.7, -1.3, C, bias, act)
    P_, S = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B))
    D_ref, S, scale = reference(P_, S, 0.7, -1.3, C, bias, act)
    assert_bound(D, D_ref, S, scale, 0.7, act, f"{v}/{out}/{act}")


@pytest.mark.parametrize("v", list(MX_VARIANTS))
def test_mxfp8_gelu_within_bound(v):
    M, N, K = 300, 520, 1024
    A, SFA, B, SFB = gi.mxfp8_operands(M, N, K, seed=33)
    gen = torch.Generator().manual_seed(34)
    bias = torch.randn(N, generator=gen).to(torch.bfloat16)
    D = run(A, B, MX_VARIANTS[v], torch.float32, 0.125, 0.0, None, bias, "gelu", SFA=SFA, SFB=SFB)
    P_, S = oracle.gemm_mxfp8(A.numpy(), B.numpy(), SFA.numpy(), SFB.numpy(), K)
    D_ref, S, scale = reference(P_, S, 0.125, 0.0, None, bias, "gelu")
    assert_bound(D, D_ref, S, scale, 0.125, "gelu", f"mxfp8 {v}")


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_odd_pitches_and_ragged_edges(out):
    """Pitches that are not multiples of 16 bytes (scalar C loads and
    stores), ragged M and N, D padding left untouched."""
    out_dtype = torch.bfloat16 if out == "bf16" else torch.float32
    M, N, K = 131, 301, 64
    A, B = ints((M, K), 12), ints((N, K), 13)
    C = ints((M, N + 6), 14, -8, 9, out_dtype)[:, :N + 5]      # pitch N + 5 (odd)
    C = C.contiguous()
    bias = ints((N,), 15, -8, 9, torch.bfloat16)
    D = run(A, B, g.VARIANT_AUTO, out_dtype, -1.0, 0.5, C, bias, "relu", ldd=N + 7)
    P_, S = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B))
    D_ref, _, _ = reference(P_, S, -1.0, 0.5, C, bias, "relu")
    assert_bitwise(D, D_ref, f"odd pitches {out}")


@pytest.mark.parametrize("v", ["1cta", "2cta"])
def test_c_by_tma_matches_loaded_c(v):
    """The pair's TMA-store kernel brings a 16-byte-aligned bf16 C in by TMA,
    one 64-column chunk ahead; the masked-store kernels load it per thread (a
    fused epilogue on one CTA always takes the masked-store kernel).  The
    arithmetic after that is the same, so the two agree bit for bit on random
    data (GELU, ragged edges, C pitch other than D's, several chunks and tiles
    per CTA), and both stay within the bound of the oracle."""
    M, N, K = 1100, 1800, 256
    A, B = gi.bf16_operands(M, N, K, seed=31)
    gen = torch.Generator().manual_seed(32)
    C = torch.randn(M, N + 24, generator=gen).to(torch.bfloat16)
    bias = torch.randn(N, generator=gen).to(torch.bfloat16)
    args = (torch.bfloat16, 0.5, -1.5, C, bias, "gelu")
    D_tma = run(A, B, BF16_VARIANTS[v], *args)
    D_ldg = run(A, B, BF16_VARIANTS[v + "_direct"], *args)
    got, want = gi.bf16_codes(D_tma), gi.bf16_codes(D_ldg)
    bad = np.argwhere(got != want)
    assert len(bad) == 0, f"{v}: {len(bad)} elements differ, first at {tuple(bad[0])}"
    P_, S = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B))
    D_ref, S, scale = reference(P_, S, 0.5, -1.5, C, bias, "gelu")
    assert_bound(D_tma, D_ref, S, scale, 0.5, "gelu", f"C by TMA {v}")


def test_c_by_tma_at_an_offset_base():
    """C starting 16 bytes past an allocation's start (still TMA-aligned) with
    a pitch other than D's: the TMA path reads the right rows and columns."""
    M, N, K = 700, 1032, 128
    A, B = ints((M, K), 51), ints((N, K), 52)
    gen = torch.Generator().manual_seed(53)
    Cbig = torch.randint(-8, 9, (M * (N + 40) + 8,), generator=gen).to(torch.bfloat16).cuda()
    Cview = Cbig[8:8 + M * (N + 40)].view(M, N + 40)[:, :N]          # base + 16 bytes, pitch N + 40
    e = g.make_epilogue(1.0, -1.0, Cview, None, "none", torch.bfloat16)
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc = g.gemm_bf16_fused(g.VARIANT_2CTA, Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K,
                           K, K, N, e, 0)
    assert rc == g.GEMM_OK and g.gemm_last_status(0) == g.GEMM_OK
    P_, S = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B))
    D_ref, _, _ = reference(P_, S, 1.0, -1.0, Cview.cpu(), None, "none")
    assert_bitwise(D.cpu(), D_ref, "C at an offset base")


def test_c_by_tma_in_place_over_several_waves():
    """C == D through the TMA path on a shape with more tiles than clusters:
    each chunk of C is read before the same chunk of D is stored."""
    M, N, K = 2600, 2000, 64
    A, B = ints((M, K), 41), ints((N, K), 42)
    D0 = ints((M, N), 43, -8, 9)
    D = D0.cuda()
    e = g.make_epilogue(2.0, -1.0, D, None, "relu", torch.bfloat16)
    Ad, Bd = A.cuda(), B.cuda()
    rc = g.gemm_bf16_fused(g.VARIANT_2CTA, Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K,
                           K, K, N, e, 0)
    assert rc == g.GEMM_OK and g.gemm_last_status(0) == g.GEMM_OK
    P_, S = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B))
    D_ref, _, _ = reference(P_, S, 2.0, -1.0, D0, None, "relu")
    assert_bitwise(D.cpu(), D_ref, "in place, several waves")


def test_relu_keeps_nan():
    M, N, K = 128, 256, 64
    A, B = ints((M, K), 16), ints((N, K), 17)
    A[5, 3] = float("nan")
    D = run(A, B, g.VARIANT_AUTO, torch.float32, 1.0, 0.0, None, None, "relu")
    assert torch.isnan(D[5]).all()
    assert not torch.isnan(D[torch.arange(M) != 5]).any()


# ------------------------------------------------------------- argument errors

def test_epilogue_validation():
    M = N = K = 256
    A = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    D = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    f = lambda e, v=g.VARIANT_AUTO, ldd=N: g.gemm_bf16_fused(
        v, A.data_ptr(), A.data_ptr(), D.data_ptr(), M, N, K, K, K, ldd, e, 0)
    ok = g.make_epilogue()
    assert f(ok) == g.GEMM_OK
    assert f(None) == g.GEMM_OK
    bad = g.make_epilogue(); bad.activation = 3
    assert f(bad) == g.GEMM_ERR_INVALID_ARG
    bad = g.make_epilogue(); bad.out_dtype = 2
    assert f(bad) == g.GEMM_ERR_INVALID_ARG
    bad = g.make_epilogue(); bad.reserved = 1
    assert f(bad) == g.GEMM_ERR_INVALID_ARG
    bad = g.make_epilogue(beta=1.0, C=D); bad.ldc = N - 1
    assert f(bad) == g.GEMM_ERR_INVALID_ARG                          # ldc < N
    D2 = torch.zeros(M, N + 8, dtype=torch.bfloat16, device="cuda")
    alias = g.make_epilogue(beta=1.0, C=D2)                          # C == D, other pitch
    assert g.gemm_bf16_fused(g.VARIANT_AUTO, A.data_ptr(), A.data_ptr(), D2.data_ptr(), M, N, K,
                             K, K, N, alias, 0) == g.GEMM_ERR_INVALID_ARG
    host_bias = torch.zeros(N)
    bad = g.make_epilogue(bias=host_bias)
    assert f(bad) == g.GEMM_ERR_INVALID_ARG
    bad = g.make_epilogue(bias=torch.zeros(N, device="cuda")); bad.bias_dtype = 5
    assert f(bad) == g.GEMM_ERR_INVALID_ARG
    assert f(ok, v=g.VARIANT_SYNC) == g.GEMM_ERR_INVALID_ARG
    torch.cuda.synchronize()


def test_matmul_fused_wrapper():
    A, B = ints((200, 128), 18), ints((300, 128), 19)
    bias = ints((300,), 20, -8, 9, torch.float32)
    D = g.matmul_fused(A.cuda(), B.cuda(), alpha=2.0, bias=bias.cuda(), activation="relu",
                       out_dtype=torch.float32)
    P_, S = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B))
    D_ref, _, _ = reference(P_, S, 2.0, 0.0, None, bias, "relu")
    assert_bitwise(D.cpu(), D_ref, "matmul_fused")


# ------------------------------------------- the fused workloads, full size

def _workload_sampled(name, n=3000):
    """The bench's configuration of a fused workload (automatic variant),
    checked on sampled outputs: oracle sums there, then the oracle epilogue."""
    w = gi.WORKLOADS[name]
    sp = gi.epilogue_spec(w)
    A, B = gi.workload_operands(name)
    C, bias = gi.epilogue_operands(w)
    out_dtype = torch.float32 if sp["out"] == "f32" else torch.bfloat16
    D = g.matmul_fused(A.cuda(), B.cuda(), alpha=sp["alpha"], beta=sp["beta"],
                       C=None if C is None else C.cuda(), bias=None if bias is None else bias.cuda(),
                       activation=sp["act"], out_dtype=out_dtype)
    assert g.gemm_last_status(0) == g.GEMM_OK
    rows, cols = P.sample_positions(w.M, w.N, n, seed=w.seed)
    P_, S = oracle.gemm_bf16_entries(gi.bf16_codes(A), gi.bf16_codes(B), rows, cols)
    Cs = None if C is None else f64(C)[rows, cols][None, :]
    bs = None if bias is None else f64(bias)[cols]
    D_ref = oracle.epilogue(np.asarray(P_).reshape(1, -1), sp["alpha"], sp["beta"], Cs, bs,
                            ACT[sp["act"]])[0]
    scale = np.abs(sp["alpha"] * np.asarray(P_))
    if Cs is not None:
        scale = scale + np.abs(sp["beta"] * Cs[0])
    if bs is not None:
        scale = scale + np.abs(bs)
    got = f64(D.cpu())[rows, cols]
    r = 2.0 ** -7 if out_dtype == torch.bfloat16 else 2.0 ** -20
    L = 1.13 if sp["act"] == "gelu" else 1.0
    bound = r * np.abs(D_ref) + L * (abs(sp["alpha"]) * 1e-3 * np.asarray(S) + 2.0 ** -18 * scale)
    assert np.all(np.abs(got - D_ref) <= bound), name


@pytest.mark.slow
@pytest.mark.parametrize("name", ["fused_gelu_8192", "fused_f32_8192"])
def test_fused_workloads_full_size(name):
    _workload_sampled(name)
