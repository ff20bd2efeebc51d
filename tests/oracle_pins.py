"""Pins for the CPU oracle: checks against facts that do not come from it.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with a value fixed by a number-format definition (checked
through torch's own conversions of every bit pattern), by exact rational
arithmetic on tiny inputs, or by a closed form (all-ones, identity, K=1 outer
product, small-integer products, NaN/Inf propagation).  The shapes are
asymmetric (M != N != K, leading dimensions wider than K) so that a
transposed operand, a swapped index or an ignored stride changes the result.

``test_oracle.py`` runs every pin on the real oracle; ``test_oracle_mutants.py``
runs them on deliberately broken copies of it and requires each copy to fail
at least one pin.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import torch

BF16_ONE = 0x3F80


# ------------------------------------------------------------------ helpers

def torch_bf16_f64(codes: np.ndarray) -> np.ndarray:
    """bf16 codes -> float64 through torch's own conversion."""
    t = torch.from_numpy(np.ascontiguousarray(codes).view(np.int16)).view(torch.bfloat16)
    return t.double().numpy()


def torch_e4m3_f64(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn)
    return t.float().double().numpy()


def random_bf16_codes(rng: np.random.Generator, shape, scale=1.0) -> np.ndarray:
    x = torch.from_numpy(rng.standard_normal(shape).astype(np.float32) * np.float32(scale))
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def random_e4m3_codes(rng: np.random.Generator, shape) -> np.ndarray:
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3F          # no NaN codes
    return c


def same(a: np.ndarray, b: np.ndarray) -> bool:
    """Equal as values, NaN equal to NaN."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return a.shape == b.shape and bool(np.all((a == b) | (np.isnan(a) & np.isnan(b))))


def exact_dot(avals, bvals) -> tuple[Fraction, Fraction]:
    s = Fraction(0)
    sa = Fraction(0)
    for a, b in zip(avals, bvals):
        p = a * b
        s += p
        sa += abs(p)
    return s, sa


# --------------------------------------------------------- number formats

def pin_bf16_decode_all(o):
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    assert same(o.bf16_to_f64(codes), torch_bf16_f64(codes)), "bf16 decode"


def pin_e4m3_decode_all(o):
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    got = o.e4m3_to_f64(codes)
    assert same(got, torch_e4m3_f64(codes)), "E4M3 decode"
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF])


def pin_ue8m0_decode_all(o):
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    got = o.ue8m0_to_f64(codes)
    if hasattr(torch, "float8_e8m0fnu"):
        ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).float().double().numpy()
        assert same(got, ref), "UE8M0 decode"
    assert got[127] == 1.0 and got[128] == 2.0 and got[126] == 0.5
    assert np.isnan(got[255])


def pin_bf16_rne(o):
    rng = np.random.default_rng(11)
    vals = [rng.standard_normal(4000).astype(np.float32),
            (rng.standard_normal(1000) * 1e-38).astype(np.float32),       # bf16 subnormals
            (rng.standard_normal(1000) * 1e38).astype(np.float32)]
    # exact midpoints between neighbouring bf16 values (ties): 9 significant bits
    mids = []
    for code in rng.integers(0x0080, 0x7F00, size=2000):
        lo = np.array([code], np.uint32) << 16
        mids.append((lo + (1 << 15)).view(np.float32)[0])
    vals.append(np.array(mids, np.float32))
    vals.append(-np.array(mids, np.float32))
    vals.append(np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, 3.4e38], np.float32))
    v = np.concatenate(vals)
    got = o.f64_to_bf16_rne(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref), "bf16 RNE"
    assert o.f64_to_bf16_rne(np.array([np.nan]))[0] & 0x7FFF > 0x7F80


# ------------------------------------------------------------- bf16 GEMM

def pin_bruteforce_bf16(o):
    rng = np.random.default_rng(1)
    for (M, N, K, lda, ldb) in [(3, 5, 7, 9, 8), (5, 2, 40, 40, 48), (1, 4, 33, 36, 33),
                                (4, 3, 1, 3, 1)]:
        A = random_bf16_codes(rng, (M, lda), 4.0)
        B = random_bf16_codes(rng, (N, ldb), 0.25)
        D, S = o.gemm_bf16(A, B, K)
        Af = torch_bf16_f64(A)
        Bf = torch_bf16_f64(B)
        for i in range(M):
            for j in range(N):
                s, sa = exact_dot([Fraction(x) for x in Af[i, :K]],
                                  [Fraction(x) for x in Bf[j, :K]])
                tol = K * 2.0 ** -52 * float(sa)
                assert abs(Fraction(D[i, j]) - s) <= Fraction(tol), ("bf16 brute", M, N, K, i, j)
                assert abs(Fraction(S[i, j]) - sa) <= Fraction(tol), ("abs sum", i, j)


def pin_all_ones(o):
    for K in (1, 8, 64, 1040, 4096):
        A = np.full((3, K + 8), BF16_ONE, np.uint16)
        B = np.full((5, K), BF16_ONE, np.uint16)
        D, S = o.gemm_bf16(A, B, K)
        assert np.all(D == K) and np.all(S == K), ("all ones", K)


def pin_identity(o):
    rng = np.random.default_rng(2)
    for K, N in ((128, 37), (256, 5), (16, 300)):
        A = np.zeros((K, K), np.uint16)
        A[np.arange(K), np.arange(K)] = BF16_ONE
        B = random_bf16_codes(rng, (N, K))
        D, _ = o.gemm_bf16(A, B)
        assert same(D, torch_bf16_f64(B).T), ("identity", K, N)


def pin_k1_outer(o):
    rng = np.random.default_rng(3)
    A = random_bf16_codes(rng, (6, 1), 3.0)
    B = random_bf16_codes(rng, (9, 1), 0.5)
    D, _ = o.gemm_bf16(A, B)
    assert same(D, np.outer(torch_bf16_f64(A)[:, 0], torch_bf16_f64(B)[:, 0])), "K=1"


def pin_small_int_bf16(o):
    rng = np.random.default_rng(4)
    M, N, K = 13, 7, 70
    Ai = rng.integers(-2, 3, size=(M, K))
    Bi = rng.integers(-2, 3, size=(N, K))
    A = torch.from_numpy(Ai.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    B = torch.from_numpy(Bi.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    D, S = o.gemm_bf16(A, B)
    assert np.array_equal(D, (Ai @ Bi.T).astype(np.float64)), "small integers"
    assert np.array_equal(S, (np.abs(Ai) @ np.abs(Bi).T).astype(np.float64)), "small integer |.|"


def pin_entries_bf16(o):
    rng = np.random.default_rng(5)
    A = random_bf16_codes(rng, (17, 50))
    B = random_bf16_codes(rng, (11, 50))
    D, S = o.gemm_bf16(A, B, 45)
    rows = rng.integers(0, 17, 40)
    cols = rng.integers(0, 11, 40)
    De, Se = o.gemm_bf16_entries(A, B, rows, cols, 45)
    assert np.array_equal(De, D[rows, cols]) and np.array_equal(Se, S[rows, cols]), "entries"


def pin_nonfinite(o):
    A = np.full((4, 6), BF16_ONE, np.uint16)
    B = np.full((3, 6), BF16_ONE, np.uint16)
    A[2, 3] = 0x7FC0                  # NaN in row 2
    A[1, 0] = 0x7F80                  # +Inf in row 1 ...
    B[2, 0] = 0x0000                  # ... meets a zero in column 2: Inf * 0 = NaN
    D, _ = o.gemm_bf16(A, B)
    assert np.all(np.isnan(D[2])), "NaN row"
    assert np.isposinf(D[1, 0]) and np.isposinf(D[1, 1]) and np.isnan(D[1, 2]), "Inf row"
    assert np.all(np.isfinite(D[[0, 3]])), "finite rows"


# ------------------------------------------------------------ MXFP8 GEMM

def _mx_exact_values(codes, sf, K):
    dec = torch_e4m3_f64(codes)
    rows = []
    for r in range(codes.shape[0]):
        rows.append([Fraction(dec[r, k]) * Fraction(2) ** (int(sf[r, k // 32]) - 127)
                     for k in range(K)])
    return rows


def pin_bruteforce_mxfp8(o):
    rng = np.random.default_rng(6)
    for (M, N, K) in [(3, 4, 40), (2, 5, 97), (4, 1, 64)]:
        nblk = (K + 31) // 32
        A = random_e4m3_codes(rng, (M, K + 16))
        B = random_e4m3_codes(rng, (N, K))
        SFA = rng.integers(112, 142, size=(M, nblk + 3), dtype=np.uint8)
        SFB = rng.integers(112, 142, size=(N, nblk), dtype=np.uint8)
        D, S = o.gemm_mxfp8(A, B, SFA, SFB, K)
        av = _mx_exact_values(A, SFA, K)
        bv = _mx_exact_values(B, SFB, K)
        for i in range(M):
            for j in range(N):
                s, sa = exact_dot(av[i], bv[j])
                tol = Fraction(K * 2.0 ** -52) * sa
                assert abs(Fraction(D[i, j]) - s) <= tol, ("mxfp8 brute", M, N, K, i, j)
                assert abs(Fraction(S[i, j]) - sa) <= tol, ("mxfp8 abs sum", i, j)


def pin_small_int_mxfp8(o):
    """Integer E4M3 values with per-(row, block) power-of-two scales: every
    partial sum is exact, so D equals an integer product rescaled exactly."""
    rng = np.random.default_rng(7)
    M, N, K = 9, 6, 160
    nblk = K // 32
    Ai = rng.integers(-4, 5, size=(M, K))
    Bi = rng.integers(-4, 5, size=(N, K))
    ea = rng.integers(120, 135, size=(M, nblk))
    eb = rng.integers(120, 135, size=(N, nblk))
    A = torch.from_numpy(Ai.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    B = torch.from_numpy(Bi.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    D, _ = o.gemm_mxfp8(A, B, ea.astype(np.uint8), eb.astype(np.uint8))
    for i in range(M):
        for j in range(N):
            ref = Fraction(0)
            for b in range(nblk):
                blk = int(Ai[i, 32 * b:32 * b + 32] @ Bi[j, 32 * b:32 * b + 32])
                ref += blk * Fraction(2) ** (int(ea[i, b]) + int(eb[j, b]) - 254)
            assert Fraction(D[i, j]) == ref, ("mxfp8 integers", i, j)


def pin_identity_mxfp8(o):
    rng = np.random.default_rng(8)
    K, N = 96, 7
    A = np.zeros((K, K), np.uint8)
    A[np.arange(K), np.arange(K)] = 0x38          # E4M3 1.0
    SFA = np.full((K, 3), 127, np.uint8)          # scale 1
    B = random_e4m3_codes(rng, (N, K))
    SFB = rng.integers(120, 135, size=(N, 3), dtype=np.uint8)
    D, _ = o.gemm_mxfp8(A, B, SFA, SFB)
    ref = np.array([[float(v) for v in row] for row in _mx_exact_values(B, SFB, K)]).T
    assert same(D, ref), "mxfp8 identity"


def pin_entries_mxfp8(o):
    rng = np.random.default_rng(9)
    A = random_e4m3_codes(rng, (8, 80))
    B = random_e4m3_codes(rng, (6, 80))
    SFA = rng.integers(120, 135, size=(8, 3), dtype=np.uint8)
    SFB = rng.integers(120, 135, size=(6, 3), dtype=np.uint8)
    D, S = o.gemm_mxfp8(A, B, SFA, SFB, 70)
    rows = rng.integers(0, 8, 30)
    cols = rng.integers(0, 6, 30)
    De, Se = o.gemm_mxfp8_entries(A, B, SFA, SFB, rows, cols, 70)
    assert np.array_equal(De, D[rows, cols]) and np.array_equal(Se, S[rows, cols]), "mx entries"


# ------------------------------------------------------ MXFP8 quantisation

def _e4m3_table():
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    vals = torch_e4m3_f64(codes)
    ok = ~np.isnan(vals)
    return codes[ok], vals[ok]


def _nearest_e4m3(x: float) -> int:
    """Brute force: the E4M3 code nearest to x, ties to the even code, zero
    keeping the sign of x."""
    codes, vals = _e4m3_table()
    d = np.abs(vals - x)
    best = codes[d == d.min()]
    if len(best) > 1:
        even = [c for c in best if (c & 1) == 0]
        best = even or list(best)
    c = int(best[0])
    if vals[codes == c][0] == 0.0:
        c = 0x80 if np.signbit(x) else 0x00
    return c


def pin_e4m3_encode(o):
    codes, vals = _e4m3_table()
    got = o.f64_to_e4m3_rne(vals)
    assert np.array_equal(got, codes), "encode(decode(c)) != c"
    # midpoints between neighbours and random values against brute force
    fin = np.sort(np.unique(vals[vals >= 0]))
    mids = (fin[1:] + fin[:-1]) / 2
    rng = np.random.default_rng(12)
    xs = np.concatenate([mids, -mids, rng.uniform(-448, 448, 300), rng.uniform(-1e-2, 1e-2, 100)])
    want = np.array([_nearest_e4m3(float(x)) for x in xs], np.uint8)
    assert np.array_equal(o.f64_to_e4m3_rne(xs), want), "E4M3 rounding"
    x32 = rng.uniform(-448, 448, 500).astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(o.f64_to_e4m3_rne(x32.astype(np.float64)), ref), "vs torch cast"


def _quant_inputs():
    rng = np.random.default_rng(13)
    X = rng.standard_normal((6, 101)).astype(np.float32)
    X[1, :32] = 0.0                              # an all-zero block
    X[2] *= 1e6                                  # large
    X[3] *= 1e-7                                 # small
    X[4, 5] = 448.0 * 8                          # amax exactly 448 * 2^3
    X[4, 40] = np.float32(448.0 * 8 * (1 + 2 ** -20))   # just above a boundary
    X[5, 3] = 1e-40                              # a float32 subnormal
    return X


def pin_quantize_definition(o):
    X = _quant_inputs()
    Q, SF = o.mxfp8_quantize(X)
    K = X.shape[1]
    for r in range(X.shape[0]):
        for b in range((K + 31) // 32):
            blk = X[r, 32 * b:32 * b + 32].astype(np.float64)
            amax = np.abs(blk).max()
            e = int(SF[r, b]) - 127
            if amax == 0:
                assert e == -127
            else:
                assert amax <= 448.0 * 2.0 ** e and amax > 448.0 * 2.0 ** (e - 1), (r, b)
            for t, x in enumerate(blk):
                assert Q[r, 32 * b + t] == _nearest_e4m3(float(x) * 2.0 ** -e), (r, b, t)


def pin_quantize_vs_inputs_encoder(o):
    """The oracle's quantiser and the torch-based input encoder are written
    independently; on finite inputs they must agree bit for bit."""
    import gemm_inputs as gi
    X = _quant_inputs()
    Q, SF = o.mxfp8_quantize(X)
    q2, sf2 = gi.mxfp8_quantize(torch.from_numpy(X))
    assert np.array_equal(Q, q2.numpy()) and np.array_equal(SF, sf2.numpy()[:, :SF.shape[1]])


def pin_quantize_nonfinite(o):
    X = np.ones((2, 40), np.float32)
    X[0, 3] = np.nan
    X[0, 7] = -np.inf
    X[1, 33] = np.inf
    Q, SF = o.mxfp8_quantize(X)
    assert Q[0, 3] & 0x7F == 0x7F and Q[0, 7] == 0xFF and Q[1, 33] == 0x7F
    assert SF[0, 0] == 127 - 8 and SF[1, 1] == 127 - 8      # scale from the finite 1.0s
    assert np.all(Q[0, [0, 1, 2]] == _nearest_e4m3(2.0 ** 8))


# ---------------------------------------------------------- fused epilogue

def _gelu_ref(v: float) -> float:
    """v * Phi(v) with Python's math.erf (an independent libm path)."""
    import math
    return v * 0.5 * (1.0 + math.erf(v / math.sqrt(2.0)))


def pin_epilogue_bruteforce(o):
    """act(alpha sum + beta C + bias[j]) on tiny asymmetric shapes, the sums
    exact in rationals, the rest in Python floats: a bias taken per row, a
    beta applied to the product, an ignored C pitch or a mixed-up activation
    changes a value."""
    rng = np.random.default_rng(9)
    M, N, K, lda = 3, 5, 7, 9
    A = random_bf16_codes(rng, (M, lda), 2.0)
    B = random_bf16_codes(rng, (N, K), 1.0)
    P, _ = o.gemm_bf16(A, B, K)
    C = rng.standard_normal((M, N + 3))
    bias = rng.standard_normal(N)
    Af, Bf = torch_bf16_f64(A), torch_bf16_f64(B)
    for act in (0, 1, 2):
        for alpha, beta, use_c, use_b in [(1.5, -0.75, True, True), (-2.0, 0.0, False, True),
                                          (0.25, 3.0, True, False)]:
            out = o.epilogue(P, alpha, beta, C if use_c else None, bias if use_b else None, act)
            for i in range(M):
                for j in range(N):
                    s, _ = exact_dot([Fraction(x) for x in Af[i, :K]], [Fraction(x) for x in Bf[j, :K]])
                    v = alpha * float(s) + (beta * C[i, j] if use_c else 0.0) + (bias[j] if use_b else 0.0)
                    want = v if act == 0 else (max(v, 0.0) if act == 1 else _gelu_ref(v))
                    assert abs(out[i, j] - want) <= 1e-12 * (1.0 + abs(want)), ("epilogue", act, i, j)


def pin_gelu_textbook(o):
    """GELU(x) = x Phi(x) at points where the standard normal distribution
    function has well-known values: Phi(0) = 1/2, Phi(1) = 0.8413447460685429,
    Phi(2) = 0.9772498680518208, Phi(-x) = 1 - Phi(x)."""
    P = np.array([[0.0, 1.0, -1.0, 2.0, -2.0]])
    out = o.epilogue(P, act=2)[0]
    want = [0.0, 0.8413447460685429, -(1.0 - 0.8413447460685429), 2 * 0.9772498680518208,
            -2 * (1.0 - 0.9772498680518208)]
    assert np.allclose(out, want, rtol=1e-14, atol=1e-15), out
    # odd part: GELU(x) - GELU(-x) = x for any x
    xs = np.linspace(-6, 6, 25).reshape(1, -1)
    g = o.epilogue(xs, act=2)[0]
    assert np.allclose(g - g[::-1], xs[0], rtol=0, atol=1e-14)


def pin_relu_and_identity(o):
    P = np.array([[-3.5, -0.0, 0.0, 2.25, np.nan, -np.inf, np.inf]])
    r = o.epilogue(P, act=1)[0]
    assert r[0] == 0.0 and r[3] == 2.25 and np.isnan(r[4]) and r[5] == 0.0 and r[6] == np.inf
    ident = o.epilogue(P)
    assert same(ident, P)
    # alpha only, no other term: exact scaling
    assert same(o.epilogue(P[:, :4], alpha=-0.5)[0], -0.5 * P[0, :4])


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


def failing_pins(o) -> list[str]:
    """Names of the pins that the given oracle fails (or crashes in)."""
    bad = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except Exception:          # an assertion or a crash both count
            bad.append(pin.__name__)
    return bad

