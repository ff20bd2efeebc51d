"""CPU reference (oracle) for the tcgen05 GEMM -- test infrastructure only.

The oracle is a plain fp64 C implementation of D = A * B^T (``oracle.c``)
plus this ctypes loader.  It exists to check the CUDA path: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  It shares no code with the CUDA library and never imports it.

What it computes and which passage each function follows is documented in
``oracle.c``.  Every function here is pinned by ``tests/test_oracle.py``
against values that do not come from the oracle itself (library conversions
of every bit pattern, exact rational brute force, closed forms such as the
all-ones and identity products, and exact small-integer products).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_default = None

_i64 = ctypes.c_int64
_p = ctypes.c_void_p


def build(force: bool = False, src: str = SRC, out: str = LIB_PATH) -> str:
    """Compile the oracle source with gcc (-O2, OpenMP, no fast-math) if stale."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    stale = not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src)
    if force or stale:
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-fno-fast-math", "-ffp-contract=off", src, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def _bind(L: ctypes.CDLL) -> ctypes.CDLL:
    L.oracle_num_threads.restype = ctypes.c_int
    for name in ("oracle_bf16_to_f64_array", "oracle_e4m3_to_f64_array",
                 "oracle_ue8m0_to_f64_array", "oracle_f64_to_bf16_rne_array"):
        getattr(L, name).argtypes = [_p, _i64, _p]
        getattr(L, name).restype = None
    L.oracle_gemm_bf16.argtypes = [_p, _p, _i64, _i64, _i64, _i64, _i64, _p, _p]
    L.oracle_gemm_bf16_entries.argtypes = [_p, _p, _i64, _i64, _i64, _p, _p, _i64, _p, _p]
    L.oracle_gemm_mxfp8.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64,
                                    _i64, _i64, _p, _p]
    L.oracle_gemm_mxfp8_entries.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _i64,
                                            _i64, _p, _p, _i64, _p, _p]
    for name in ("oracle_gemm_bf16", "oracle_gemm_bf16_entries",
                 "oracle_gemm_mxfp8", "oracle_gemm_mxfp8_entries"):
        getattr(L, name).restype = None
    L.oracle_epilogue.argtypes = [_p, _i64, _i64, ctypes.c_double, ctypes.c_double, _p, _i64, _p,
                                  ctypes.c_int, _p]
    L.oracle_epilogue.restype = None
    L.oracle_mxfp8_quantize.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _p, _i64]
    L.oracle_mxfp8_quantize.restype = None
    L.oracle_f64_to_e4m3_rne.argtypes = [ctypes.c_double]
    L.oracle_f64_to_e4m3_rne.restype = ctypes.c_uint8
    return L


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _as_c(a, dtype) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return np.ascontiguousarray(a)


def _check_2d(X, rows, K, name):
    if X.ndim != 2 or X.shape[0] < rows or X.shape[1] < K:
        raise ValueError(f"{name} has shape {X.shape}, needs at least [{rows}, {K}]")


def _check_sf(SF, rows, K, name):
    nblk = (K + 31) // 32
    if SF.ndim != 2 or SF.shape[0] < rows or SF.shape[1] < nblk:
        raise ValueError(f"{name} has shape {SF.shape}, needs at least [{rows}, {nblk}]")


def _entries(rows, cols, nA, nB):
    r = _as_c(np.asarray(rows, np.int64), np.int64)
    c = _as_c(np.asarray(cols, np.int64), np.int64)
    if r.shape != c.shape:
        raise ValueError("rows and cols differ in shape")
    if r.size and (r.min() < 0 or r.max() >= nA or c.min() < 0 or c.max() >= nB):
        raise IndexError("entry index out of range")
    return r, c


class Oracle:
    """The oracle's functions bound to one compiled library."""

    def __init__(self, path: str):
        self.path = path
        self.L = _bind(ctypes.CDLL(path))

    def num_threads(self) -> int:
        """OpenMP threads the oracle's GEMM loops use."""
        return int(self.L.oracle_num_threads())

    # -------------------------------------------------------------- decoders
    def _map(self, fn, codes, in_dtype, out_dtype):
        c = _as_c(codes, in_dtype)
        out = np.empty(c.shape, out_dtype)
        getattr(self.L, fn)(_ptr(c), c.size, _ptr(out))
        return out

    def bf16_to_f64(self, codes) -> np.ndarray:
        return self._map("oracle_bf16_to_f64_array", codes, np.uint16, np.float64)

    def e4m3_to_f64(self, codes) -> np.ndarray:
        return self._map("oracle_e4m3_to_f64_array", codes, np.uint8, np.float64)

    def ue8m0_to_f64(self, codes) -> np.ndarray:
        return self._map("oracle_ue8m0_to_f64_array", codes, np.uint8, np.float64)

    def f64_to_bf16_rne(self, values) -> np.ndarray:
        """Round fp64 values to bf16 (round-to-nearest-even); uint16 codes."""
        return self._map("oracle_f64_to_bf16_rne_array",
                         np.asarray(values, np.float64), np.float64, np.uint16)

    def f64_to_e4m3_rne(self, values) -> np.ndarray:
        """Round fp64 values (|v| <= 448) to E4M3 codes, ties to even."""
        v = np.asarray(values, np.float64).ravel()
        return np.array([self.L.oracle_f64_to_e4m3_rne(float(x)) for x in v],
                        np.uint8).reshape(np.shape(values))

    def epilogue(self, P, alpha=1.0, beta=0.0, C=None, bias=None, act=0):
        """act(alpha P + beta C + bias[j]) elementwise in fp64 (the fused
        epilogue); P, C [M, N] and bias [N] as fp64 values."""
        f64 = lambda x: np.ascontiguousarray(np.asarray(x, dtype=np.float64))
        P = f64(P)
        M, N = P.shape
        out = np.empty((M, N), dtype=np.float64)
        Cp, ldc = None, 0
        if C is not None:
            C = f64(C)
            if C.shape[0] != M or C.shape[1] < N:
                raise ValueError("C must be [M, >=N]")
            Cp, ldc = _ptr(C), C.shape[1]
        bp = None
        if bias is not None:
            bias = f64(bias).reshape(-1)
            if bias.shape[0] < N:
                raise ValueError("bias must hold N values")
            bp = _ptr(bias)
        if act not in (0, 1, 2):
            raise ValueError("act must be 0, 1 or 2")
        self.L.oracle_epilogue(_ptr(P), M, N, float(alpha), float(beta), Cp, ldc, bp, int(act),
                               _ptr(out))
        return out

    def mxfp8_quantize(self, X, K: int | None = None):
        """MXFP8-encode float32 rows X [rows, ldx] (first K columns): returns
        (Q uint8 [rows, K], SF uint8 [rows, ceil(K/32)])."""
        X = _as_c(X, np.float32)
        rows = X.shape[0]
        K = X.shape[1] if K is None else int(K)
        _check_2d(X, rows, K, "X")
        nblk = (K + 31) // 32
        Q = np.empty((rows, K), np.uint8)
        SF = np.empty((rows, nblk), np.uint8)
        self.L.oracle_mxfp8_quantize(_ptr(X), rows, K, X.shape[1], _ptr(Q), K, _ptr(SF), nblk)
        return Q, SF

    # ----------------------------------------------------------------- GEMMs
    def gemm_bf16(self, A, B, K: int | None = None):
        """D = A * B^T over bf16 codes.

        A: uint16 [M, lda] (row-major bf16 bit patterns), B: uint16 [N, ldb].
        Only the first K columns are used (default: all of A's columns).
        Returns (D, S), float64 [M, N]: the fp64 sum and the sum of |terms|.
        """
        A = _as_c(A, np.uint16)
        B = _as_c(B, np.uint16)
        M, N = A.shape[0], B.shape[0]
        K = A.shape[1] if K is None else int(K)
        _check_2d(A, M, K, "A")
        _check_2d(B, N, K, "B")
        D = np.empty((M, N), np.float64)
        S = np.empty((M, N), np.float64)
        self.L.oracle_gemm_bf16(_ptr(A), _ptr(B), M, N, K, A.shape[1], B.shape[1],
                                _ptr(D), _ptr(S))
        return D, S

    def gemm_bf16_entries(self, A, B, rows, cols, K: int | None = None):
        """Entries D[rows[t], cols[t]] of A * B^T (see ``gemm_bf16``)."""
        A = _as_c(A, np.uint16)
        B = _as_c(B, np.uint16)
        K = A.shape[1] if K is None else int(K)
        _check_2d(A, A.shape[0], K, "A")
        _check_2d(B, B.shape[0], K, "B")
        r, c = _entries(rows, cols, A.shape[0], B.shape[0])
        D = np.empty(r.shape, np.float64)
        S = np.empty(r.shape, np.float64)
        self.L.oracle_gemm_bf16_entries(_ptr(A), _ptr(B), K, A.shape[1], B.shape[1],
                                        _ptr(r), _ptr(c), r.size, _ptr(D), _ptr(S))
        return D, S

    def gemm_mxfp8(self, A, B, SFA, SFB, K: int | None = None):
        """D = A * B^T for E4M3 codes A [M, lda], B [N, ldb] (uint8) with UE8M0
        scales SFA [M, ldsfa], SFB [N, ldsfb] (uint8), one per 32 consecutive
        k.  Returns (D, S), float64 [M, N]."""
        A = _as_c(A, np.uint8)
        B = _as_c(B, np.uint8)
        SFA = _as_c(SFA, np.uint8)
        SFB = _as_c(SFB, np.uint8)
        M, N = A.shape[0], B.shape[0]
        K = A.shape[1] if K is None else int(K)
        _check_2d(A, M, K, "A")
        _check_2d(B, N, K, "B")
        _check_sf(SFA, M, K, "SFA")
        _check_sf(SFB, N, K, "SFB")
        D = np.empty((M, N), np.float64)
        S = np.empty((M, N), np.float64)
        self.L.oracle_gemm_mxfp8(_ptr(A), _ptr(B), _ptr(SFA), _ptr(SFB), M, N, K,
                                 A.shape[1], B.shape[1], SFA.shape[1], SFB.shape[1],
                                 _ptr(D), _ptr(S))
        return D, S

    def gemm_mxfp8_entries(self, A, B, SFA, SFB, rows, cols, K: int | None = None):
        """Entries D[rows[t], cols[t]] of the block-scaled product."""
        A = _as_c(A, np.uint8)
        B = _as_c(B, np.uint8)
        SFA = _as_c(SFA, np.uint8)
        SFB = _as_c(SFB, np.uint8)
        K = A.shape[1] if K is None else int(K)
        _check_2d(A, A.shape[0], K, "A")
        _check_2d(B, B.shape[0], K, "B")
        _check_sf(SFA, A.shape[0], K, "SFA")
        _check_sf(SFB, B.shape[0], K, "SFB")
        r, c = _entries(rows, cols, A.shape[0], B.shape[0])
        D = np.empty(r.shape, np.float64)
        S = np.empty(r.shape, np.float64)
        self.L.oracle_gemm_mxfp8_entries(_ptr(A), _ptr(B), _ptr(SFA), _ptr(SFB), K,
                                         A.shape[1], B.shape[1], SFA.shape[1], SFB.shape[1],
                                         _ptr(r), _ptr(c), r.size, _ptr(D), _ptr(S))
        return D, S


def default() -> Oracle:
    """The oracle built from ``oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def num_threads() -> int:
    return default().num_threads()


def bf16_to_f64(codes):
    return default().bf16_to_f64(codes)


def e4m3_to_f64(codes):
    return default().e4m3_to_f64(codes)


def ue8m0_to_f64(codes):
    return default().ue8m0_to_f64(codes)


def f64_to_bf16_rne(values):
    return default().f64_to_bf16_rne(values)


def f64_to_e4m3_rne(values):
    return default().f64_to_e4m3_rne(values)


def mxfp8_quantize(X, K=None):
    return default().mxfp8_quantize(X, K)


def epilogue(P, alpha=1.0, beta=0.0, C=None, bias=None, act=0):
    return default().epilogue(P, alpha, beta, C, bias, act)


def gemm_bf16(A, B, K=None):
    return default().gemm_bf16(A, B, K)


def gemm_bf16_entries(A, B, rows, cols, K=None):
    return default().gemm_bf16_entries(A, B, rows, cols, K)


def gemm_mxfp8(A, B, SFA, SFB, K=None):
    return default().gemm_mxfp8(A, B, SFA, SFB, K)


def gemm_mxfp8_entries(A, B, SFA, SFB, rows, cols, K=None):
    return default().gemm_mxfp8_entries(A, B, SFA, SFB, rows, cols, K)
