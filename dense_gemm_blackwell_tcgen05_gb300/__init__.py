"""Python binding of the GB300 tcgen05 GEMM library (``include/gemm_gb300.h``).

Argument marshalling only: every step of the GEMM runs in the CUDA library's
own kernels.  The entry points keep the C names and arguments (raw device
pointers as integers, sizes, leading dimensions in elements, a CUDA stream
handle); ``matmul_bf16`` / ``matmul_mxfp8`` are conveniences that take torch
CUDA tensors, call the same entry points on the current stream and raise on
a non-zero status.  There is no CPU or library fallback: when the CUDA
library cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import threading

from . import _build

__all__ = [
    "GEMM_OK", "GEMM_ERR_INVALID_ARG", "GEMM_ERR_ALIGNMENT", "GEMM_ERR_UNSUPPORTED_DEVICE",
    "GEMM_ERR_LAUNCH", "GEMM_ERR_TIMEOUT", "GEMM_ERR_DEVICE_FAULT",
    "VARIANT_AUTO", "VARIANT_1CTA", "VARIANT_2CTA", "VARIANT_SYNC", "VARIANT_SMALLK",
    "VARIANT_SMALLK_TC",
    "VARIANT_DIRECT_STORE",
    "GemmError", "load", "library_path", "EXPORTED_SYMBOLS",
    "gemm_bf16", "gemm_bf16_variant", "gemm_mxfp8", "gemm_mxfp8_variant", "gemm_mxfp8_tiled",
    "matmul_mxfp8_tiled", "gemm_mxfp8_quantize_tiled", "quantize_mxfp8_tiled", "gemm_last_status", "gemm_last_status_word", "gemm_status_string", "gemm_set_watchdog_ms",
    "gemm_kernel_plan", "gemm_last_cuda_error", "gemm_debug_stall_next_launch",
    "gemm_mxfp8_quantize", "quantize_mxfp8", "gemm_bf16_streamk", "gemm_mxfp8_streamk",
    "gemm_streamk_workspace_bytes", "gemm_last_schedule", "streamk_workspace",
    "gemm_bf16_streamk_noalloc", "gemm_set_streamk_mode", "STREAMK_AUTO", "STREAMK_ALWAYS",
    "STREAMK_NEVER", "gemm_streamk_plan", "gemm_set_tail_split", "gemm_tail_split_plan",
    "gemm_set_edge_last", "gemm_bf16_fused", "gemm_mxfp8_fused", "GemmEpilogue",
    "make_epilogue", "matmul_fused", "DTYPE_BF16", "DTYPE_F32", "ACT_NONE", "ACT_RELU", "ACT_GELU", "matmul_bf16",
    "matmul_mxfp8",
]

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = -1
GEMM_ERR_ALIGNMENT = -2
GEMM_ERR_UNSUPPORTED_DEVICE = -3
GEMM_ERR_LAUNCH = -4
GEMM_ERR_TIMEOUT = -5
GEMM_ERR_DEVICE_FAULT = -6

VARIANT_AUTO = 0
VARIANT_1CTA = 1
VARIANT_2CTA = 2
VARIANT_SYNC = 3
VARIANT_SMALLK = 4
VARIANT_SMALLK_TC = 5
VARIANT_DIRECT_STORE = 0x100

# Every function include/gemm_gb300.h declares.
EXPORTED_SYMBOLS = (
    "gemm_bf16", "gemm_bf16_variant", "gemm_mxfp8", "gemm_mxfp8_variant", "gemm_last_status",
    "gemm_last_status_word", "gemm_status_string", "gemm_set_watchdog_ms", "gemm_kernel_plan",
    "gemm_last_cuda_error", "gemm_debug_stall_next_launch", "gemm_mxfp8_quantize",
    "gemm_bf16_streamk", "gemm_mxfp8_streamk", "gemm_streamk_workspace_bytes",
    "gemm_last_schedule", "gemm_bf16_streamk_noalloc", "gemm_set_streamk_mode",
    "gemm_streamk_plan", "gemm_bf16_fused", "gemm_mxfp8_fused", "gemm_mxfp8_tiled",
    "gemm_mxfp8_quantize_tiled", "gemm_set_tail_split", "gemm_tail_split_plan",
    "gemm_set_edge_last",
)

_lock = threading.Lock()
_lib = None
_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        if status == GEMM_ERR_LAUNCH:
            what = f"{what} (cuda error {gemm_last_cuda_error()})"
        super().__init__(f"{what}: {gemm_status_string(status)} ({status})" if what
                         else f"{gemm_status_string(status)} ({status})")


def library_path() -> str:
    return _build.LIB_PATH


DTYPE_BF16, DTYPE_F32 = 0, 1
ACT_NONE, ACT_RELU, ACT_GELU = 0, 1, 2


class GemmEpilogue(ctypes.Structure):
    """Mirror of gemm_epilogue_t: D = act(alpha acc + beta C + bias[col])."""
    _fields_ = [("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("C", ctypes.c_void_p),
                ("ldc", ctypes.c_int64), ("bias", ctypes.c_void_p), ("bias_dtype", ctypes.c_int32),
                ("activation", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


def load() -> ctypes.CDLL:
    """Load the CUDA library, building it in-tree first if it is missing or
    older than its sources.  Raises if it cannot be built or loaded."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = ctypes.CDLL(path)
            L.gemm_bf16.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _i64, _vp]
            L.gemm_bf16_variant.argtypes = [ctypes.c_int, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                                            _i64, _i64, _vp]
            L.gemm_mxfp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _i64,
                                     _i64, _i64, _vp]
            L.gemm_mxfp8_variant.argtypes = [ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _i64, _i64,
                                             _i64, _i64, _i64, _i64, _i64, _i64, _vp]
            L.gemm_mxfp8_tiled.argtypes = [ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64,
                                           _i64, _i64, _i64, _vp]
            for name in ("gemm_bf16", "gemm_bf16_variant", "gemm_mxfp8", "gemm_mxfp8_variant",
                         "gemm_mxfp8_tiled"):
                getattr(L, name).restype = ctypes.c_int
            L.gemm_bf16_streamk.argtypes = [ctypes.c_int, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                                            _i64, _i64, _vp, _i64, _vp]
            L.gemm_bf16_streamk.restype = ctypes.c_int
            L.gemm_mxfp8_streamk.argtypes = [ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _i64, _i64,
                                             _i64, _i64, _i64, _i64, _i64, _i64, _vp, _i64, _vp]
            L.gemm_mxfp8_streamk.restype = ctypes.c_int
            L.gemm_streamk_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
            L.gemm_streamk_workspace_bytes.restype = _i64
            L.gemm_bf16_streamk_noalloc.argtypes = [ctypes.c_int, _vp, _vp, _vp, _i64, _i64, _i64,
                                                    _i64, _i64, _i64, _vp]
            L.gemm_bf16_streamk_noalloc.restype = ctypes.c_int
            L.gemm_bf16_fused.argtypes = [ctypes.c_int, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                          _i64, ctypes.POINTER(GemmEpilogue), _vp]
            L.gemm_bf16_fused.restype = ctypes.c_int
            L.gemm_mxfp8_fused.argtypes = [ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64,
                                           _i64, _i64, _i64, _i64, _i64,
                                           ctypes.POINTER(GemmEpilogue), _vp]
            L.gemm_mxfp8_fused.restype = ctypes.c_int
            L.gemm_streamk_plan.argtypes = [_i64, _i64, _i64, _i64, ctypes.c_int,
                                            ctypes.POINTER(_i64)]
            L.gemm_streamk_plan.restype = ctypes.c_int
            L.gemm_set_streamk_mode.argtypes = [ctypes.c_int]
            L.gemm_set_streamk_mode.restype = ctypes.c_int
            L.gemm_last_schedule.argtypes = [ctypes.POINTER(_i64)]
            L.gemm_last_schedule.restype = ctypes.c_int
            L.gemm_set_tail_split.argtypes = [ctypes.c_int]
            L.gemm_set_tail_split.restype = ctypes.c_int
            L.gemm_set_edge_last.argtypes = [ctypes.c_int]
            L.gemm_set_edge_last.restype = ctypes.c_int
            L.gemm_tail_split_plan.argtypes = [_i64, _i64]
            L.gemm_tail_split_plan.restype = _i64
            L.gemm_mxfp8_quantize.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp]
            L.gemm_mxfp8_quantize.restype = ctypes.c_int
            L.gemm_mxfp8_quantize_tiled.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp]
            L.gemm_mxfp8_quantize_tiled.restype = ctypes.c_int
            L.gemm_last_status.argtypes = [_vp]
            L.gemm_last_status.restype = ctypes.c_int
            L.gemm_last_status_word.argtypes = [_vp]
            L.gemm_last_status_word.restype = ctypes.c_uint64
            L.gemm_status_string.argtypes = [ctypes.c_int]
            L.gemm_status_string.restype = ctypes.c_char_p
            L.gemm_debug_stall_next_launch.argtypes = [_i64]
            L.gemm_debug_stall_next_launch.restype = ctypes.c_int
            L.gemm_last_cuda_error.argtypes = []
            L.gemm_last_cuda_error.restype = ctypes.c_int
            L.gemm_set_watchdog_ms.argtypes = [_i64]
            L.gemm_set_watchdog_ms.restype = _i64
            P = ctypes.POINTER(ctypes.c_int32)
            L.gemm_kernel_plan.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P, P, P, P, P]
            L.gemm_kernel_plan.restype = ctypes.c_int
            _lib = L
    return _lib


# ------------------------------------------------------------- C entry points

def gemm_bf16(A: int, B: int, D: int, M: int, N: int, K: int, lda: int, ldb: int, ldd: int,
              stream: int = 0) -> int:
    return load().gemm_bf16(A, B, D, M, N, K, lda, ldb, ldd, stream)


def gemm_bf16_variant(variant: int, A: int, B: int, D: int, M: int, N: int, K: int, lda: int,
                      ldb: int, ldd: int, stream: int = 0) -> int:
    return load().gemm_bf16_variant(variant, A, B, D, M, N, K, lda, ldb, ldd, stream)


def gemm_mxfp8(A: int, B: int, SFA: int, SFB: int, D: int, M: int, N: int, K: int, lda: int,
               ldb: int, ldsfa: int, ldsfb: int, ldd: int, stream: int = 0) -> int:
    return load().gemm_mxfp8(A, B, SFA, SFB, D, M, N, K, lda, ldb, ldsfa, ldsfb, ldd, stream)


def gemm_mxfp8_variant(variant: int, A: int, B: int, SFA: int, SFB: int, D: int, M: int, N: int,
                       K: int, lda: int, ldb: int, ldsfa: int, ldsfb: int, ldd: int,
                       stream: int = 0) -> int:
    return load().gemm_mxfp8_variant(variant, A, B, SFA, SFB, D, M, N, K, lda, ldb, ldsfa, ldsfb,
                                     ldd, stream)


def gemm_mxfp8_tiled(variant: int, A: int, B: int, SFA: int, SFB: int, D: int, M: int, N: int,
                     K: int, lda: int, ldb: int, ldd: int, stream: int = 0) -> int:
    return load().gemm_mxfp8_tiled(variant, A, B, SFA, SFB, D, M, N, K, lda, ldb, ldd, stream)


def gemm_bf16_streamk(variant: int, A: int, B: int, D: int, M: int, N: int, K: int, lda: int,
                      ldb: int, ldd: int, workspace: int, workspace_bytes: int,
                      stream: int = 0) -> int:
    return load().gemm_bf16_streamk(variant, A, B, D, M, N, K, lda, ldb, ldd, workspace,
                                    workspace_bytes, stream)


def gemm_mxfp8_streamk(variant: int, A: int, B: int, SFA: int, SFB: int, D: int, M: int, N: int,
                       K: int, lda: int, ldb: int, ldsfa: int, ldsfb: int, ldd: int,
                       workspace: int, workspace_bytes: int, stream: int = 0) -> int:
    return load().gemm_mxfp8_streamk(variant, A, B, SFA, SFB, D, M, N, K, lda, ldb, ldsfa, ldsfb,
                                     ldd, workspace, workspace_bytes, stream)


def gemm_bf16_streamk_noalloc(variant: int, A: int, B: int, D: int, M: int, N: int, K: int,
                              lda: int, ldb: int, ldd: int, stream: int = 0) -> int:
    return load().gemm_bf16_streamk_noalloc(variant, A, B, D, M, N, K, lda, ldb, ldd, stream)


def gemm_streamk_workspace_bytes(mxfp8: bool, variant: int) -> int:
    return int(load().gemm_streamk_workspace_bytes(int(bool(mxfp8)), variant))


STREAMK_AUTO, STREAMK_ALWAYS, STREAMK_NEVER = 0, 1, 2


def gemm_set_streamk_mode(mode: int) -> int:
    return load().gemm_set_streamk_mode(mode)


def gemm_set_tail_split(enable: int) -> int:
    return load().gemm_set_tail_split(enable)


def gemm_set_edge_last(enable: int) -> int:
    return load().gemm_set_edge_last(enable)


def gemm_tail_split_plan(tiles: int, resident: int) -> int:
    return int(load().gemm_tail_split_plan(tiles, resident))


def gemm_bf16_fused(variant: int, A: int, B: int, D: int, M: int, N: int, K: int, lda: int,
                    ldb: int, ldd: int, epi: GemmEpilogue | None, stream: int = 0) -> int:
    return load().gemm_bf16_fused(variant, A, B, D, M, N, K, lda, ldb, ldd,
                                  None if epi is None else ctypes.byref(epi), stream)


def gemm_mxfp8_fused(variant: int, A: int, B: int, SFA: int, SFB: int, D: int, M: int, N: int,
                     K: int, lda: int, ldb: int, ldsfa: int, ldsfb: int, ldd: int,
                     epi: GemmEpilogue | None, stream: int = 0) -> int:
    return load().gemm_mxfp8_fused(variant, A, B, SFA, SFB, D, M, N, K, lda, ldb, ldsfa, ldsfb,
                                   ldd, None if epi is None else ctypes.byref(epi), stream)


_ACTS = {"none": ACT_NONE, "relu": ACT_RELU, "gelu": ACT_GELU}


def make_epilogue(alpha=1.0, beta=0.0, C=None, bias=None, activation="none",
                  out_dtype=None) -> GemmEpilogue:
    """A GemmEpilogue from torch tensors: C [M, >=N] of the output dtype,
    bias [N] bf16 or float32, activation "none" | "relu" | "gelu"."""
    import torch
    out_dtype = torch.bfloat16 if out_dtype is None else out_dtype
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out_dtype must be bfloat16 or float32")
    e = GemmEpilogue()
    e.alpha, e.beta = float(alpha), float(beta)
    e.out_dtype = DTYPE_F32 if out_dtype == torch.float32 else DTYPE_BF16
    e.activation = _ACTS[activation]
    if C is not None:
        _check_2d(C, "C")
        if C.dtype != out_dtype:
            raise TypeError("C must have the output dtype")
        e.C, e.ldc = C.data_ptr(), C.stride(0)
    if bias is not None:
        if bias.dim() != 1 or bias.stride(0) != 1 or bias.dtype not in (torch.bfloat16, torch.float32):
            raise TypeError("bias must be a contiguous 1-D bfloat16 or float32 tensor")
        e.bias = bias.data_ptr()
        e.bias_dtype = DTYPE_F32 if bias.dtype == torch.float32 else DTYPE_BF16
    return e


def matmul_fused(A, B, SFA=None, SFB=None, *, alpha=1.0, beta=0.0, C=None, bias=None,
                 activation="none", out_dtype=None, out=None, variant: int = VARIANT_AUTO,
                 stream=None):
    """D = act(alpha A @ B.T + beta C + bias): bf16 A [M,K], B [N,K], or
    MXFP8 codes with SFA/SFB as in matmul_mxfp8; D of out_dtype (bf16 or fp32)."""
    import torch
    _check_2d(A, "A")
    _check_2d(B, "B")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise ValueError("A and B disagree on K")
    out_dtype = torch.bfloat16 if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty(M, N, dtype=out_dtype, device=A.device)
    _check_2d(out, "out")
    if out.dtype != out_dtype:
        raise TypeError("out must have out_dtype")
    e = make_epilogue(alpha, beta, C, bias, activation, out_dtype)
    if SFA is None:
        if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
            raise TypeError("A and B must be bfloat16 (or pass SFA/SFB for MXFP8)")
        rc = gemm_bf16_fused(variant, A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K,
                             A.stride(0), B.stride(0), out.stride(0), e, _stream_handle(stream))
    else:
        rc = gemm_mxfp8_fused(variant, A.data_ptr(), B.data_ptr(), SFA.data_ptr(), SFB.data_ptr(),
                              out.data_ptr(), M, N, K, A.stride(0), B.stride(0), SFA.stride(0),
                              SFB.stride(0), out.stride(0), e, _stream_handle(stream))
    if rc != GEMM_OK:
        raise GemmError(rc, "matmul_fused")
    return out


def gemm_streamk_plan(tiles: int, resident: int, k_tiles: int, unit: int,
                      mode: int = STREAMK_AUTO) -> dict:
    """The stream-K schedule for a tile count (host only)."""
    out = (ctypes.c_int64 * 3)()
    rc = load().gemm_streamk_plan(tiles, resident, k_tiles, unit, mode, out)
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_streamk_plan")
    return {"dp_tiles": out[0], "sk_tiles": out[1], "clusters": out[2]}


def gemm_last_schedule() -> dict:
    """Schedule of this thread's last persistent-kernel launch."""
    out = (ctypes.c_int64 * 7)()
    rc = load().gemm_last_schedule(out)
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_last_schedule")
    return {"clusters": out[0], "ctas_per_cluster": out[1], "dp_tiles": out[2],
            "sk_tiles": out[3], "sk_unit": out[4], "half_tiles": out[5], "edge_last": out[6]}


def streamk_workspace(mxfp8: bool = False, variant: int = VARIANT_AUTO, device=None):
    """A zeroed device buffer sized for the stream-K entry points (one per
    stream: calls sharing a workspace must not overlap on the GPU)."""
    import torch
    n = gemm_streamk_workspace_bytes(mxfp8, variant)
    if n < 0:
        raise GemmError(n, "gemm_streamk_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def gemm_mxfp8_quantize(X: int, rows: int, K: int, ldx: int, Q: int, ldq: int, SF: int,
                        ldsf: int, stream: int = 0) -> int:
    return load().gemm_mxfp8_quantize(X, rows, K, ldx, Q, ldq, SF, ldsf, stream)


def gemm_mxfp8_quantize_tiled(X: int, rows: int, K: int, ldx: int, Q: int, ldq: int, SF: int,
                              stream: int = 0) -> int:
    return load().gemm_mxfp8_quantize_tiled(X, rows, K, ldx, Q, ldq, SF, stream)


def gemm_last_status(stream: int = 0) -> int:
    return load().gemm_last_status(stream)


def gemm_last_status_word(stream: int = 0) -> int:
    return int(load().gemm_last_status_word(stream))


def gemm_status_string(status: int) -> str:
    return load().gemm_status_string(status).decode()


def gemm_last_cuda_error() -> int:
    return int(load().gemm_last_cuda_error())


def gemm_debug_stall_next_launch(k_iteration: int) -> int:
    return int(load().gemm_debug_stall_next_launch(k_iteration))


def gemm_set_watchdog_ms(ms: int) -> int:
    return int(load().gemm_set_watchdog_ms(ms))


def gemm_kernel_plan(mxfp8, variant: int) -> dict:
    """mxfp8: False/0 bf16, True/1 MXFP8, 2 MXFP8 with tiled scales."""
    vals = [ctypes.c_int32() for _ in range(7)]
    rc = load().gemm_kernel_plan(int(mxfp8), variant, *[ctypes.byref(v) for v in vals])
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_kernel_plan")
    keys = ("stages", "smem_bytes", "tmem_cols", "threads", "cluster", "tile_m", "tile_n")
    return {k: v.value for k, v in zip(keys, vals)}


# ------------------------------------------------------- torch conveniences

def _stream_handle(stream) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _check_2d(t, name):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D tensor with unit column stride")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def matmul_bf16(A, B, out=None, variant: int = VARIANT_AUTO, stream=None, workspace=None):
    """D = A @ B.T for bf16 CUDA tensors A [M,K], B [N,K]; returns D [M,N] bf16.
    With `workspace` (from streamk_workspace) the stream-K schedule is used."""
    import torch
    _check_2d(A, "A")
    _check_2d(B, "B")
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise TypeError("A and B must be bfloat16")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise ValueError("A and B disagree on K")
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=A.device)
    _check_2d(out, "out")
    if workspace is None:
        rc = gemm_bf16_variant(variant, A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K,
                               A.stride(0), B.stride(0), out.stride(0), _stream_handle(stream))
    else:
        rc = gemm_bf16_streamk(variant, A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K,
                               A.stride(0), B.stride(0), out.stride(0), workspace.data_ptr(),
                               workspace.numel() * workspace.element_size(),
                               _stream_handle(stream))
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_bf16")
    return out


def matmul_mxfp8(A, SFA, B, SFB, out=None, variant: int = VARIANT_AUTO, stream=None,
                 workspace=None):
    """Block-scaled D = A @ B.T: A [M,K], B [N,K] E4M3 codes (uint8 or
    float8_e4m3fn), SFA [M,>=ceil(K/32)], SFB [N,>=ceil(K/32)] UE8M0 bytes.
    With `workspace` (from streamk_workspace) the stream-K schedule is used."""
    import torch
    for t, n in ((A, "A"), (B, "B"), (SFA, "SFA"), (SFB, "SFB")):
        _check_2d(t, n)
        if t.element_size() != 1:
            raise TypeError(f"{n} must hold one byte per element")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise ValueError("A and B disagree on K")
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=A.device)
    _check_2d(out, "out")
    if workspace is None:
        rc = gemm_mxfp8_variant(variant, A.data_ptr(), B.data_ptr(), SFA.data_ptr(),
                                SFB.data_ptr(), out.data_ptr(), M, N, K, A.stride(0), B.stride(0),
                                SFA.stride(0), SFB.stride(0), out.stride(0),
                                _stream_handle(stream))
    else:
        rc = gemm_mxfp8_streamk(variant, A.data_ptr(), B.data_ptr(), SFA.data_ptr(),
                                SFB.data_ptr(), out.data_ptr(), M, N, K, A.stride(0), B.stride(0),
                                SFA.stride(0), SFB.stride(0), out.stride(0), workspace.data_ptr(),
                                workspace.numel() * workspace.element_size(),
                                _stream_handle(stream))
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_mxfp8")
    return out


def quantize_mxfp8_tiled(X, stream=None):
    """MXFP8-encode a float32 CUDA tensor X [rows, K]: returns (Q uint8 [rows, K],
    SF uint8, flat, in the tiled layout of gemm_mxfp8_tiled)."""
    import torch
    _check_2d(X, "X")
    if X.dtype != torch.float32:
        raise TypeError("X must be float32")
    rows, K = X.shape
    n = (rows + 127) // 128 * (((K + 31) // 32 + 3) // 4) * 512
    Q = torch.empty(rows, K, dtype=torch.uint8, device=X.device)
    SF = torch.empty(n, dtype=torch.uint8, device=X.device)
    rc = gemm_mxfp8_quantize_tiled(X.data_ptr(), rows, K, X.stride(0), Q.data_ptr(), Q.stride(0),
                                   SF.data_ptr(), _stream_handle(stream))
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_mxfp8_quantize_tiled")
    return Q, SF


def matmul_mxfp8_tiled(A, SFA, B, SFB, out=None, variant: int = VARIANT_AUTO, stream=None):
    """Block-scaled D = A @ B.T with the scale matrices in the tiled layout of
    gemm_mxfp8_tiled (1-D byte tensors, e.g. from gemm_inputs.tile_scales)."""
    import torch
    for t, n in ((A, "A"), (B, "B")):
        _check_2d(t, n)
        if t.element_size() != 1:
            raise TypeError(f"{n} must hold one byte per element")
    for t, n in ((SFA, "SFA"), (SFB, "SFB")):
        if not t.is_cuda or t.element_size() != 1 or not t.is_contiguous():
            raise TypeError(f"{n} must be a contiguous CUDA byte tensor")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise ValueError("A and B disagree on K")
    kt = (K + 127) // 128
    for t, n, R in ((SFA, "SFA", M), (SFB, "SFB", N)):
        if t.numel() < (R + 127) // 128 * kt * 512:
            raise ValueError(f"{n} is smaller than the tiled layout of {R} rows")
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=A.device)
    _check_2d(out, "out")
    rc = gemm_mxfp8_tiled(variant, A.data_ptr(), B.data_ptr(), SFA.data_ptr(), SFB.data_ptr(),
                          out.data_ptr(), M, N, K, A.stride(0), B.stride(0), out.stride(0),
                          _stream_handle(stream))
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_mxfp8_tiled")
    return out


def quantize_mxfp8(X, stream=None):
    """MXFP8-encode a float32 CUDA tensor X [rows, K]: returns (Q uint8
    [rows, K], SF uint8 [rows, pitch]) with the scale pitch padded to a
    multiple of 16 bytes (the pitch gemm_mxfp8 requires), padding zeroed."""
    import torch
    _check_2d(X, "X")
    if X.dtype != torch.float32:
        raise TypeError("X must be float32")
    rows, K = X.shape
    pitch = max(16, ((K + 31) // 32 + 15) // 16 * 16)
    Q = torch.empty(rows, K, dtype=torch.uint8, device=X.device)
    SF = torch.zeros(rows, pitch, dtype=torch.uint8, device=X.device)
    rc = gemm_mxfp8_quantize(X.data_ptr(), rows, K, X.stride(0), Q.data_ptr(), Q.stride(0),
                             SF.data_ptr(), SF.stride(0), _stream_handle(stream))
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_mxfp8_quantize")
    return Q, SF
