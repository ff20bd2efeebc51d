"""Seeded synthetic inputs for the GEMM workloads.

This module only draws and encodes operands; it holds none of the GEMM's
arithmetic.  Both the CUDA path (through tests and ``bench.py``) and the CPU
oracle receive the operands it produces, so parity never depends on random
number stability across versions: every run regenerates the same tensors for
both sides.

Recipe (one torch CPU generator per workload, A drawn before B, row-major):

===================== ===================================== ==================
workload               shape / distribution                  seed
===================== ===================================== ==================
single_tile            M=N=128, K=64, uniform[-1,1) -> bf16   0
square_4096            M=N=K=4096, N(0,1) -> bf16              1
ragged_k1040           M=4099, N=2053, K=1040, N(0,1) -> bf16  2
ragged_k8              M=4099, N=2053, K=8,    N(0,1) -> bf16  2
square_8192            M=N=K=8192, 0.5*N(0,1) -> bf16          3
mxfp8_8192             M=N=K=8192, N(0,1) -> MXFP8             4
                       (scales passed to the GEMM in the tiled layout)
mxfp8_8192_rows        the same operands, scales passed row-major  4
quantize_8192          [8192, 8192] float32 N(0,1) (the A       4
                       operand above, before encoding)
fused_gelu_8192        square_8192's A, B; C [M,N] N(0,1) ->   3 (+100 for C,
                       bf16, bias [N] N(0,1) -> bf16             bias)
fused_f32_8192         square_8192's A, B; bias [N] N(0,1)     3 (+100)
                       float32
streamk_1024x16384     M=N=1024, K=16384, N(0,1) -> bf16       5
streamk_mxfp8_1024x32768  M=N=1024, K=32768, N(0,1) -> MXFP8   6
===================== ===================================== ==================

Epilogue inputs come from a second generator seeded with seed + 100: C
first (when the workload has one), then the bias vector.

bf16 rounding is torch's float32 -> bfloat16 cast (round-to-nearest-even).
MXFP8 encoding of a float32 row: for each block of 32 consecutive k (the
last block may be partial) take amax = max |x|, the scale exponent e is the
smallest integer with amax <= 448 * 2^e (clamped to [-127, 127]; amax = 0
gives e = -127), the scale byte is e + 127 (UE8M0) and each element is
x * 2^-e rounded to E4M3 (round-to-nearest-even; |x * 2^-e| <= 448 by
construction, so no saturation is needed).  Scale rows are padded with zero
bytes to a multiple of 16, the row pitch the library requires.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    seed: int
    dist: str            # "uniform" | "normal"
    scale: float = 1.0
    kind: str = "bf16"   # "bf16" | "mxfp8" | "quant" (MXFP8 encoding of float32 rows [M, K])
    # fused epilogue: "" (plain bf16 store), or "alpha,beta,act,out,bias" with
    # act none|relu|gelu, out bf16|f32, bias none|bf16|f32 (beta != 0 adds C)
    epilogue: str = ""
    schedule: str = "dp"  # "dp" | "streamk" (caller workspace, automatic split)
    variant: int = 0      # kernel variant the bench runs it with (0 = automatic)
    # MXFP8: the layout the scale matrices are handed to the GEMM in -- "rows"
    # (row-major, gemm_mxfp8) or "tiled" (tile_scales of the same bytes,
    # gemm_mxfp8_tiled).  The operands and their values are the same.
    sf_layout: str = "rows"

    @property
    def flops(self) -> int:
        return 0 if self.kind == "quant" else 2 * self.M * self.N * self.K


WORKLOADS = {
    w.name: w for w in [
        Workload("single_tile", 128, 128, 64, 0, "uniform"),
        Workload("square_4096", 4096, 4096, 4096, 1, "normal"),
        Workload("ragged_k1040", 4099, 2053, 1040, 2, "normal"),
        Workload("ragged_k8", 4099, 2053, 8, 2, "normal"),
        Workload("square_8192", 8192, 8192, 8192, 3, "normal", 0.5),
        Workload("mxfp8_8192", 8192, 8192, 8192, 4, "normal", 1.0, "mxfp8", sf_layout="tiled"),
        Workload("mxfp8_8192_rows", 8192, 8192, 8192, 4, "normal", 1.0, "mxfp8"),
        Workload("quantize_8192", 8192, 0, 8192, 4, "normal", 1.0, "quant"),
        Workload("fused_gelu_8192", 8192, 8192, 8192, 3, "normal", 0.5, "bf16",
                 epilogue="1.0,1.0,gelu,bf16,bf16"),
        Workload("fused_f32_8192", 8192, 8192, 8192, 3, "normal", 0.5, "bf16",
                 epilogue="0.5,0.0,relu,f32,f32"),
        Workload("streamk_1024x16384", 1024, 1024, 16384, 5, "normal", 1.0, "bf16",
                 schedule="streamk"),
        Workload("streamk_mxfp8_1024x32768", 1024, 1024, 32768, 6, "normal", 1.0, "mxfp8",
                 schedule="streamk"),
    ]
}


def epilogue_spec(w: Workload) -> dict | None:
    """The parsed epilogue string of a workload (None: plain store)."""
    if not w.epilogue:
        return None
    alpha, beta, act, out, bias = w.epilogue.split(",")
    return {"alpha": float(alpha), "beta": float(beta), "act": act, "out": out, "bias": bias}


def epilogue_operands(w: Workload):
    """(C or None, bias or None) of a fused-epilogue workload: C [M, N] in the
    output dtype, bias [N] in its dtype, drawn N(0,1) from seed + 100."""
    spec = epilogue_spec(w)
    if spec is None:
        return None, None
    g = torch.Generator().manual_seed(w.seed + 100)
    out_dt = torch.float32 if spec["out"] == "f32" else torch.bfloat16
    C = torch.randn(w.M, w.N, generator=g).to(out_dt) if spec["beta"] != 0.0 else None
    bias = None
    if spec["bias"] != "none":
        bias = torch.randn(w.N, generator=g).to(torch.float32 if spec["bias"] == "f32" else torch.bfloat16)
    return C, bias


def _draw(g: torch.Generator, rows: int, cols: int, dist: str, scale: float) -> torch.Tensor:
    if dist == "uniform":
        x = torch.rand(rows, cols, generator=g, dtype=torch.float32) * 2 - 1
    elif dist == "normal":
        x = torch.randn(rows, cols, generator=g, dtype=torch.float32)
    else:
        raise ValueError(dist)
    if scale != 1.0:
        x = x * scale
    return x


def float_operands(M: int, N: int, K: int, seed: int, dist: str = "normal",
                   scale: float = 1.0):
    """float32 A [M,K] and B [N,K], A drawn first."""
    g = torch.Generator().manual_seed(seed)
    A = _draw(g, M, K, dist, scale)
    B = _draw(g, N, K, dist, scale)
    return A, B


def bf16_operands(M: int, N: int, K: int, seed: int, dist: str = "normal",
                  scale: float = 1.0):
    """bf16 A [M,K] and B [N,K] (CPU tensors, contiguous)."""
    A, B = float_operands(M, N, K, seed, dist, scale)
    return A.to(torch.bfloat16), B.to(torch.bfloat16)


def sf_pitch(K: int) -> int:
    """Row pitch, in bytes, of a scale-factor matrix for reduction length K."""
    nblk = (K + 31) // 32
    return max(16, (nblk + 15) // 16 * 16)


def mxfp8_quantize(x: torch.Tensor):
    """Encode float32 rows [R, K] as (E4M3 codes uint8 [R, K], UE8M0 scale
    bytes uint8 [R, sf_pitch(K)]), one scale per 32 consecutive k."""
    if x.dtype != torch.float32 or x.dim() != 2:
        raise TypeError("expected a 2-D float32 tensor")
    R, K = x.shape
    nblk = (K + 31) // 32
    pad = nblk * 32 - K
    xp = torch.nn.functional.pad(x, (0, pad)) if pad else x
    blocks = xp.reshape(R, nblk, 32).double()
    amax = blocks.abs().amax(dim=2)                                  # [R, nblk]
    # smallest integer e with amax <= 448 * 2^e: a float guess, then exact fix-ups
    safe = torch.where(amax > 0, amax, torch.ones_like(amax))
    e = torch.ceil(torch.log2(safe / 448.0))
    four48 = torch.full_like(e, 448.0)
    for _ in range(2):
        e = torch.where(amax > torch.ldexp(four48, e), e + 1, e)
        e = torch.where(amax <= torch.ldexp(four48, e - 1), e - 1, e)
    e = torch.where(amax > 0, e, torch.full_like(e, -127.0)).clamp(-127, 127)
    scaled = torch.ldexp(blocks, -e.unsqueeze(2))                    # exact
    q = scaled.float().to(torch.float8_e4m3fn).view(torch.uint8)
    q = q.reshape(R, nblk * 32)[:, :K].contiguous()
    sf = torch.zeros(R, sf_pitch(K), dtype=torch.uint8)
    sf[:, :nblk] = (e + 127).to(torch.uint8)
    return q, sf


def mxfp8_operands(M: int, N: int, K: int, seed: int, dist: str = "normal",
                   scale: float = 1.0):
    """(A codes [M,K], SFA [M,pitch], B codes [N,K], SFB [N,pitch]), uint8."""
    A, B = float_operands(M, N, K, seed, dist, scale)
    qa, sfa = mxfp8_quantize(A)
    qb, sfb = mxfp8_quantize(B)
    return qa, sfa, qb, sfb


def tile_scales(sf: torch.Tensor, rows: int, K: int) -> torch.Tensor:
    """Row-major UE8M0 scales [rows, >= ceil(K/32)] rearranged into the tiled
    layout gemm_mxfp8_tiled takes (a pure permutation plus zero padding): 512-byte
    chunks of 128 rows x 4 blocks, chunk (row block rb, block group g) at
    512 * (rb * ceil(nblk/4) + g); inside it row 128 rb + 32 c + l, block
    4 g + j at byte 16 l + 4 c + j.  Returns a flat uint8 tensor on sf's device."""
    nb = (K + 31) // 32
    R, C = (rows + 127) // 128 * 128, (nb + 3) // 4 * 4
    p = torch.zeros(R, C, dtype=torch.uint8, device=sf.device)
    p[:rows, :nb] = sf[:rows, :nb]
    # [rb, c, l, g, j] -> [rb, g, l, c, j]
    t = p.view(R // 128, 4, 32, C // 4, 4).permute(0, 3, 2, 1, 4)
    return t.contiguous().view(-1)


def workload_operands(name: str):
    """Operands of a named workload: (A, B) for bf16, (A, SFA, B, SFB) for MXFP8,
    (X,) float32 for the quantiser (the MXFP8 workload's A operand)."""
    w = WORKLOADS[name]
    if w.kind == "quant":
        return (float_operands(w.M, 1, w.K, w.seed, w.dist, w.scale)[0],)
    if w.kind == "bf16":
        return bf16_operands(w.M, w.N, w.K, w.seed, w.dist, w.scale)
    return mxfp8_operands(w.M, w.N, w.K, w.seed, w.dist, w.scale)


def bf16_codes(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a CPU bf16 tensor (a view, no arithmetic)."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected bfloat16")
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def u8_codes(t: torch.Tensor) -> np.ndarray:
    if t.dtype != torch.uint8:
        raise TypeError("expected uint8")
    return t.contiguous().numpy()
