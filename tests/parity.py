"""Helpers shared by the GPU parity tests: the acceptance bound, sampled
output positions and device/host marshalling.  No GEMM arithmetic here: the
expected values always come from the oracle."""
from __future__ import annotations

import numpy as np
import torch

import gemm_inputs as gi

# Per-element acceptance for a bf16 output (fp32 accumulation):
#   |D - D_ref| <= 2^-7 |D_ref| + 1e-3 * sum_k |a_ik b_jk|
REL = 2.0 ** -7
ABS_SCALE = 1e-3


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    """Decode a bf16 tensor (any device) to float64 on the host."""
    return t.detach().to("cpu").float().double().numpy()


def check_within_bound(D_gpu: np.ndarray, D_ref: np.ndarray, S: np.ndarray, what: str = "") -> float:
    """Assert the bound on every finite element and identical non-finite
    classes elsewhere; return max(|err| / bound) over finite elements."""
    D_gpu = np.asarray(D_gpu, np.float64)
    D_ref = np.asarray(D_ref, np.float64)
    S = np.asarray(S, np.float64)
    assert D_gpu.shape == D_ref.shape == S.shape, what
    fin = np.isfinite(D_ref)
    # non-finite where the exact result is non-finite (NaN stays NaN; +-Inf may
    # also surface as NaN when the fp32 path overflows on both signs)
    nf = ~fin
    if nf.any():
        assert np.all(~np.isfinite(D_gpu[nf])), f"{what}: finite output where the reference is not"
        assert np.all(np.isnan(D_gpu[np.isnan(D_ref)])), f"{what}: NaN lost"
    bound = REL * np.abs(D_ref[fin]) + ABS_SCALE * S[fin]
    err = np.abs(D_gpu[fin] - D_ref[fin])
    assert np.all(np.isfinite(D_gpu[fin])), f"{what}: non-finite output where the reference is finite"
    bad = err > bound
    if bad.any():
        idx = np.flatnonzero(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside the bound; first "
                             f"err={err[idx]}, bound={bound[idx]}, ref={D_ref[fin][idx]}")
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / bound, 0.0)
    return float(ratio.max()) if ratio.size else 0.0


def sample_positions(M: int, N: int, n_random: int, seed: int, tile_m: int = 128,
                     tile_n: int = 256):
    """Output positions to check at sizes too large for the full oracle:
    random positions plus every tile-boundary row/column pair and the corners."""
    rng = np.random.default_rng(seed)
    rows = list(rng.integers(0, M, n_random))
    cols = list(rng.integers(0, N, n_random))
    edge_r = sorted({0, M - 1, *[r for t in range(tile_m, M, tile_m) for r in (t - 1, t)]})
    edge_c = sorted({0, N - 1, *[c for t in range(tile_n, N, tile_n) for c in (t - 1, t)]})
    for r in edge_r:
        rows.append(r)
        cols.append(int(rng.integers(0, N)))
    for c in edge_c:
        rows.append(int(rng.integers(0, M)))
        cols.append(c)
    for r in (0, M - 1):
        for c in (0, N - 1):
            rows.append(r)
            cols.append(c)
    return np.array(rows, np.int64), np.array(cols, np.int64)


def bf16_from_ints(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def e4m3_from_ints(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)


def codes16(t: torch.Tensor) -> np.ndarray:
    return gi.bf16_codes(t.cpu())
