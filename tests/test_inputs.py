"""The seeded input generators: shapes, determinism and the MXFP8 encoder."""
import numpy as np
import torch

import gemm_inputs as gi
import oracle


def test_workload_table():
    w = gi.WORKLOADS
    assert (w["single_tile"].M, w["single_tile"].N, w["single_tile"].K) == (128, 128, 64)
    assert (w["ragged_k1040"].M, w["ragged_k1040"].N, w["ragged_k1040"].K) == (4099, 2053, 1040)
    assert w["ragged_k8"].K == 8 and w["ragged_k8"].seed == w["ragged_k1040"].seed
    assert w["square_8192"].scale == 0.5 and w["mxfp8_8192"].kind == "mxfp8"


def test_deterministic():
    a1, b1 = gi.bf16_operands(33, 17, 40, seed=5)
    a2, b2 = gi.bf16_operands(33, 17, 40, seed=5)
    assert torch.equal(a1, a2) and torch.equal(b1, b2)
    assert a1.dtype == torch.bfloat16 and a1.shape == (33, 40) and b1.shape == (17, 40)


def test_uniform_range():
    a, b = gi.bf16_operands(128, 128, 64, seed=0, dist="uniform")
    assert float(a.float().min()) >= -1.0 and float(a.float().max()) <= 1.0


def _nearest_e4m3(v: np.ndarray) -> np.ndarray:
    """Brute force: for each value the E4M3 code(s) at minimum distance,
    ties resolved to the even mantissa."""
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    vals = oracle.e4m3_to_f64(codes)
    ok = ~np.isnan(vals)
    codes, vals = codes[ok], vals[ok]
    out = np.empty(v.shape, np.uint8)
    for t, x in enumerate(v):
        d = np.abs(vals - x)
        best = np.flatnonzero(d == d.min())
        best = [c for c in codes[best] if not (vals[codes == c][0] == 0 and x != 0
                                               and np.signbit(x) != bool(c & 0x80))]
        if len(best) > 1:
            best = [c for c in best if (c & 1) == 0] or best
        out[t] = best[0]
    return out


def test_mxfp8_encoder():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(6, 100, generator=g)
    x[1, :32] = 0.0                      # an all-zero block
    x[2] *= 1e6                          # large values
    x[3] *= 1e-6                         # small values
    x[4, 5] = 448.0 * 2 ** 3             # amax exactly on a power-of-two boundary
    q, sf = gi.mxfp8_quantize(x)
    assert q.shape == (6, 100) and sf.shape == (6, gi.sf_pitch(100)) and sf.shape[1] % 16 == 0
    assert torch.all(sf[:, 4:] == 0)
    xd = x.double().numpy()
    e = sf.numpy()[:, :4].astype(np.int64) - 127
    for r in range(6):
        for b in range(4):
            blk = xd[r, 32 * b:32 * b + 32]
            amax = np.abs(blk).max()
            if amax == 0:
                assert e[r, b] == -127
            else:
                assert amax <= 448.0 * 2.0 ** e[r, b] and amax > 448.0 * 2.0 ** (e[r, b] - 1)
            want = _nearest_e4m3(blk * 2.0 ** -e[r, b])
            assert np.array_equal(q.numpy()[r, 32 * b:32 * b + len(blk)], want), (r, b)
    assert e[4, 0] == 3
