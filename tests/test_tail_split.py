"""Tail split of the data-parallel schedule: the tiles of a last, partial
round are cut into two column halves (N = UMMA_N / 2 MMAs) when the halves fit
in one round.  And its variant for a cheap last column block (right-edge tiles
last): plain bf16 launches whose last column block holds at most half a tile
run those tiles as first halves, ordered after all others, with rounds dealt
in alternating directions.

The halves cover disjoint columns of D and run the same K loop, so each
element must come out bit for bit as it does from the whole tile: every GPU
case compares a launch with the split against one without it on the same
operands (normal inputs, so rounding is exercised), and against the oracle
(bitwise on small integers, within the bound otherwise).  The planner
arithmetic is checked on the CPU."""
import numpy as np
import pytest
import torch

import dense_gemm_blackwell_tcgen05_gb300 as g
import gemm_inputs as gi
import oracle
from tests import parity as P


# ------------------------------------------------------------ planner (CPU)

def expected_half_tiles(tiles, resident):
    r = tiles % resident if resident else 0
    return r if r != 0 and 2 * r <= resident else 0


def test_plan_cuts_a_short_last_round():
    prev = g.gemm_set_tail_split(1)
    try:
        for resident in (1, 2, 3, 76, 152):
            for tiles in range(0, 4 * resident + 3):
                assert g.gemm_tail_split_plan(tiles, resident) == \
                    expected_half_tiles(tiles, resident), (tiles, resident)
        # the headline shapes: 1024 pair tiles over 76 clusters leave 36
        assert g.gemm_tail_split_plan(1024, 76) == 36
        # 4096^3: 256 tiles, 28 in the last round
        assert g.gemm_tail_split_plan(256, 76) == 28
        # a last round more than half full is left whole
        assert g.gemm_tail_split_plan(76 + 39, 76) == 0
        # one partial round: every tile is cut when the halves fit
        assert g.gemm_tail_split_plan(30, 76) == 30
        assert g.gemm_tail_split_plan(40, 76) == 0
    finally:
        g.gemm_set_tail_split(prev)


def test_plan_switch_and_validation():
    prev = g.gemm_set_tail_split(0)
    try:
        assert g.gemm_tail_split_plan(80, 76) == 0
        assert g.gemm_set_tail_split(1) == 0
        assert g.gemm_tail_split_plan(80, 76) == 4
    finally:
        g.gemm_set_tail_split(prev)
    assert g.gemm_set_tail_split(2) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_set_tail_split(-1) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_tail_split_plan(-1, 76) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_tail_split_plan(10, -1) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_tail_split_plan(1 << 32, 76) == g.GEMM_ERR_INVALID_ARG


# ------------------------------------------------------------ GPU parity

def _launch(fn, split, edge=False):
    prev = g.gemm_set_tail_split(1 if split else 0)
    prev_e = g.gemm_set_edge_last(1 if edge else 0)
    try:
        D = fn()
        sched = g.gemm_last_schedule()
    finally:
        g.gemm_set_tail_split(prev)
        g.gemm_set_edge_last(prev_e)
    return D, sched


def _bf16(A, B, variant, ldd=None, epi=None):
    def fn():
        Ad, Bd = A.cuda(), B.cuda()
        M, K = A.shape
        N = B.shape[0]
        pitch = N if ldd is None else ldd
        D = torch.full((M, pitch), float("nan"), dtype=torch.bfloat16, device="cuda")
        s = torch.cuda.current_stream().cuda_stream
        if epi is None:
            rc = g.gemm_bf16_variant(variant, Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K,
                                     K, K, pitch, s)
        else:
            rc = g.gemm_bf16_fused(variant, Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K,
                                   K, K, pitch, epi, s)
        assert rc == g.GEMM_OK, g.gemm_status_string(rc)
        assert g.gemm_last_status(s) == g.GEMM_OK
        D = D.cpu()
        if pitch > N:
            assert torch.isnan(D[:, N:].float()).all(), "padding columns written"
        return D[:, :N]
    return fn


def _mx_tiled(A, SFA, B, SFB, variant):
    def fn():
        M, K = A.shape
        N = B.shape[0]
        SAt, SBt = gi.tile_scales(SFA, M, K).cuda(), gi.tile_scales(SFB, N, K).cuda()
        Ad, Bd = A.cuda(), B.cuda()
        D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        s = torch.cuda.current_stream().cuda_stream
        rc = g.gemm_mxfp8_tiled(variant, Ad.data_ptr(), Bd.data_ptr(), SAt.data_ptr(),
                                SBt.data_ptr(), D.data_ptr(), M, N, K, K, K, N, s)
        assert rc == g.GEMM_OK, g.gemm_status_string(rc)
        assert g.gemm_last_status(s) == g.GEMM_OK
        return D.cpu()
    return fn


def _assert_same(D1, D0, what):
    a, b = gi.bf16_codes(D1), gi.bf16_codes(D0)
    bad = np.argwhere(a != b)
    assert len(bad) == 0, f"{what}: split differs from whole tiles at {len(bad)} elements, " \
                          f"first {tuple(bad[0])}"


def _assert_oracle_bitwise(D, D_ref, what):
    want = oracle.f64_to_bf16_rne(D_ref)
    got = gi.bf16_codes(D)
    bad = np.argwhere(got != want)
    assert len(bad) == 0, f"{what}: {len(bad)} mismatches against the oracle, first {tuple(bad[0])}"


def _ints(M, N, K, seed):
    gen = torch.Generator().manual_seed(seed)
    A = torch.randint(-3, 4, (M, K), generator=gen).to(torch.bfloat16)
    B = torch.randint(-3, 4, (N, K), generator=gen).to(torch.bfloat16)
    return A, B


# (variant, M, N, K): shapes whose last round is cut.  Pair tiles are 256 x 256,
# one-CTA tiles 128 x 256; 76 pair clusters / 152 CTAs on a GB300.  Ragged N
# puts a column half past N (1100 = 4 x 256 + 76) or partly past it (2000).
BF16_CASES = [
    ("2cta", 2560, 2048, 192),          # 80 tiles: 4 cut
    ("2cta", 2600, 2000, 136),          # 88 tiles, ragged M and N
    ("2cta_direct", 2600, 2000, 136),
    ("2cta", 700, 1100, 200),           # one round, all 15 cut; second halves of the last column empty
    ("1cta", 2560, 2048, 128),          # 160 tiles: 8 cut
    ("1cta_direct", 2690, 2000, 72),    # 168 tiles, odd M
    ("auto", 128, 1100, 64),            # M = 128: one CTA, one round
]
VARIANT = {"2cta": g.VARIANT_2CTA, "2cta_direct": g.VARIANT_2CTA | g.VARIANT_DIRECT_STORE,
           "1cta": g.VARIANT_1CTA, "1cta_direct": g.VARIANT_1CTA | g.VARIANT_DIRECT_STORE,
           "auto": g.VARIANT_AUTO}


@pytest.mark.gpu
@pytest.mark.parametrize("case", BF16_CASES, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}x{c[3]}")
def test_bf16_split_matches_whole_tiles_and_oracle(case):
    v, M, N, K = case
    # normal inputs: the split must reproduce the whole-tile rounding exactly
    A, B = gi.bf16_operands(M, N, K, seed=M + N + K)
    D1, s1 = _launch(_bf16(A, B, VARIANT[v]), split=True)
    D0, s0 = _launch(_bf16(A, B, VARIANT[v]), split=False)
    assert s1["half_tiles"] > 0 and s0["half_tiles"] == 0, (s1, s0)
    assert s1["clusters"] >= s0["clusters"]
    _assert_same(D1, D0, f"bf16 {case}")
    # sampled against the oracle within the bound
    rows, cols = P.sample_positions(M, N, 1500, seed=K, tile_n=128)
    Dr, S = oracle.gemm_bf16_entries(gi.bf16_codes(A), gi.bf16_codes(B), rows, cols)
    P.check_within_bound(D1.float().numpy()[rows, cols], Dr, S, f"bf16 split {case}")
    # small integers: bitwise against the oracle everywhere
    Ai, Bi = _ints(M, N, min(K, 96), seed=K + 1)
    Di, si = _launch(_bf16(Ai, Bi, VARIANT[v]), split=True)
    assert si["half_tiles"] > 0
    D_ref, _ = oracle.gemm_bf16(gi.bf16_codes(Ai), gi.bf16_codes(Bi))
    _assert_oracle_bitwise(Di, D_ref, f"bf16 split ints {case}")


@pytest.mark.gpu
def test_bf16_split_odd_pitch_leaves_padding():
    A, B = gi.bf16_operands(2600, 2000, 136, seed=11)
    D1, s1 = _launch(_bf16(A, B, g.VARIANT_AUTO, ldd=2003), split=True)
    D0, _ = _launch(_bf16(A, B, g.VARIANT_AUTO, ldd=2003), split=False)
    assert s1["half_tiles"] > 0
    _assert_same(D1, D0, "odd pitch")


@pytest.mark.gpu
def test_fused_epilogue_columns_follow_the_halves():
    """Bias and C are indexed by the output column, which a second half
    offsets by UMMA_N / 2."""
    M, N, K = 2600, 2000, 136
    A, B = _ints(M, N, K, seed=5)
    gen = torch.Generator().manual_seed(6)
    bias = torch.randint(-8, 9, (N,), generator=gen).to(torch.float32)
    C = torch.randint(-8, 9, (M, N), generator=gen).to(torch.bfloat16)
    bd, Cd = bias.cuda(), C.cuda()
    epi = g.make_epilogue(2.0, -1.0, Cd, bd, "relu", torch.bfloat16)
    D1, s1 = _launch(_bf16(A, B, g.VARIANT_2CTA, epi=epi), split=True)
    D0, _ = _launch(_bf16(A, B, g.VARIANT_2CTA, epi=epi), split=False)
    assert s1["half_tiles"] > 0
    _assert_same(D1, D0, "fused")
    P_ref, _ = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B))
    Cf = C.float().double().numpy()
    want = np.maximum(2.0 * P_ref - Cf + bias.double().numpy()[None, :], 0.0)
    _assert_oracle_bitwise(D1, want, "fused split")


@pytest.mark.gpu
def test_fused_fp32_output_over_the_halves():
    """fp32 output (the masked-store kernel, per-thread C loads) with column
    halves: C, bias and the store all follow the half's column offset."""
    M, N, K = 2600, 2000, 72
    A, B = _ints(M, N, K, seed=15)
    gen = torch.Generator().manual_seed(16)
    bias = torch.randint(-8, 9, (N,), generator=gen).to(torch.float32)
    C = torch.randint(-8, 9, (M, N), generator=gen).to(torch.float32)
    bd, Cd = bias.cuda(), C.cuda()
    epi = g.make_epilogue(0.5, 2.0, Cd, bd, "relu", torch.float32)

    def fn():
        Ad, Bd = A.cuda(), B.cuda()
        D = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        s = torch.cuda.current_stream().cuda_stream
        rc = g.gemm_bf16_fused(g.VARIANT_2CTA, Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K,
                               K, K, N, epi, s)
        assert rc == g.GEMM_OK, g.gemm_status_string(rc)
        assert g.gemm_last_status(s) == g.GEMM_OK
        return D.cpu()
    D1, s1 = _launch(fn, split=True)
    assert s1["half_tiles"] > 0
    P_ref, _ = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B))
    want = np.maximum(0.5 * P_ref + 2.0 * C.double().numpy() + bias.double().numpy()[None, :], 0.0)
    got = D1.double().numpy()
    bad = np.argwhere(got != want)
    assert len(bad) == 0, f"{len(bad)} mismatches, first at {tuple(bad[0])}"


MX_CASES = [("auto", 2600, 2000, 256), ("auto", 700, 1100, 384), ("1cta", 2560, 2048, 128)]
MX_VARIANT = {"auto": g.VARIANT_AUTO, "1cta": g.VARIANT_1CTA}


@pytest.mark.gpu
@pytest.mark.parametrize("case", MX_CASES, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}x{c[3]}")
def test_mxfp8_tiled_split_matches_whole_tiles_and_oracle(case):
    v, M, N, K = case
    A, SFA, B, SFB = gi.mxfp8_operands(M, N, K, seed=M + 3 * N + K)
    D1, s1 = _launch(_mx_tiled(A, SFA, B, SFB, MX_VARIANT[v]), split=True)
    D0, s0 = _launch(_mx_tiled(A, SFA, B, SFB, MX_VARIANT[v]), split=False)
    assert s1["half_tiles"] > 0 and s0["half_tiles"] == 0, (s1, s0)
    _assert_same(D1, D0, f"mxfp8 {case}")
    rows, cols = P.sample_positions(M, N, 1500, seed=K, tile_n=128)
    Dr, S = oracle.gemm_mxfp8_entries(A.numpy(), B.numpy(), SFA.numpy(), SFB.numpy(), rows, cols)
    P.check_within_bound(D1.float().numpy()[rows, cols], Dr, S, f"mxfp8 split {case}")


# ------------------------------------------------------------ right-edge tiles last

def test_edge_last_switch_validation():
    prev = g.gemm_set_edge_last(0)
    try:
        assert g.gemm_set_edge_last(1) == 0
        assert g.gemm_set_edge_last(1) == 1
    finally:
        g.gemm_set_edge_last(prev)
    assert g.gemm_set_edge_last(2) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_set_edge_last(-1) == g.GEMM_ERR_INVALID_ARG


# (variant, M, N, K, ldd): plain bf16 launches whose last column block holds
# 1 <= N mod 256 <= 128 columns, over one or several rounds; the first is the
# ragged bench workload (4099 x 2053 x 1040, 153 pair tiles, 17 of them edge
# tiles).
EDGE_CASES = [
    ("2cta", 4099, 2053, 1040, 2053),
    ("2cta", 5000, 1100, 136, 1100),
    ("2cta_direct", 3000, 2053, 72, 2053),
    ("1cta", 2560, 1100, 128, 1104),
    ("1cta_direct", 5000, 1100, 72, 1103),
    ("auto", 128, 1100, 64, 1100),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", EDGE_CASES, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}x{c[3]}-ld{c[4]}")
def test_edge_last_matches_whole_tiles_and_oracle(case):
    v, M, N, K, ldd = case
    A, B = gi.bf16_operands(M, N, K, seed=M + 2 * N + K)
    D1, s1 = _launch(_bf16(A, B, VARIANT[v], ldd=ldd), split=True, edge=True)
    D0, s0 = _launch(_bf16(A, B, VARIANT[v], ldd=ldd), split=False, edge=False)
    assert s1["edge_last"] == 1 and s1["half_tiles"] == 0, s1
    assert s0["edge_last"] == 0 and s0["half_tiles"] == 0, s0
    assert s1["dp_tiles"] == s0["dp_tiles"]
    _assert_same(D1, D0, f"edge-last {case}")
    rows, cols = P.sample_positions(M, N, 1500, seed=K, tile_n=128)
    cols[:64] = np.arange(N - 64, N)   # every column of the edge block
    Dr, S = oracle.gemm_bf16_entries(gi.bf16_codes(A), gi.bf16_codes(B), rows, cols)
    P.check_within_bound(D1.float().numpy()[rows, cols], Dr, S, f"edge-last {case}")
    Ai, Bi = _ints(M, N, min(K, 96), seed=K + 3)
    Di, si = _launch(_bf16(Ai, Bi, VARIANT[v], ldd=ldd), split=True, edge=True)
    assert si["edge_last"] == 1
    D_ref, _ = oracle.gemm_bf16(gi.bf16_codes(Ai), gi.bf16_codes(Bi))
    _assert_oracle_bitwise(Di, D_ref, f"edge-last ints {case}")


@pytest.mark.gpu
def test_edge_last_only_for_plain_launches_with_a_cheap_edge():
    # more than half a tile of live columns in the last block: the tail split
    A, B = _ints(2600, 2000, 64, seed=21)
    _, s = _launch(_bf16(A, B, g.VARIANT_2CTA), split=True, edge=True)
    assert s["edge_last"] == 0 and s["half_tiles"] > 0, s
    # N a multiple of the tile width: nothing to move
    A, B = _ints(2600, 2048, 64, seed=22)
    _, s = _launch(_bf16(A, B, g.VARIANT_2CTA), split=True, edge=True)
    assert s["edge_last"] == 0, s
    # a fused epilogue runs the general build: no edge ordering
    A, B = _ints(2600, 1100, 64, seed=23)
    bias = torch.zeros(1100, dtype=torch.float32, device="cuda")
    epi = g.make_epilogue(1.0, 0.0, None, bias, "none", torch.bfloat16)
    Df, s = _launch(_bf16(A, B, g.VARIANT_2CTA, epi=epi), split=True, edge=True)
    assert s["edge_last"] == 0, s
    D_ref, _ = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B))
    _assert_oracle_bitwise(Df, D_ref, "fused, edge ordering off")
    # the MXFP8 kernels never take it
    Am, SFA, Bm, SFB = gi.mxfp8_operands(700, 1100, 256, seed=24)
    _, s = _launch(_mx_tiled(Am, SFA, Bm, SFB, g.VARIANT_AUTO), split=True, edge=True)
    assert s["edge_last"] == 0, s
