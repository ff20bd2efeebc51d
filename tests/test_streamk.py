"""Stream-K schedule (gemm_bf16_streamk / gemm_mxfp8_streamk) on the GPU,
element by element against the oracle.

The schedule only changes which CTA adds which K-range of a tile, so the
results obey the same rules as the data-parallel path: bitwise where every
partial sum is exact in fp32 (small integers; the order of the fp32 additions
then does not matter), within |D - D_ref| <= 2^-7 |D_ref| + 1e-3 sum|a b|
otherwise.  Every case asserts from gemm_last_schedule() that the regime it is
named for (fewer tiles than CTAs, several full waves plus a partial one, a
K-split so fine that a tile has many contributors) was the one launched."""
import numpy as np
import pytest
import torch

import dense_gemm_blackwell_tcgen05_gb300 as g
import gemm_inputs as gi
import oracle
from tests import parity as P
from tests.test_gemm_mxfp8 import int_operands as mx_int_operands

pytestmark = pytest.mark.gpu

BF16_VARIANTS = {
    "1cta": g.VARIANT_1CTA,
    "2cta": g.VARIANT_2CTA,
    "1cta_direct": g.VARIANT_1CTA | g.VARIANT_DIRECT_STORE,
    "2cta_direct": g.VARIANT_2CTA | g.VARIANT_DIRECT_STORE,
}
MX_VARIANTS = {
    "1cta": g.VARIANT_1CTA,
    "1cta_direct": g.VARIANT_1CTA | g.VARIANT_DIRECT_STORE,
    "2cta": g.VARIANT_2CTA,
}

_WS = {}


@pytest.fixture(autouse=True)
def _always_split():
    """Parity cases force the split (the cost model would keep small cases
    data-parallel); the mode is restored after each test."""
    old = g.gemm_set_streamk_mode(g.STREAMK_ALWAYS)
    yield
    g.gemm_set_streamk_mode(old)


def workspace(mx, variant):
    key = (bool(mx), variant & 0xFF)
    if key not in _WS:
        _WS[key] = g.streamk_workspace(mx, variant)
    return _WS[key]


def flags_are_zero(ws, mx, variant, sched):
    """The flag words (32 bytes per launched CTA at the start of the
    workspace) are back at zero.  Only a split launch uses the workspace."""
    if sched["sk_tiles"] == 0:
        return True
    ctas = sched["clusters"] * sched["ctas_per_cluster"]
    return bool(torch.all(ws[:ctas * 32] == 0).item())


def expected_split(sched, M, N, tile_m, tile_n, kt, unit):
    """Tiles the launcher must split when forced: those of the partial last
    wave plus one full wave, or all tiles when there are fewer tiles than
    resident clusters (then at most one cluster per K-unit is launched)."""
    tiles = -(-M // tile_m) * -(-N // tile_n)
    G = sched["clusters"]
    units = -(-kt // unit)
    assert sched["dp_tiles"] + sched["sk_tiles"] == tiles
    if units < 2 or sched["sk_tiles"] == 0:
        return 0
    if sched["dp_tiles"] == 0:
        assert G <= tiles * units
        return tiles
    return tiles % G + G


def run_bf16(A_cpu, B_cpu, variant, ldd=None, calls=1):
    A = A_cpu.cuda()
    B = B_cpu.cuda()
    M, K = A.shape
    N = B.shape[0]
    ldd = N if ldd is None else ldd
    ws = workspace(False, variant)
    out = []
    for _ in range(calls):
        D = torch.full((M, ldd), float("nan"), dtype=torch.bfloat16, device="cuda")
        s = torch.cuda.current_stream()
        rc = g.gemm_bf16_streamk(variant, A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, K, K,
                                 ldd, ws.data_ptr(), ws.numel(), s.cuda_stream)
        assert rc == g.GEMM_OK, g.gemm_status_string(rc)
        sched = g.gemm_last_schedule()
        st = g.gemm_last_status(s.cuda_stream)
        assert st == g.GEMM_OK, g.gemm_status_string(st)
        assert flags_are_zero(ws, False, variant, sched)
        if ldd > N:
            assert torch.isnan(D[:, N:].float()).all(), "wrote past N"
        out.append(D[:, :N].cpu())
    return out, sched


def run_mx(A, SFA, B, SFB, variant, calls=1):
    M, K = A.shape
    N = B.shape[0]
    ws = workspace(True, variant)
    dA, dB, dSFA, dSFB = (t.cuda() for t in (A, B, SFA, SFB))
    out = []
    for _ in range(calls):
        D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        s = torch.cuda.current_stream()
        rc = g.gemm_mxfp8_streamk(variant, dA.data_ptr(), dB.data_ptr(), dSFA.data_ptr(),
                                  dSFB.data_ptr(), D.data_ptr(), M, N, K, A.stride(0),
                                  B.stride(0), SFA.stride(0), SFB.stride(0), N, ws.data_ptr(),
                                  ws.numel(), s.cuda_stream)
        assert rc == g.GEMM_OK, g.gemm_status_string(rc)
        sched = g.gemm_last_schedule()
        st = g.gemm_last_status(s.cuda_stream)
        assert st == g.GEMM_OK, g.gemm_status_string(st)
        assert flags_are_zero(ws, True, variant, sched)
        out.append(D.cpu())
    return out, sched


def int_bf16(M, N, K, seed, lo=-3, hi=4):
    gen = torch.Generator().manual_seed(seed)
    A = torch.randint(lo, hi, (M, K), generator=gen).to(torch.bfloat16)
    B = torch.randint(lo, hi, (N, K), generator=gen).to(torch.bfloat16)
    return A, B


def assert_bitwise(D, D_ref, what):
    want = oracle.f64_to_bf16_rne(D_ref)
    got = gi.bf16_codes(D)
    bad = np.argwhere(got != want)
    assert len(bad) == 0, f"{what}: {len(bad)} mismatches, first at {tuple(bad[0])}"


def plan(mx, variant):
    p = g.gemm_kernel_plan(bool(mx), variant)
    bk = 128 if mx else 64
    return p["tile_m"], p["tile_n"], bk


# ------------------------------------------------------ bf16, full oracle

# (M, N, K): fewer tiles than CTAs with many K-ranges per tile; a K of two
# K-tiles (two units per tile); ragged K with an 8-element tail tile
BF16_SMALL = [(300, 520, 1040), (300, 520, 128), (257, 300, 1096), (129, 1031, 640)]


@pytest.mark.parametrize("v", list(BF16_VARIANTS))
@pytest.mark.parametrize("shape", BF16_SMALL)
def test_bf16_small_integers_bitwise(v, shape):
    M, N, K = shape
    variant = BF16_VARIANTS[v]
    A, B = int_bf16(M, N, K, seed=M * 7 + K)
    (D1, D2), sched = run_bf16(A, B, variant, calls=2)
    tm, tn, bk = plan(False, variant)
    assert sched["sk_tiles"] == expected_split(sched, M, N, tm, tn, -(-K // bk), 1) > 0
    D_ref, _ = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B))
    assert_bitwise(D1, D_ref, f"{v} {shape}")
    assert torch.equal(D1, D2), "second call on the same workspace differs"


@pytest.mark.parametrize("v", list(BF16_VARIANTS))
@pytest.mark.parametrize("shape", [(300, 520, 1040), (129, 1031, 640)])
def test_bf16_random_within_bound(v, shape):
    M, N, K = shape
    A, B = gi.bf16_operands(M, N, K, seed=K + 11)
    (D,), _ = run_bf16(A, B, BF16_VARIANTS[v])
    D_ref, S = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B))
    P.check_within_bound(P.bf16_to_f64(D), D_ref, S, f"streamk {v} {shape}")


@pytest.mark.parametrize("v", ["1cta", "2cta"])
def test_bf16_ragged_n_pitch_untouched(v):
    M, N, K = 300, 300, 1040
    A, B = int_bf16(M, N, K, seed=5)
    (D,), sched = run_bf16(A, B, BF16_VARIANTS[v], ldd=320)
    assert sched["sk_tiles"] > 0
    D_ref, _ = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B))
    assert_bitwise(D, D_ref, v)


# ------------------------------------- bf16, several full waves + a partial one

@pytest.mark.parametrize("v", ["1cta", "2cta", "2cta_direct"])
def test_bf16_waves_plus_partial(v):
    # 80 x 4 one-CTA tiles or 40 x 4 pair tiles: two full waves and a partial
    # one on any device with 100 < SMs < 160
    M, N, K = 10240, 1024, 320
    variant = BF16_VARIANTS[v]
    A, B = int_bf16(M, N, K, seed=99)
    (D,), sched = run_bf16(A, B, variant)
    tm, tn, bk = plan(False, variant)
    want = expected_split(sched, M, N, tm, tn, K // bk, 1)
    assert sched["sk_tiles"] == want
    if want == 0:
        pytest.skip(f"{sched['clusters']} clusters divide the tile count")
    assert sched["dp_tiles"] > 0
    # every row band of every tile row is checked against the oracle on
    # sampled columns; whole bands for the first and last tile rows
    rows, cols = P.sample_positions(M, N, 6000, seed=3)
    D_ref, _ = oracle.gemm_bf16_entries(gi.bf16_codes(A), gi.bf16_codes(B), rows, cols)
    want_codes = oracle.f64_to_bf16_rne(D_ref)
    got = gi.bf16_codes(D)[rows, cols]
    assert np.array_equal(got, want_codes)
    for r0 in (0, M - tm):
        D_ref, _ = oracle.gemm_bf16(gi.bf16_codes(A[r0:r0 + tm]), gi.bf16_codes(B))
        assert_bitwise(D[r0:r0 + tm], D_ref, f"{v} rows {r0}+")


def test_bf16_no_split_when_waves_are_full_or_k_is_one_tile():
    # K of one K-tile: nothing to split, the launch is data-parallel
    A, B = int_bf16(300, 520, 64, seed=1)
    (D,), sched = run_bf16(A, B, g.VARIANT_1CTA)
    assert sched["sk_tiles"] == 0
    D_ref, _ = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B))
    assert_bitwise(D, D_ref, "k=64")


def test_bf16_workload_ragged_k1040_sampled():
    w = gi.WORKLOADS["ragged_k1040"]
    A, B = gi.workload_operands("ragged_k1040")
    (D,), sched = run_bf16(A, B, g.VARIANT_2CTA)
    rows, cols = P.sample_positions(w.M, w.N, 3000, seed=w.seed)
    D_ref, S = oracle.gemm_bf16_entries(gi.bf16_codes(A), gi.bf16_codes(B), rows, cols)
    P.check_within_bound(P.bf16_to_f64(D)[rows, cols], D_ref, S, "ragged_k1040 streamk")


# ------------------------------------------------------------------ MXFP8

MX_SMALL = [(300, 520, 2080), (129, 300, 1040), (256, 448, 4096)]


@pytest.mark.parametrize("v", list(MX_VARIANTS))
@pytest.mark.parametrize("shape", MX_SMALL)
def test_mxfp8_exact_integers(v, shape):
    M, N, K = shape
    variant = MX_VARIANTS[v]
    A, SFA, B, SFB = mx_int_operands(M, N, K, seed=K + M)
    (D1, D2), sched = run_mx(A, SFA, B, SFB, variant, calls=2)
    tm, tn, bk = plan(True, variant)
    assert sched["sk_unit"] == 4
    assert sched["sk_tiles"] == expected_split(sched, M, N, tm, tn, -(-K // bk), 4) > 0
    D_ref, _ = oracle.gemm_mxfp8(A.numpy(), B.numpy(), SFA.numpy(), SFB.numpy(), K)
    assert_bitwise(D1, D_ref, f"mxfp8 {v} {shape}")
    assert torch.equal(D1, D2)


@pytest.mark.parametrize("v", list(MX_VARIANTS))
def test_mxfp8_quantised_normal(v):
    M, N, K = 300, 520, 2080
    A, SFA, B, SFB = gi.mxfp8_operands(M, N, K, seed=17)
    (D,), _ = run_mx(A, SFA, B, SFB, MX_VARIANTS[v])
    D_ref, S = oracle.gemm_mxfp8(A.numpy(), B.numpy(), SFA.numpy(), SFB.numpy(), K)
    P.check_within_bound(P.bf16_to_f64(D), D_ref, S, f"mxfp8 streamk {v}")


@pytest.mark.parametrize("v", ["1cta", "2cta"])
def test_mxfp8_waves_plus_partial(v):
    M, N, K = 10240, 1024, 1040
    variant = MX_VARIANTS[v]
    A, SFA, B, SFB = mx_int_operands(M, N, K, seed=8)
    (D,), sched = run_mx(A, SFA, B, SFB, variant)
    tm, tn, bk = plan(True, variant)
    want = expected_split(sched, M, N, tm, tn, -(-K // bk), 4)
    assert sched["sk_tiles"] == want
    if want == 0:
        pytest.skip(f"{sched['clusters']} clusters divide the tile count")
    rows, cols = P.sample_positions(M, N, 6000, seed=4)
    D_ref, _ = oracle.gemm_mxfp8_entries(A.numpy(), B.numpy(), SFA.numpy(), SFB.numpy(), rows,
                                         cols, K)
    assert np.array_equal(gi.bf16_codes(D)[rows, cols], oracle.f64_to_bf16_rne(D_ref))


# -------------------------------------------------- the automatic choice

def test_auto_mode_splits_a_long_k_problem_with_few_tiles():
    g.gemm_set_streamk_mode(g.STREAMK_AUTO)
    M, N, K = 1024, 1024, 16384
    A, B = int_bf16(M, N, K, seed=12, lo=-1, hi=2)
    for v in ("1cta", "2cta"):
        (D,), sched = run_bf16(A, B, BF16_VARIANTS[v])
        assert sched["sk_tiles"] > 0 and sched["dp_tiles"] == 0
        rows, cols = P.sample_positions(M, N, 3000, seed=5)
        D_ref, _ = oracle.gemm_bf16_entries(gi.bf16_codes(A), gi.bf16_codes(B), rows, cols)
        assert np.array_equal(gi.bf16_codes(D)[rows, cols], oracle.f64_to_bf16_rne(D_ref))


def test_auto_mode_keeps_short_k_data_parallel():
    g.gemm_set_streamk_mode(g.STREAMK_AUTO)
    A, B = int_bf16(300, 520, 1040, seed=3)
    (D,), sched = run_bf16(A, B, g.VARIANT_2CTA)
    assert sched["sk_tiles"] == 0
    D_ref, _ = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B))
    assert_bitwise(D, D_ref, "auto short k")


def test_never_mode_is_data_parallel():
    g.gemm_set_streamk_mode(g.STREAMK_NEVER)
    A, B = int_bf16(1024, 1024, 4096, seed=4, lo=-1, hi=2)
    (_,), sched = run_bf16(A, B, g.VARIANT_1CTA)
    # 32 tiles: one partial round, cut into 64 column halves by the tail split
    assert sched["sk_tiles"] == 0 and sched["dp_tiles"] == 32
    assert sched["clusters"] == 32 + sched["half_tiles"]
    assert sched["half_tiles"] == g.gemm_tail_split_plan(
        32, torch.cuda.get_device_properties(0).multi_processor_count)


# ------------------------------------------------------------ argument errors

def test_workspace_validation():
    A = torch.zeros(256, 1024, dtype=torch.bfloat16, device="cuda")
    D = torch.zeros(256, 256, dtype=torch.bfloat16, device="cuda")
    ws = workspace(False, g.VARIANT_2CTA)
    f = lambda wp, wb, v=g.VARIANT_2CTA: g.gemm_bf16_streamk(
        v, A.data_ptr(), A.data_ptr(), D.data_ptr(), 256, 256, 1024, 1024, 1024, 256, wp, wb, 0)
    assert f(0, ws.numel()) == g.GEMM_ERR_INVALID_ARG                    # NULL
    assert f(ws.data_ptr(), 1024) == g.GEMM_ERR_INVALID_ARG              # too small
    assert f(ws.data_ptr() + 4, ws.numel() - 4) == g.GEMM_ERR_INVALID_ARG  # misaligned
    assert f(ws.data_ptr(), ws.numel(), g.VARIANT_SYNC) == g.GEMM_ERR_INVALID_ARG
    host = torch.zeros(ws.numel(), dtype=torch.uint8)
    assert f(host.data_ptr(), host.numel()) == g.GEMM_ERR_INVALID_ARG    # host memory
    assert f(ws.data_ptr(), ws.numel()) == g.GEMM_OK
    torch.cuda.synchronize()
    assert g.gemm_streamk_workspace_bytes(False, g.VARIANT_SYNC) == g.GEMM_ERR_INVALID_ARG


def test_matmul_wrappers_take_a_workspace():
    A, B = int_bf16(300, 520, 1040, seed=2)
    ws = workspace(False, g.VARIANT_AUTO)
    D = g.matmul_bf16(A.cuda(), B.cuda(), workspace=ws)
    assert g.gemm_last_schedule()["sk_tiles"] > 0
    D_ref, _ = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B))
    assert_bitwise(D.cpu(), D_ref, "matmul_bf16")


# ------------------------------------------------------------- watchdog

@pytest.mark.parametrize("v", ["1cta", "2cta"])
@pytest.mark.parametrize("stall", [0, 3])
def test_streamk_stall_times_out_then_recovers(v, stall):
    """A stage that never fills (the watchdog test hook) in a split launch:
    the kernel gives up on its bounded waits, drains its own copies, returns
    GEMM_ERR_TIMEOUT; after the workspace is zeroed again the next call is
    exact."""
    variant = BF16_VARIANTS[v]
    M, N, K = 1024, 1024, 4096
    A, B = int_bf16(M, N, K, seed=77, lo=-1, hi=2)
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    ws = workspace(False, variant)
    s = torch.cuda.current_stream().cuda_stream
    call = lambda: g.gemm_bf16_streamk(variant, Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N,
                                       K, K, K, N, ws.data_ptr(), ws.numel(), s)
    old_ms = g.gemm_set_watchdog_ms(100)
    try:
        assert g.gemm_debug_stall_next_launch(stall) == g.GEMM_OK
        assert call() == g.GEMM_OK
        assert g.gemm_last_schedule()["sk_tiles"] > 0
        assert g.gemm_last_status(s) == g.GEMM_ERR_TIMEOUT
    finally:
        g.gemm_set_watchdog_ms(old_ms)
    ws.zero_()
    assert call() == g.GEMM_OK
    assert g.gemm_last_status(s) == g.GEMM_OK
    D_ref, _ = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B))
    assert_bitwise(D.cpu(), D_ref, f"after recovery {v}")


# ---------------------------------------- the stream-K workloads, full size

@pytest.mark.parametrize("name", ["streamk_1024x16384", "streamk_mxfp8_1024x32768"])
def test_streamk_workloads_full_size(name):
    """The bench's configuration (automatic split decision, automatic
    variant) on sampled outputs; the split must have been taken."""
    g.gemm_set_streamk_mode(g.STREAMK_AUTO)
    w = gi.WORKLOADS[name]
    ops = gi.workload_operands(name)
    rows, cols = P.sample_positions(w.M, w.N, 3000, seed=w.seed)
    if w.kind == "bf16":
        A, B = ops
        D = g.matmul_bf16(A.cuda(), B.cuda(), workspace=workspace(False, g.VARIANT_AUTO))
        D_ref, S = oracle.gemm_bf16_entries(gi.bf16_codes(A), gi.bf16_codes(B), rows, cols)
    else:
        A, SFA, B, SFB = ops
        D = g.matmul_mxfp8(A.cuda(), SFA.cuda(), B.cuda(), SFB.cuda(),
                           workspace=workspace(True, g.VARIANT_AUTO))
        D_ref, S = oracle.gemm_mxfp8_entries(A.numpy(), B.numpy(), SFA.numpy(), SFB.numpy(), rows,
                                             cols, w.K)
    assert g.gemm_last_schedule()["sk_tiles"] > 0
    assert g.gemm_last_status(0) == g.GEMM_OK
    P.check_within_bound(P.bf16_to_f64(D.cpu())[rows, cols], D_ref, S, name)
