"""gemm_bf16_streamk_noalloc (library-owned static scratch) against the
caller-workspace entry point gemm_bf16_streamk, two calls in a row.

Collected last on purpose: it must pass both alone and after every other
test has used the library (other workspaces, other schedules, watchdog
timeouts) in the same process."""
import pytest
import torch

import dense_gemm_blackwell_tcgen05_gb300 as g
import gemm_inputs as gi
import oracle
from tests import parity as P

pytestmark = pytest.mark.gpu


def _existing(A, B, variant, ws):
    M, K = A.shape
    N = B.shape[0]
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_bf16_streamk(variant, A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, K, K, N,
                             ws.data_ptr(), ws.numel(), s)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    assert g.gemm_last_status(s) == g.GEMM_OK
    return D.cpu()


def _noalloc(A, B, variant):
    M, K = A.shape
    N = B.shape[0]
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_bf16_streamk_noalloc(variant, A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K,
                                     K, K, N, s)
    assert rc == g.GEMM_OK, g.gemm_status_string(rc)
    sched = g.gemm_last_schedule()
    assert g.gemm_last_status(s) == g.GEMM_OK
    return D.cpu(), sched


@pytest.mark.parametrize("variant", [g.VARIANT_AUTO, g.VARIANT_1CTA, g.VARIANT_2CTA,
                                     g.VARIANT_1CTA | g.VARIANT_DIRECT_STORE])
@pytest.mark.parametrize("shape", [(300, 520, 1040), (129, 1031, 640), (10240, 1024, 320)])
def test_noalloc_matches_workspace_entry_point(variant, shape):
    M, N, K = shape
    A_cpu, B_cpu = gi.bf16_operands(M, N, K, seed=M + N + K)
    A, B = A_cpu.cuda(), B_cpu.cuda()
    ws = g.streamk_workspace(False, variant)
    # force the split so that the scratch is used whatever the cost model says
    old_mode = g.gemm_set_streamk_mode(g.STREAMK_ALWAYS)
    try:
        _compare(A, B, A_cpu, B_cpu, variant, ws, M, N)
    finally:
        g.gemm_set_streamk_mode(old_mode)


def _compare(A, B, A_cpu, B_cpu, variant, ws, M, N):
    want = _existing(A, B, variant, ws)
    # the bound's scale sum|a||b| from the oracle, on sampled entries
    rows, cols = P.sample_positions(M, N, 2000, seed=7)
    _, S = oracle.gemm_bf16_entries(gi.bf16_codes(A_cpu), gi.bf16_codes(B_cpu), rows, cols)
    for call in range(2):
        got, sched = _noalloc(A, B, variant)
        assert sched["sk_tiles"] > 0, "the stream-K split was expected for this shape"
        P.check_within_bound(P.bf16_to_f64(got)[rows, cols], P.bf16_to_f64(want)[rows, cols], S,
                             f"noalloc call {call}")
        assert not torch.isnan(got.float()).any()


def test_noalloc_rejects_what_it_cannot_run():
    A = torch.zeros(256, 256, dtype=torch.bfloat16, device="cuda")
    D = torch.empty(256, 256, dtype=torch.bfloat16, device="cuda")
    f = lambda v: g.gemm_bf16_streamk_noalloc(v, A.data_ptr(), A.data_ptr(), D.data_ptr(), 256,
                                              256, 256, 256, 256, 256, 0)
    assert f(g.VARIANT_SYNC) == g.GEMM_ERR_INVALID_ARG
    assert f(0x40) == g.GEMM_ERR_INVALID_ARG
    assert f(g.VARIANT_2CTA) == g.GEMM_OK
    torch.cuda.synchronize()
