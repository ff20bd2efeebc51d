"""gemm_bf16_streamk_noalloc (library-owned static scratch, for callers that
cannot allocate device memory where they multiply) against the
caller-workspace entry point gemm_bf16_streamk and against the oracle.

The owner of a split tile adds the later K-ranges' fp32 partials in K order,
so both entry points give the same bits on the same schedule: the whole of D
must be equal bit for bit, on two calls in a row, and within the bound of the
oracle's values on sampled entries.

Collected last on purpose: it must pass both alone and after every other
test has used the library (other workspaces, other schedules, watchdog
timeouts) in the same process."""
import os
import subprocess
import sys
import textwrap

import pytest
import torch

import dense_gemm_blackwell_tcgen05_gb300 as g
import gemm_inputs as gi
import oracle
from tests import parity as P

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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


def _same_bits(x, y):
    return torch.equal(x.view(torch.int16), y.view(torch.int16))


@pytest.fixture
def split_always():
    # force the split so that the scratch is used whatever the cost model says
    old_mode = g.gemm_set_streamk_mode(g.STREAMK_ALWAYS)
    yield
    g.gemm_set_streamk_mode(old_mode)


@pytest.mark.parametrize("variant", [g.VARIANT_AUTO, g.VARIANT_1CTA, g.VARIANT_2CTA,
                                     g.VARIANT_1CTA | g.VARIANT_DIRECT_STORE])
@pytest.mark.parametrize("shape", [(300, 520, 1040), (129, 1031, 640), (10240, 1024, 320)])
def test_noalloc_matches_workspace_entry_point(split_always, variant, shape):
    M, N, K = shape
    A_cpu, B_cpu = gi.bf16_operands(M, N, K, seed=M + N + K)
    A, B = A_cpu.cuda(), B_cpu.cuda()
    ws = g.streamk_workspace(False, variant)
    want = _existing(A, B, variant, ws)
    rows, cols = P.sample_positions(M, N, 2000, seed=7)
    D_ref, S = oracle.gemm_bf16_entries(gi.bf16_codes(A_cpu), gi.bf16_codes(B_cpu), rows, cols)
    for call in range(2):
        got, sched = _noalloc(A, B, variant)
        assert sched["sk_tiles"] > 0, "the stream-K split was expected for this shape"
        assert _same_bits(got, want), f"call {call}: D differs from gemm_bf16_streamk's"
        P.check_within_bound(P.bf16_to_f64(got)[rows, cols], D_ref, S, f"noalloc call {call}")


def test_noalloc_after_a_timeout(split_always):
    """A no-alloc call whose launch gives up (watchdog test hook) leaves flag
    words and partials behind in the shared scratch; later calls, of another
    kernel variant and then the same one, must still be exact."""
    M, N, K = 1024, 1024, 4096
    A_cpu, B_cpu = gi.bf16_operands(M, N, K, seed=91)
    A, B = A_cpu.cuda(), B_cpu.cuda()
    D = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    old_ms = g.gemm_set_watchdog_ms(100)
    try:
        assert g.gemm_debug_stall_next_launch(2) == g.GEMM_OK
        assert g.gemm_bf16_streamk_noalloc(g.VARIANT_2CTA, A.data_ptr(), B.data_ptr(), D.data_ptr(),
                                           M, N, K, K, K, N, s) == g.GEMM_OK
        assert g.gemm_last_schedule()["sk_tiles"] > 0
        assert g.gemm_last_status(s) == g.GEMM_ERR_TIMEOUT
    finally:
        g.gemm_set_watchdog_ms(old_ms)
    rows, cols = P.sample_positions(M, N, 2000, seed=8)
    D_ref, S = oracle.gemm_bf16_entries(gi.bf16_codes(A_cpu), gi.bf16_codes(B_cpu), rows, cols)
    for variant in (g.VARIANT_1CTA, g.VARIANT_2CTA):
        want = _existing(A, B, variant, g.streamk_workspace(False, variant))
        got, sched = _noalloc(A, B, variant)
        assert sched["sk_tiles"] > 0
        assert _same_bits(got, want), f"variant {variant} after the timeout"
        P.check_within_bound(P.bf16_to_f64(got)[rows, cols], D_ref, S, "after the timeout")


_FIRST_CALL = textwrap.dedent("""
    import sys
    sys.path.insert(0, {root!r})
    import torch
    import dense_gemm_blackwell_tcgen05_gb300 as g
    import gemm_inputs as gi
    g.gemm_set_streamk_mode(g.STREAMK_ALWAYS)
    M, N, K = 700, 900, 2048
    A, B = (t.cuda() for t in gi.bf16_operands(M, N, K, seed=5))
    torch.cuda.synchronize()
    side = torch.cuda.Stream()            # a non-blocking stream of torch's pool
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc = g.gemm_bf16_streamk_noalloc(g.VARIANT_AUTO, A.data_ptr(), B.data_ptr(), D.data_ptr(),
                                     M, N, K, K, K, N, side.cuda_stream)
    assert rc == g.GEMM_OK, rc
    assert g.gemm_last_schedule()["sk_tiles"] > 0
    assert g.gemm_last_status(side.cuda_stream) == g.GEMM_OK
    ws = g.streamk_workspace(False, g.VARIANT_AUTO)
    W = torch.full_like(D, float("nan"))
    rc = g.gemm_bf16_streamk(g.VARIANT_AUTO, A.data_ptr(), B.data_ptr(), W.data_ptr(), M, N, K,
                             K, K, N, ws.data_ptr(), ws.numel(), 0)
    assert rc == g.GEMM_OK and g.gemm_last_status(0) == g.GEMM_OK
    assert torch.equal(D.view(torch.int16), W.view(torch.int16)), "first call differs"
    print("first-call-ok")
""")


def test_noalloc_first_call_on_a_non_blocking_stream():
    """In a fresh process (so that this is the scratch's first use on the
    device): the set-up clear is ordered before the kernel on the caller's
    own non-blocking stream, and the result equals the workspace entry
    point's bit for bit."""
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL.format(root=ROOT)], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "first-call-ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]


def test_noalloc_rejects_what_it_cannot_run():
    A = torch.zeros(256, 256, dtype=torch.bfloat16, device="cuda")
    D = torch.empty(256, 256, dtype=torch.bfloat16, device="cuda")
    f = lambda v: g.gemm_bf16_streamk_noalloc(v, A.data_ptr(), A.data_ptr(), D.data_ptr(), 256,
                                              256, 256, 256, 256, 256, 0)
    assert f(g.VARIANT_SYNC) == g.GEMM_ERR_INVALID_ARG
    assert f(0x40) == g.GEMM_ERR_INVALID_ARG
    assert f(g.VARIANT_2CTA) == g.GEMM_OK
    torch.cuda.synchronize()
