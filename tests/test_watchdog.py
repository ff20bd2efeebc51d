"""The device watchdog: a stage that never fills makes the kernel's bounded
waits run out; the launch must return with GEMM_ERR_TIMEOUT in the status
word (no fault, no trap, no hang) and the context must stay usable."""
import numpy as np
import pytest
import torch

import dense_gemm_blackwell_tcgen05_gb300 as g
import gemm_inputs as gi
import oracle
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture
def short_watchdog():
    old = g.gemm_set_watchdog_ms(100)
    yield
    g.gemm_set_watchdog_ms(old)


def _bf16(variant, A, B, D, s):
    M, K = A.shape
    N = B.shape[0]
    return g.gemm_bf16_variant(variant, A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, K, K,
                               N, s)


@pytest.mark.parametrize("variant", [g.VARIANT_1CTA, g.VARIANT_2CTA,
                                     g.VARIANT_1CTA | g.VARIANT_DIRECT_STORE])
@pytest.mark.parametrize("stall", [0, 5])
def test_bf16_stall_times_out_then_recovers(short_watchdog, variant, stall):
    M, N, K = 512, 768, 1024
    A, B = gi.bf16_operands(M, N, K, seed=21)
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert g.gemm_debug_stall_next_launch(stall) == g.GEMM_OK
    assert _bf16(variant, Ad, Bd, D, s) == g.GEMM_OK
    word = g.gemm_last_status_word(s)
    assert word >> 56 == 5, hex(word)                  # timeout code recorded
    assert g.gemm_last_status(s) == g.GEMM_ERR_TIMEOUT
    assert g.gemm_last_status(s) == g.GEMM_OK          # cleared by the read
    # the next launch (no stall requested) is correct
    assert _bf16(variant, Ad, Bd, D, s) == g.GEMM_OK
    assert g.gemm_last_status(s) == g.GEMM_OK
    D_ref, S = oracle.gemm_bf16(gi.bf16_codes(A), gi.bf16_codes(B))
    P.check_within_bound(P.bf16_to_f64(D), D_ref, S, "after recovery")


@pytest.mark.parametrize("variant", [g.VARIANT_1CTA | g.VARIANT_DIRECT_STORE, g.VARIANT_2CTA])
def test_mxfp8_stall_times_out_then_recovers(short_watchdog, variant):
    M, N, K = 384, 512, 1024
    A, SFA, B, SFB = gi.mxfp8_operands(M, N, K, seed=22)
    t = [x.cuda() for x in (A, SFA, B, SFB)]
    D = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream

    def call():
        return g.gemm_mxfp8_variant(variant, t[0].data_ptr(), t[2].data_ptr(), t[1].data_ptr(),
                                    t[3].data_ptr(), D.data_ptr(), M, N, K, K, K, SFA.shape[1],
                                    SFB.shape[1], N, s)

    assert g.gemm_debug_stall_next_launch(3) == g.GEMM_OK
    assert call() == g.GEMM_OK
    assert g.gemm_last_status(s) == g.GEMM_ERR_TIMEOUT
    assert call() == g.GEMM_OK
    assert g.gemm_last_status(s) == g.GEMM_OK
    D_ref, S = oracle.gemm_mxfp8(A.numpy(), B.numpy(), SFA.numpy(), SFB.numpy())
    P.check_within_bound(P.bf16_to_f64(D), D_ref, S, "mx after recovery")


def test_stall_request_is_one_shot_and_validated():
    assert g.gemm_debug_stall_next_launch(-1) == g.GEMM_ERR_INVALID_ARG
