"""Each plausible slip in the oracle must trip at least one pin.

Mutants are textual edits of ``oracle.c`` compiled into a temporary library
on the CPU: a flipped sign, a dropped term, a transposed or mis-strided
operand, wrong exponent biases, a wrong scale block, a wrong rounding rule.
"""
import os

import pytest

import oracle
from tests import oracle_pins

MUTANTS = {
    "sign": ("acc += p;", "acc -= p;"),
    "dropped_last_term": ("for (int64_t k = 0; k < K; ++k) {\n        double p = oracle_bf16",
                          "for (int64_t k = 0; k < K - 1; ++k) {\n        double p = oracle_bf16"),
    "transposed_B_row": ("dot_bf16(A + i * lda, B + j * ldb", "dot_bf16(A + j * lda, B + i * ldb"),
    "ignores_lda": ("dot_bf16(A + i * lda", "dot_bf16(A + i * K"),
    "entries_swapped": ("dot_bf16(A + rows[t] * lda, B + cols[t] * ldb",
                        "dot_bf16(A + cols[t] * lda, B + rows[t] * ldb"),
    "e4m3_bias": ("e - 7);     /* normal */", "e - 8);     /* normal */"),
    "e4m3_mantissa": ("(double)m / 8.0", "(double)m / 16.0"),
    "e4m3_subnormal": ("ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    "e4m3_nan": ("if (e == 0xF && m == 0x7)", "if (e == 0xF && m == 0x6)"),
    "ue8m0_bias": ("(int)e - 127", "(int)e - 128"),
    "scale_block_16": ("sfa[k / 32]", "sfa[k / 16]"),
    "scale_operand_swap": ("oracle_ue8m0_to_f64(sfb[k / 32])", "oracle_ue8m0_to_f64(sfa[k / 32])"),
    "mx_row_stride": ("SFA + i * ldsfa", "SFA + i * ldsfb"),
    "abs_sum": ("abs_acc += fabs(p);", "abs_acc += p;"),
    "bf16_trunc": ("rint(x / quantum)", "trunc(x / quantum)"),
    "bf16_ties_away": ("rint(x / quantum)", "round(x / quantum)"),
    "bf16_precision": ("ldexp(1.0, lead - 7)", "ldexp(1.0, lead - 8)"),
    "bf16_decode_shift": ("(uint32_t)h << 16", "(uint32_t)h << 15"),
    "e4m3_enc_trunc": ("rint(a / quantum) * quantum;   /* ties to even */",
                       "trunc(a / quantum) * quantum;   /* ties to even */"),
    "e4m3_enc_min_exp": ("    if (lead < -6)\n        lead = -6;", "    if (lead < -7)\n        lead = -7;"),
    "quant_448": ("amax <= ldexp(448.0, e - 1)", "amax <= ldexp(480.0, e - 1)"),
    "quant_not_minimal": ("e = (int)ceil(log2(amax / 448.0));\n                while (amax > ldexp(448.0, e))\n                    ++e;\n                while (e > -127 && amax <= ldexp(448.0, e - 1))\n                    --e;",
                          "e = (int)ceil(log2(amax / 448.0)) + 1;\n                while (amax > ldexp(448.0, e))\n                    ++e;"),
    "quant_block_16": ("int64_t k0 = b * 32, k1 = k0 + 32 < K ? k0 + 32 : K;", "int64_t k0 = b * 32, k1 = k0 + 16 < K ? k0 + 16 : K;"),
    "quant_scale_sign": ("oracle_f64_to_e4m3_rne(ldexp(x, -e))", "oracle_f64_to_e4m3_rne(ldexp(x, e))"),
    "epi_bias_by_row": ("if (bias) v += bias[j];", "if (bias) v += bias[i];"),
    "epi_beta_as_alpha": ("if (C) v += beta * C[i * ldc + j];", "if (C) v += alpha * C[i * ldc + j];"),
    "epi_ignores_ldc": ("if (C) v += beta * C[i * ldc + j];", "if (C) v += beta * C[i * N + j];"),
    "epi_relu_sign": ("return v < 0.0 ? 0.0 : v;", "return v > 0.0 ? 0.0 : v;"),
    "epi_gelu_scale": ("erf(v / sqrt(2.0))", "erf(v / 2.0)"),
    "epi_gelu_half": ("return v * 0.5 * (1.0 + erf", "return v * (1.0 + erf"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(oracle.SRC).read()
    assert src.count(before) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(before, after, 1)
    path = tmp_path / "oracle_mutant.c"
    path.write_text(mutated)
    lib = oracle.build(force=True, src=str(path), out=str(tmp_path / f"lib_{name}.so"))
    failed = oracle_pins.failing_pins(oracle.Oracle(lib))
    assert failed, f"mutant {name} passes every pin"
