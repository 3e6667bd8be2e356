"""The pins are strong enough: each plausible slip planted in a copy of the oracle
source (swapped nibble, dropped min term, wrong sign or index, transposed
operand, wrong exponent bias...) makes at least one pin check fail.

The mistakes are planted in temporary copies compiled on the CPU; the real
oracle is untouched."""
import os

import pytest

import oracle
from tests import pin_checks

MUTANTS = {
    "q4k_low_nibble_swapped": ("int q_lo = qs[32 * c + l] & 15;", "int q_lo = qs[32 * c + l] >> 4;"),
    "q4k_min_dropped": ("d * sc_lo * q_lo - dmin * m_lo", "d * sc_lo * q_lo"),
    "q4k_min_sign": ("d * sc_hi * q_hi - dmin * m_hi", "d * sc_hi * q_hi + dmin * m_hi"),
    "q4k_high_bits_index": ("((s[j - 4] >> 6) << 4)", "((s[j] >> 6) << 4)"),
    "q4k_min_index": ("*m = s[j + 4] & 63;", "*m = s[j] & 63;"),
    "q4k_dmin_is_d": ("double dmin = orc_fp16_value(rd16(blk + 2));",
                      "double dmin = orc_fp16_value(rd16(blk));"),
    "q4k_hi_weight_slot": ("out[64 * c + 32 + l] =", "out[64 * c + 31 + l] ="),
    "q8_unsigned_bytes": ("int q = (int8_t)blk[2 + i];", "int q = blk[2 + i];"),
    "q8_block_stride": ("orc_decode_q8_0_block(row + 34 * b, out + 32 * b);",
                        "orc_decode_q8_0_block(row + 32 * b, out + 32 * b);"),
    "q4_0_nibble_order": ("int u_lo = qs[l] & 15;", "int u_lo = qs[l] >> 4;"),
    "q4_0_offset": ("(double)(u_hi - 8)", "(double)(u_hi - 7)"),
    "q4_0_unsigned_codes": ("(double)(u_lo - 8)", "(double)u_lo"),
    "q4_0_hi_weight_slot": ("out[16 + l] =", "out[15 + l] ="),
    "q4_0_nibbles_at": ("const uint8_t* qs = blk + 2;", "const uint8_t* qs = blk + 1;"),
    "q4_0_block_stride": ("orc_decode_q4_0_block(row + 18 * b", "orc_decode_q4_0_block(row + 16 * b"),
    "q4_0_row_bytes": ("cols / 32 * 18;", "cols / 32 * 16;"),
    "q6k_qh_shift": ("(qh[32 * h + l] >> (2 * g)) & 3", "(qh[32 * h + l] >> g) & 3"),
    "q6k_ql_half": ("ql[64 * h + 32 * (g & 1) + l]", "ql[64 * h + 32 * (g >> 1) + l]"),
    "q6k_nibble_shift": (">> (4 * (g >> 1))) & 15", ">> (4 * (g & 1))) & 15"),
    "q6k_offset": ("(double)(u - 32)", "(double)(u - 31)"),
    "q6k_unsigned_scales": ("const int8_t* sc = (const int8_t*)(blk + 192);", "const uint8_t* sc = blk + 192;"),
    "q6k_scale_index": ("sc[8 * h + 2 * g + l / 16]", "sc[8 * h + g + l / 16]"),
    "q6k_d_at": ("rd16(blk + 208)", "rd16(blk + 206)"),
    "q6k_high_bits_at": ("const uint8_t* qh = blk + 128;", "const uint8_t* qh = blk + 127;"),
    "q6k_row_bytes": ("cols / 256 * 210;", "cols / 256 * 208;"),
    "f32_row_stride": ("case ORC_F32: return 4 * cols;", "case ORC_F32: return 4 * cols + 4;"),
    "fp16_bias": ("expo - 25);", "expo - 24);"),
    "fp16_subnormal_scale": ("ldexp((double)frac, -24);", "ldexp((double)frac, -25);"),
    "bf16_widen": ("(uint32_t)b << 16;", "(uint32_t)b << 15;"),
    "gemv_x_row_stride": ("const float* xm = x + m * cols;", "const float* xm = x + m * rows;"),
    "gemv_last_column": ("for (int64_t c = 0; c < cols; ++c) {\n                double p = (double)w[c] * (double)xm[c];",
                         "for (int64_t c = 0; c + 1 < cols; ++c) {\n                double p = (double)w[c] * (double)xm[c];"),
    "gemv_abs_sum": ("aacc += fabs(p);\n            }\n            y[m * rows + r] = acc;\n            if (absy)",
                     "aacc += p;\n            }\n            y[m * rows + r] = acc;\n            if (absy)"),
    "gemm_bf16_widen": ("xd[i] = orc_bf16_value(X[i]);", "xd[i] = orc_bf16_value((uint16_t)(X[i] & 0xFFFE));"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(before) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(before, after))
    lib = oracle.compile_oracle(str(path), str(tmp_path / f"lib{name}.so"))
    mutant = oracle.Oracle(lib)
    failures = []
    for check in pin_checks.ALL_CHECKS:
        try:
            check(mutant)
        except (AssertionError, ValueError):
            failures.append(check.__name__)
    assert failures, f"no pin catches mutant {name}"
    os.remove(lib)
