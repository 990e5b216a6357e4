"""Planted mistakes in the oracle must fail a pin.

Each mutant is a copy of oracle.c with one plausible mistake (a dropped
term, a wrong sign, index or bias, a transposed operand, a double rounding),
compiled on the CPU into a temporary library.  The pins of
test_oracle_pins run against it, and at least one must fail.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

MUTANTS = {
    "nibble_order_swapped": (
        "return (k & 1) ? (unsigned)(byte >> 4) : (unsigned)(byte & 0xFu);",
        "return (k & 1) ? (unsigned)(byte & 0xFu) : (unsigned)(byte >> 4);"),
    "sign_bit_wrong": (
        "return (code & 8u) ? -mag : mag;", "return (code & 4u) ? -mag : mag;"),
    "table_3_4_swapped": (
        "{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}", "{0.0, 0.5, 1.0, 1.5, 2.0, 4.0, 3.0, 6.0}"),
    "e8m0_bias_off_by_one": (
        "return ldexp(1.0, (int)code - 127);", "return ldexp(1.0, (int)code - 126);"),
    "scale_b_dropped": (
        "double b = vb * oracle_e8m0_value(eb);",
        "double b = vb;"),
    "scale_block_16": (
        "unsigned ea = sarow[k / 32], eb = sbrow[k / 32];",
        "unsigned ea = sarow[k / 16], eb = sbrow[k / 32];"),
    "scale_a_indexed_by_n": (
        "const uint8_t *sarow = j->SA + (int64_t)m * j->ldsa;",
        "const uint8_t *sarow = j->SA + (int64_t)(n % j->M) * j->ldsa;"),
    "last_k_dropped": (
        "for (int64_t k = 0; k < j->K; ++k) {", "for (int64_t k = 0; k + 1 < j->K; ++k) {"),
    "beta_term_dropped": ("y = p1 + p2;", "y = p1;"),
    "alpha_ignored": ("double p1 = j->alpha * acc;", "double p1 = acc;"),
    "alpha_beta_swapped": (
        "double p1 = j->alpha * acc;\n        double p2 = j->beta * c;",
        "double p1 = j->beta * acc;\n        double p2 = j->alpha * c;"),
    "double_rounding_via_float": (
        "*d = oracle_bf16_rne(y);", "*d = oracle_bf16_rne((double)(float)y);"),
    "ties_away_from_zero": (
        "if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) != 0.0))", "if (frac >= 0.5)"),
    "no_subnormal_clamp": (
        "int q = (E - 1 > -126 ? E - 1 : -126) - 7;", "int q = E - 1 - 7;"),
    "quant_ties_to_odd": (
        "if (d < best_d || (d == best_d && (c & 1u) == 0u)) {",
        "if (d < best_d || (d == best_d && (c & 1u) == 1u)) {"),
    "quant_exponent_rounded_up": (
        "while (ldexp(6.0, s + 1) <= amax)", "while (ldexp(4.0, s + 1) <= amax)"),
    "quant_scale_bias_126": (
        "S[(int64_t)r * lds + b] = (uint8_t)(s + 127);", "S[(int64_t)r * lds + b] = (uint8_t)(s + 126);"),
    "quant_nibbles_swapped": (
        "(uint8_t)(code[0] | (code[1] << 4));", "(uint8_t)(code[1] | (code[0] << 4));"),
    "quant_amax_half_block": (
        "for (int i = 0; i < 32; ++i) {\n                const double v = fabs(",
        "for (int i = 0; i < 16; ++i) {\n                const double v = fabs("),
    "quant_sign_dropped_for_zero": ("if (signbit(v))", "if (v < 0.0)"),
    "fp8_e4m3_bias_8": (
        "bias = fmt == 1 ? 7 : 15;", "bias = fmt == 1 ? 8 : 15;"),
    "fp8_e5m2_three_mantissa_bits": (
        "mbits = fmt == 1 ? 3 : 2,", "mbits = fmt == 1 ? 3 : 3,"),
    "fp8_subnormal_implicit_one": (
        "(e == 0 ? 0.0 : 1.0) + ldexp", "1.0 + ldexp"),
    "fp8_e4m3_nan_whole_top_binade": (
        "if (fmt == 1 && e == emax && m == (1u << mbits) - 1u)", "if (fmt == 1 && e == emax)"),
    "fp8_adjacent_elements_swapped": (
        "return oracle_fp8_value_q(row[k], fmt, q);",
        "return oracle_fp8_value_q(row[k ^ 1], fmt, q);"),
    "fp8_b_decoded_in_a_format": (
        "vb = byte_form_value(brow, k, j->fmt_b, &qb);",
        "vb = byte_form_value(brow, k, j->fmt_a, &qb);"),
    "fp6_e2m3_bias_0": ("bias = fmt == 3 ? 1 : 3;", "bias = fmt == 3 ? 0 : 3;"),
    "fp6_e3m2_bias_4": ("bias = fmt == 3 ? 1 : 3;", "bias = fmt == 3 ? 1 : 4;"),
    "fp6_sign_bit_7": ("const unsigned s = (code >> 5) & 1u;", "const unsigned s = (code >> 7) & 1u;"),
    "fp6_subnormal_implicit_one": (
        "const unsigned sig = e == 0 ? m : (m | (1u << mbits));",
        "const unsigned sig = m | (1u << mbits);"),
    "fp6_field_widths_swapped": (
        "const int ebits = fmt == 3 ? 2 : 3, mbits = fmt == 3 ? 3 : 2,",
        "const int ebits = fmt == 3 ? 3 : 2, mbits = fmt == 3 ? 2 : 3,"),
    "fp6_padding_read_as_data": (
        "const uint8_t *g = row + (k >> 4) * 16;", "const uint8_t *g = row + (k >> 4) * 12;"),
    "fp6_codes_msb_first": (
        "const int bit = 6 * (int)(k & 15);", "const int bit = 6 * (int)(15 - (k & 15));"),
    "fp4_padded_nibbles_swapped": (
        "return (k & 1) ? pair >> 4 : pair & 15u;", "return (k & 1) ? pair & 15u : pair >> 4;"),
    "fp4_padded_padding_read_as_data": (
        "const unsigned pair = row[(k >> 4) * 16 + ((k & 15) >> 1)];",
        "const unsigned pair = row[(k >> 4) * 8 + ((k & 15) >> 1)];"),
    "fp4_padded_granule_too_coarse": ("*q = -1;                       /* E2M1",
                                      "*q = 1;                       /* E2M1"),
    "fp6_decoded_as_fp8": ("    if (fmt >= 3)\n        return oracle_fp6_value_q(",
                           "    if (fmt > 3)\n        return oracle_fp6_value_q("),
    "fp8_granule_of_fp4": (
        "int g = qa + qb + (int)ea + (int)eb - 254;", "int g = (int)ea + (int)eb - 256;"),
    "quant8_ties_to_odd": (
        "if (d < best_d || (d == best_d && !(c & 1u))) {",
        "if (d < best_d || (d == best_d && (c & 1u))) {"),
    "quant8_e4m3_emax_7": (
        "static const int kEmax[6] = {0, 8, 15, 2, 4, 2};",
        "static const int kEmax[6] = {0, 7, 15, 2, 4, 2};"),
    "quant8_e3m2_emax_3": (
        "static const int kEmax[6] = {0, 8, 15, 2, 4, 2};",
        "static const int kEmax[6] = {0, 8, 15, 2, 3, 2};"),
    "quant8_e2m1_sign_bit_7": (
        "static const unsigned kSign[6] = {0u, 0x80u, 0x80u, 0x20u, 0x20u, 0x8u};",
        "static const unsigned kSign[6] = {0u, 0x80u, 0x80u, 0x20u, 0x20u, 0x80u};"),
    "quant8_fp6_straddle_dropped": (
        "if (at % 8 > 2)", "if (at % 8 > 4)"),
    "quant8_padding_not_cleared": ("        memset(g, 0, 16);", "        memset(g, 0, 12);"),
    "quant8_scale_bias_126": ("(uint8_t)(127 + s);", "(uint8_t)(126 + s);"),
    "quant8_sign_dropped_for_zero": ("if (signbit(v) != 0)", "if (v < 0.0)"),
    "quant8_amax_half_block": (
        "for (int i = 0; i < 32; ++i)\n                amax = fmax(",
        "for (int i = 0; i < 16; ++i)\n                amax = fmax("),
    "nv_scale_block_32": (
        "double an = va * oracle_ue4m3_value_q(sarow[k / 16], &sa_q);",
        "double an = va * oracle_ue4m3_value_q(sarow[k / 32], &sa_q);"),
    "nv_b_scale_from_a": (
        "double bn = vb * oracle_ue4m3_value_q(sbrow[k / 16], &sb_q);",
        "double bn = vb * oracle_ue4m3_value_q(sarow[k / 16], &sb_q);"),
    "nv_scale_read_as_e8m0": (
        "    return oracle_fp8_value_q(code, 1, ulp_exp);\n}",
        "    if (ulp_exp)\n        *ulp_exp = 0;\n    return oracle_e8m0_value(code);\n}"),
    "nv_sign_bit_accepted": (
        "    if (code & 0x80u) {\n        if (ulp_exp)",
        "    if (code & 0x100u) {\n        if (ulp_exp)"),
    "nv_granule_without_scales": (
        "                min_g = qa + qb + sa_q + sb_q;",
        "                min_g = qa + qb;"),
    "nv_beta_dropped_only_for_nv": (
        "    j.M = M; j.N = N; j.K = K; j.nv = 1;\n    j.A = A; j.lda_bytes = lda / 2; j.B = B; j.ldb_bytes = ldb / 2;\n    j.SA = SA; j.ldsa = ldsa; j.SB = SB; j.ldsb = ldsb;\n    j.alpha = alpha; j.beta = beta; j.C = C; j.ldc = ldc;\n    j.D = D; j.ldd = ldd;",
        "    j.M = M; j.N = N; j.K = K; j.nv = 1;\n    j.A = A; j.lda_bytes = lda / 2; j.B = B; j.ldb_bytes = ldb / 2;\n    j.SA = SA; j.ldsa = ldsa; j.SB = SB; j.ldsb = ldsb;\n    j.alpha = alpha; j.beta = 0.0; j.C = C; j.ldc = ldc;\n    j.D = D; j.ldd = ldd;"),
    "transposed_d_store": (
        "if (!one_output(j, m, n, &j->D[(int64_t)m * j->ldd + n],",
        "if (!one_output(j, m, n, &j->D[(int64_t)(n % j->M) * j->ldd + (m % j->N)],"),
}


@pytest.fixture(scope="module")
def source():
    with open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation site for {name} not found"
    src = tmp_path / "oracle_mutant.c"
    src.write_text(source.replace(old, new))
    so = tmp_path / "liboracle_mutant.so"
    subprocess.check_call(["gcc", *oracle.GCC_FLAGS, str(src), "-o", str(so), "-lm"])
    monkeypatch.setattr(oracle, "_lib", oracle.bind(str(so)))
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(oracle)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"mutant {name} passed every pin"
