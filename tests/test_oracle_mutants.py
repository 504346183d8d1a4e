"""Planted mistakes: each mutant is a copy of the oracle's C source with one plausible error (a
dropped term, a wrong sign, a shifted bit, a transposed index).  The pin suite must reject every
one of them, which shows the pins constrain each part of the oracle and not only its happy path.
The mistakes are planted in a temporary copy of the oracle, on the CPU; nothing here touches a GPU.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "tmap_oracle.c")

MUTANTS = {
    "swizzle_row_bits_shifted": ("(off >> 7)", "(off >> 8)"),
    "swizzle_64b_takes_three_row_bits": ("xor_bits = 2;", "xor_bits = 3;"),
    "swizzle_32b_takes_two_row_bits": ("xor_bits = 1;", "xor_bits = 2;"),
    "swizzle_sector_bits_shifted": ("return off ^ (line << 4);", "return off ^ (line << 5);"),
    # other valid-looking XOR patterns for the narrow modes (involutions that keep every chunk in
    # its row, depend on row % 8 and still spread a column over eight bank sectors)
    "swizzle_64b_row_bits_reversed": (
        "uint64_t line = (off >> 7) & ((1u << xor_bits) - 1u);",
        "uint64_t line = xor_bits == 2 ? (((off >> 8) & 1u) | (((off >> 7) & 1u) << 1))\n"
        "                                : (off >> 7) & ((1u << xor_bits) - 1u);"),
    "swizzle_32b_mixes_row_bits": (
        "uint64_t line = (off >> 7) & ((1u << xor_bits) - 1u);",
        "uint64_t line = xor_bits == 1 ? (((off >> 7) ^ (off >> 6)) & 1u)\n"
        "                                : (off >> 7) & ((1u << xor_bits) - 1u);"),
    "oob_upper_off_by_one": ("(uint64_t)g[i] >= m->dim[i]", "(uint64_t)g[i] > m->dim[i]"),
    "oob_negative_dropped": ("if (g[i] < 0 || (uint64_t)g[i]", "if ((uint64_t)g[i] + 0 == 0 && (uint64_t)g[i]"),
    "image_axes_transposed": (
        "    for (uint32_t e1 = 0; e1 < orc_extent(m, 1); e1++)\n"
        "    for (uint32_t e0 = 0; e0 < orc_extent(m, 0); e0++) {",
        "    for (uint32_t e0 = 0; e0 < orc_extent(m, 0); e0++)\n"
        "    for (uint32_t e1 = 0; e1 < orc_extent(m, 1); e1++) {"),
    "element_stride_ignored": ("(int64_t)e[i] * step_of(m, i);", "(int64_t)e[i];"),
    "element_stride_in_bytes": ("(int64_t)e[i] * step_of(m, i);",
                                "(int64_t)e[i] * step_of(m, i) / (int64_t)m->esize;"),
    "extent_floor_not_ceil": ("(m->box[i] + m->estride[i] - 1) / m->estride[i]",
                              "m->box[i] / m->estride[i] + (m->box[i] < m->estride[i])"),
    "f32_fill_is_infinity": ("case ORC_FILL_NAN_F32: v = 0x7FC00000u;",
                             "case ORC_FILL_NAN_F32: v = 0x7F800000u;"),
    "fill_bytes_reversed": ("return (uint8_t)(v >> (8 * k));",
                            "return (uint8_t)(v >> (8 * (m->esize - 1 - k)));"),
    "gemm_drops_last_k": ("    for (uint64_t i = 0; i < k; i++) {\n        acc += bf16_to_double(a[m * lda + i]) * bf16_to_double(b[n * ldb + i]);",
                          "    for (uint64_t i = 0; i + 1 < k; i++) {\n        acc += bf16_to_double(a[m * lda + i]) * bf16_to_double(b[n * ldb + i]);"),
    "gemm_b_transposed": ("acc += bf16_to_double(a[m * lda + i]) * bf16_to_double(b[n * ldb + i]);",
                          "acc += bf16_to_double(a[m * lda + i]) * bf16_to_double(b[i * ldb + n]);"),
    "gemm_float_accumulator": ("    double acc = 0.0;\n    for (uint64_t i = 0; i < k; i++) {\n        acc += bf16_to_double(a[m * lda + i])",
                               "    float acc = 0.0f;\n    for (uint64_t i = 0; i < k; i++) {\n        acc += bf16_to_double(a[m * lda + i])"),
    "gemm_block_rows_swapped": ("out[(m - m0) * (n1 - n0) + (n - n0)] = orc_gemm_dot(a, lda, b, ldb, k, m, n);",
                                "out[(m - m0) * (n1 - n0) + (n - n0)] = orc_gemm_dot(a, lda, b, ldb, k, n, m);"),
    "grid_floor_not_ceil": ("return (m->dim[i] + m->box[i] - 1) / m->box[i];",
                            "return m->dim[i] / m->box[i] + (m->dim[i] < m->box[i]);"),
    "stride_index_transposed": ("off += g[i] * m->stride[i];",
                                "off += g[i] * m->stride[m->rank - 1 - i];"),
    "reduce_wrong_sign": ("d = d + a;", "d = d - a;"),
    "checksum_tree_halves": ("sums[i] = sums[2 * i] + sums[2 * i + 1];",
                             "sums[i] = sums[i] + sums[i + n / 2];"),
    "mbar_ignores_tx": ("if (b->pending == 0 && b->tx == 0) {", "if (b->pending == 0) {"),
    "store_writes_oob": ("    if (!in_bounds(m, g)) return;\n    uint8_t* dst = element_address(m, g);\n    for",
                         "    uint8_t* dst = element_address(m, g);\n    if (!in_bounds(m, g)) dst = dst + 0;\n    for"),
    "checksum_bits_dropped_high_byte": ("(img[orc_swz(off + 1, span)] << 8)",
                                        "(img[orc_swz(off + 1, span)] << 0)"),
    "half_add_rounds_half_up": ("double n = nearbyint(v / q);", "double n = floor(v / q + 0.5);"),
    "s32_min_compares_unsigned": ("        if (op == ORC_MIN) return (uint32_t)(x < y ? x : y);",
                                  "        if (op == ORC_MIN) return a < b ? a : b;"),
    "subnormals_flushed": ("if (E < emin) E = emin;", "if (E < emin) return sign_bit;"),
    "float_max_picks_smaller": ("if (op == ORC_MAX) return x > y ? a : (y > x ? b : a);",
                                "if (op == ORC_MAX) return x < y ? a : (y < x ? b : a);"),
    "half_add_drops_operand": ("    const double sum = x + y;", "    const double sum = x + 0 * y;"),
    "half_infinity_becomes_max_finite": ("    if (isinf(v)) return sign_bit | all_ones;\n",
                                         "    if (isinf(v)) return sign_bit | (all_ones - 1u);\n"),
    "half_nan_becomes_infinity": ("    if (isnan(v)) return all_ones | (1u << (mbits - 1));",
                                  "    if (isnan(v)) return all_ones;"),
    "min_takes_nan_src": ("    if (op == ORC_MIN) return x < y ? a : (y < x ? b : a);",
                          "    if (op == ORC_MIN) return x < y ? a : (x != x || y != y || y < x ? b : a);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    d = tmp_path / "oracle"
    d.mkdir()
    shutil.copy(os.path.join(ROOT, "oracle", "tmap_oracle.h"), d)
    (d / "tmap_oracle.c").write_text(src.replace(old, new))
    lib = d / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", str(lib), str(d / "tmap_oracle.c"), "-lm"], check=True)
    env = dict(os.environ, TMAP_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_reduce_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_stride_fill_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_gemm_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
