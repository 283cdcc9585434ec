"""Mutation check of the oracle's pins (CPU only).

Each mutant below plants one plausible mistake in oracle/w4_oracle.c -- a
dropped term, a wrong sign, index or divisor, a transposed operand, ties
rounded the wrong way -- builds the changed source with the oracle's own
compiler flags into a temporary library, and runs the pin suites
(tests/test_oracle_pins.py, tests/test_oracle_ternary_pins.py) against it in
a child process (the oracle loads the library that
W4_ORACLE_LIB names).  Every mutant must make at least one pin fail; the
unchanged source, built and run the same way, must pass them all.

Mutants that cannot change any result are not listed, since no pin could
tell them apart from the oracle: the int4 quantiser's lower clamp at -8,
which max|W|/7 scaling never reaches, or moving the half conversion's
overflow test from 65520 to just above it, where the normal path's rounding
carry reaches infinity by itself.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

from oracle.build import SRC, compile_oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = [os.path.join(ROOT, "tests", name) for name in ("test_oracle_pins.py", "test_oracle_ternary_pins.py")]

# (name, [(text in w4_oracle.c, replacement), ...]); each text occurs once.
MUTANTS = [
    # fused dequant GEMV over the row-packed words
    ("gemv_zero_sign", [("double w = ((double)val - zero) * scale;",
                         "double w = ((double)val + zero) * scale;")]),
    ("gemv_nibble_order", [("uint32_t val = (packed_val >> (j * 4)) & 0x0Fu;",
                            "uint32_t val = (packed_val >> ((7 - j) * 4)) & 0x0Fu;")]),
    ("gemv_scale_dropped", [("double scale = load_elem(scales, act_dtype, row);\n"
                             "            double zero = load_elem(zeros, act_dtype, row);\n"
                             "            double sum = 0.0, abs_sum = 0.0;\n"
                             "            for (long i = 0; i < k_blocks; ++i) {",
                             "double scale = 1.0;\n"
                             "            double zero = load_elem(zeros, act_dtype, row);\n"
                             "            double sum = 0.0, abs_sum = 0.0;\n"
                             "            for (long i = 0; i < k_blocks; ++i) {")]),
    ("gemv_x_reversed", [("load_elem(x, act_dtype, c * K + i * 8 + j)",
                          "load_elem(x, act_dtype, c * K + i * 8 + (7 - j))")]),
    ("gemv_output_transposed", [("            d[c * N + row] = sum;\n            if (ref_abs) ref_abs[c * N + row] = abs_sum;\n"
                                 "        }\n    }\n}\n\n/*\n * Large-M",
                                 "            d[row * C + c] = sum;\n            if (ref_abs) ref_abs[row * C + c] = abs_sum;\n"
                                 "        }\n    }\n}\n\n/*\n * Large-M")]),
    # GEMM evaluated at sampled coordinates
    ("gemm_nibbles_swapped", [("double w0 = ((double)b_lo - z) * s;", "double w0 = ((double)b_hi - z) * s;"),
                              ("double w1 = ((double)b_hi - z) * s;", "double w1 = ((double)b_lo - z) * s;")]),
    ("gemm_zero_dropped", [("double z = (double)bf16_bits_to_float(zero[n]);", "double z = 0.0;")]),
    ("gemm_odd_a_row", [("double a1 = (double)bf16_bits_to_float(A[m * K + 2 * kp + 1]);",
                         "double a1 = (double)bf16_bits_to_float(A[m * K + 2 * kp]);")]),
    # int4 quantise and pack
    ("quant_divisor_8", [("float s = amax / 7.0f;", "float s = amax / 8.0f;")]),
    ("quant_ties_even", [("roundf(w / s);\n                if (r < -8.0f)", "rintf(w / s);\n                if (r < -8.0f)")]),
    ("quant_upper_clamp", [("if (r > 7.0f) r = 7.0f;", "if (r > 6.0f) r = 6.0f;")]),
    ("pack_nibbles_swapped", [("(uint8_t)(((unsigned)q[0] & 0x0Fu) | (((unsigned)q[1] & 0x0Fu) << 4));",
                               "(uint8_t)(((unsigned)q[1] & 0x0Fu) | (((unsigned)q[0] & 0x0Fu) << 4));")]),
    ("pack_offset_binary", [("(uint8_t)(((unsigned)q[0] & 0x0Fu) | (((unsigned)q[1] & 0x0Fu) << 4));",
                             "(uint8_t)(((unsigned)(q[0] + 8) & 0x0Fu) | (((unsigned)(q[1] + 8) & 0x0Fu) << 4));")]),
    # GEMV over the quantiser's packed columns
    ("packed_no_sign_extension", [("((byte >> 4) & 0x0Fu);\n                int q = (nib >= 8u) ? (int)nib - 16 : (int)nib;",
                                   "((byte >> 4) & 0x0Fu);\n                int q = (int)nib;")]),
    ("packed_halves_swapped", [("(k % 2 == 0) ? (byte & 0x0Fu) : ((byte >> 4) & 0x0Fu)",
                                "(k % 2 == 1) ? (byte & 0x0Fu) : ((byte >> 4) & 0x0Fu)")]),
    # int4 permute
    ("permute_table_entries", [("{0, 4, 8, 12, 2, 6, 10, 14, 1, 5, 9, 13, 3, 7, 11, 15}",
                                "{0, 8, 4, 12, 2, 6, 10, 14, 1, 5, 9, 13, 3, 7, 11, 15}")]),
    ("permute_no_nibble_swap", [("for (long g = 0; g < total_k; g += 4) {", "for (long g = 0; g < 0; g += 4) {")]),
    ("permute_swap_partner", [("stream[g + 0] = (uint8_t)((b0 & 0x0F) | ((b2 & 0x0F) << 4));",
                               "stream[g + 0] = (uint8_t)((b0 & 0x0F) | ((b1 & 0x0F) << 4));")]),
    ("permute_column_order", [("32 * (n_id % 4) +", "32 * (3 - n_id % 4) +")]),
    # int8 quantise, permute and GEMV
    ("int8_divisor_128", [("float s = amax / 127.0f;", "float s = amax / 128.0f;")]),
    ("int8_ties_even", [("roundf(w / s);\n            if (r < -128.0f)", "rintf(w / s);\n            if (r < -128.0f)")]),
    ("int8_permute_table", [("{0, 2, 4, 6, 8, 10, 12, 14, 1, 3, 5, 7, 9, 11, 13, 15}",
                             "{0, 2, 4, 6, 8, 10, 12, 14, 3, 1, 5, 7, 9, 11, 13, 15}")]),
    ("int8_column_order", [("64 * (n_id % 2) +", "64 * (1 - n_id % 2) +")]),
    ("int8_gemv_scale_dropped", [("double w = (double)q[k * N + n] * s;\n                double xv",
                                  "double w = (double)q[k * N + n];\n                double xv")]),
    ("int8_gemm_transposed_q", [("double w = (double)q[k * N + n] * s;\n            acc",
                                 "double w = (double)q[n * K + k] * s;\n            acc")]),
    ("packed_gemm_unsigned", [("unsigned nib = (k % 2 == 0) ? (byte & 0x0Fu) : (byte >> 4);\n            int q = (nib >= 8u) ? (int)nib - 16 : (int)nib;",
                               "unsigned nib = (k % 2 == 0) ? (byte & 0x0Fu) : (byte >> 4);\n            int q = (int)nib;")]),
    ("packed_gemm_halves", [("unsigned nib = (k % 2 == 0) ? (byte & 0x0Fu) : (byte >> 4);",
                             "unsigned nib = (k % 2 == 1) ? (byte & 0x0Fu) : (byte >> 4);")]),
    ("int8_gemm_a_column", [("double a = (double)bf16_bits_to_float(A[m * K + k]);\n            double w = (double)q[k * N + n] * s;",
                             "double a = (double)bf16_bits_to_float(A[k * M + m]);\n            double w = (double)q[k * N + n] * s;")]),
    ("packed_gemm_a_column", [("double a = (double)bf16_bits_to_float(A[m * K + k]);\n            double w = (double)q * s;",
                               "double a = (double)bf16_bits_to_float(A[k * M + m]);\n            double w = (double)q * s;")]),
    # fp32 -> half conversion used by block_q8_1
    ("half_ties_down", [("if (rest > 0x1000u || (rest == 0x1000u && (half & 1u))) ++half;",
                         "if (rest > 0x1000u) ++half;")]),
    ("half_subnormal_ties_down", [("if (frac > 0.5 || (frac == 0.5 && (r & 1u))) ++r;", "if (frac > 0.5) ++r;")]),
    ("half_exponent_bias", [("uint32_t exp = ((mag >> 23) - 127 + 15);", "uint32_t exp = ((mag >> 23) - 127 + 14);")]),
    ("half_overflow_threshold", [("if (mag >= 0x477FF000u) return", "if (mag >= 0x48000000u) return")]),
    ("half_decode_subnormal_scale", [("? ldexp((double)m, -24) :", "? ldexp((double)m, -23) :")]),
    ("half_decode_bias", [("ldexp((double)(m | 0x400), e - 25)", "ldexp((double)(m | 0x400), e - 24)")]),
    ("half_decode_infinity", [("v = (m == 0) ? HUGE_VAL : NAN;", "v = (m == 0) ? 65536.0 : NAN;")]),
    # block_q8_1 in the PT layout and the W4A8 GEMV
    ("q8_1_divisor_128", [("float d = amax / 127.0f;", "float d = amax / 128.0f;")]),
    ("q8_1_s_without_d", [("float_to_half_bits(d * (float)sum)", "float_to_half_bits((float)sum)")]),
    ("q8_1_block_major_layout", [("v[16 * ((e / 16) * bpr + i) + e % 16] = (uint8_t)(int8_t)q;",
                                  "v[16 * (i * 8 + e / 16) + e % 16] = (uint8_t)(int8_t)q;")]),
    ("w4a8_zero_correction_sign", [("total += db * (double)dot - zero * sb;",
                                    "total += db * (double)dot + zero * sb;")]),
    ("w4a8_block_major_read", [("int qs = (int)(int8_t)v[16 * ((e / 16) * bpr + i) + e % 16];",
                                "int qs = (int)(int8_t)v[16 * (i * 8 + e / 16) + e % 16];")]),
    ("w4a8_d_and_s_swapped", [("double db = half_bits_to_double((uint16_t)(ds[0] | (ds[1] << 8)));",
                               "double db = half_bits_to_double((uint16_t)(ds[2] | (ds[3] << 8)));")]),
    # ternary PTQ1_0 / PTQ1_1 formats and their MMVQ
    ("ternary_contiguous_head", [("if (e < 80) { *pos = e >> 4; return e & 15; }",
                                  "if (e < 80) { *pos = e % 5; return e / 5; }")]),
    ("ternary_contiguous_middle", [("if (e < 120) { *pos = (e - 80) >> 3; return 16 + ((e - 80) & 7); }",
                                    "if (e < 120) { *pos = (e - 80) % 5; return 16 + (e - 80) / 5; }")]),
    ("ternary_digit_weights_reversed", [("return (byte / k_pow3[pos]) % 3;", "return (byte / k_pow3[4 - pos]) % 3;"),
                                        ("(blk[byte] + (t + 1) * k_pow3[pos])", "(blk[byte] + (t + 1) * k_pow3[4 - pos])")]),
    ("ternary_qh_field_order", [("(int)((qh >> (2 * pos)) & 3u)", "(int)((qh >> (2 * (7 - pos))) & 3u)")]),
    ("ternary_codebook_rarest_first", [("return (x->count < y->count) - (x->count > y->count);",
                                        "return (x->count > y->count) - (x->count < y->count);")]),
    ("ternary_codebook_ties_descending", [("return (x->key > y->key) - (x->key < y->key);",
                                           "return (x->key < y->key) - (x->key > y->key);")]),
    ("ternary_free_trit_position", [("(idx / 256) * k_pow3[4]", "(idx / 256) * k_pow3[3]")]),
    ("ternary_mantissa_bit_order", [("m |= 1u << bit;", "m |= 1u << (9 - bit);")]),
    ("ternary_escape_lookup", [("pattern = esc_patt + 8 * i; break;", "pattern = esc_patt; break;")]),
    ("ternary_superblock_qs_shift", [("trit_digit(o[24 * s + byte], pos)", "trit_digit(o[24 * ((s + 1) % 8) + byte], pos)")]),
    ("ternary_superblock_tail_order", [("int u = 8 * s + j;\n            t[128 * s + 120 + j]",
                                        "int u = 8 * j + s;\n            t[128 * s + 120 + j]")]),
    ("mmvq_digit_for_trit", [("dot += (long)t[128 * b + e] * qs;", "dot += (long)(t[128 * b + e] + 1) * qs;")]),
    ("mmvq_s_for_d", [("double dx = half_bits_to_double((uint16_t)(ds[0] | (ds[1] << 8)));",
                       "double dx = half_bits_to_double((uint16_t)(ds[2] | (ds[3] << 8)));")]),
    ("mmvq_first_block_scale", [("double w = half_bits_to_double(dw[b]);", "double w = half_bits_to_double(dw[0]);")]),
]


def _mutate(source, edits):
    for old, new in edits:
        assert source.count(old) == 1, "mutation text must occur exactly once: %r" % old
        source = source.replace(old, new)
    return source


def _run_pins(name, source, workdir):
    """Build `source` as a library and run the pin suite against it; return
    (exit code, last lines of output)."""
    src = os.path.join(workdir, name + ".c")
    lib = os.path.join(workdir, name + ".so")
    with open(src, "w") as f:
        f.write(source)
    compile_oracle(src, lib)
    env = dict(os.environ, W4_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", *PINS, "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    tail = "\n".join((r.stdout + r.stderr).strip().splitlines()[-15:])
    return r.returncode, tail


def test_every_mutant_fails_a_pin(tmp_path):
    with open(SRC) as f:
        original = f.read()
    jobs = [("unchanged", original)] + [(name, _mutate(original, edits)) for name, edits in MUTANTS]
    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=workers) as pool:
        results = dict(zip([n for n, _ in jobs],
                           pool.map(lambda job: _run_pins(job[0], job[1], str(tmp_path)), jobs)))
    code, tail = results.pop("unchanged")
    assert code == 0, "the unchanged oracle must pass its pins:\n" + tail
    survivors = {name: tail for name, (code, tail) in results.items() if code != 1}
    assert not survivors, "mutants no pin caught (or that broke the run):\n" + "\n\n".join(
        "%s:\n%s" % item for item in survivors.items())


def test_mutant_names_are_unique():
    names = [name for name, _ in MUTANTS]
    assert len(names) == len(set(names))
