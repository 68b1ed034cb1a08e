"""The oracle's pins catch planted mistakes.

Each case below plants one plausible mistake in a copy of oracle/lean_oracle.c
(a swapped nibble order, a wrong offset or sign, a wrong Q6_K bit or sub-scale
index, a wrong binary16 exponent, a dropped term, a transposed operand, a
wrong rounding rule in the quantizer ...), compiles the copy, routes the
oracle module to it and runs the pins of test_oracle_pins.py and
test_oracle_quant_pins.py.  Every mistake must make at least one pin fail; the
unmodified source, compiled the same way, must pass them all.  CPU only.
"""
import numpy as np
import pytest

import oracle
import test_oracle_pins as P
import test_oracle_quant_pins as QP
import test_oracle_swiglu_pins as SP
import test_oracle_x_int8_pins as XP

Q4_0, Q8_0, I8_B64, Q6_K = oracle.Q4_0, oracle.Q8_0, oracle.I8_B64, oracle.Q6_K

# (name, text in lean_oracle.c (must occur exactly once), replacement)
MUTANTS = [
    ("q4_0 nibble order swapped",
     "int q = (j < 16) ? (qs[j] & 0x0f) : (qs[j - 16] >> 4);",
     "int q = (j < 16) ? (qs[j] >> 4) : (qs[j - 16] & 0x0f);"),
    ("q4_0 offset sign",
     "return d * (double)(q - 8);",
     "return d * (double)(8 - q);"),
    ("q4_0 offset off by one",
     "return d * (double)(q - 8);",
     "return d * (double)(q - 7);"),
    ("int8 read unsigned",
     "int q = (int)(int8_t)blk[2 + j];",
     "int q = (int)blk[2 + j];"),
    ("q6_k low nibble from the wrong ql byte",
     "int lo = (ql[64 * h + 32 * (g % 2) + l] >> (4 * (g / 2))) & 0x0f;",
     "int lo = (ql[64 * h + 32 * (g / 2) + l] >> (4 * (g % 2))) & 0x0f;"),
    ("q6_k high bits at the wrong shift",
     "int hi = (qh[32 * h + l] >> (2 * g)) & 0x03;",
     "int hi = (qh[32 * h + l] >> g) & 0x03;"),
    ("q6_k sub-scale per 32 elements",
     "return d * (double)sc[j / 16] * (double)(q - 32);",
     "return d * (double)sc[j / 32] * (double)(q - 32);"),
    ("q6_k offset off by one",
     "return d * (double)sc[j / 16] * (double)(q - 32);",
     "return d * (double)sc[j / 16] * (double)(q - 31);"),
    ("q6_k halves swapped",
     "int h = j / 128;          /* which half of the super-block      */",
     "int h = 1 - j / 128;      /* which half of the super-block      */"),
    ("fp16 exponent bias",
     "v = ldexp((double)(1024 + f), e - 25);",
     "v = ldexp((double)(1024 + f), e - 24);"),
    ("fp16 subnormal scale",
     "v = ldexp((double)f, -24);",
     "v = ldexp((double)f, -25);"),
    ("fp16 sign dropped",
     "return sign ? -v : v;",
     "return v;"),
    ("accumulation drops the running sum",
     "double p = w[k] * (double)xm[k];\n                acc += p;\n",
     "double p = w[k] * (double)xm[k];\n                acc = p;\n"),
    ("accumulation in fp32",
     "double p = w[k] * (double)xm[k];\n                acc += p;\n",
     "double p = w[k] * (double)xm[k];\n                acc = (double)((float)acc + (float)p);\n"),
    ("bound without the absolute value",
     "acc += p;\n                mag += fabs(p);\n            }\n            j->y",
     "acc += p;\n                mag += p;\n            }\n            j->y"),
    ("x read transposed",
     "const float *xm = j->x + m * j->K;",
     "const float *xm = j->x + m;"),
    ("block stride wrong",
     "w[k] = block_value(fmt, row + (k / be) * bb, (int)(k % be));",
     "w[k] = block_value(fmt, row + (k / be) * be, (int)(k % be));"),
    # the quantizers
    ("quantizer: ties to even",
     "if (a - f >= 0.5) f += 1.0;",
     "if (a - f > 0.5 || (a - f == 0.5 && fmod(f, 2.0) == 1.0)) f += 1.0;"),
    ("quantizer: q8 divides by the unrounded scale",
     "q = round_half_away((double)w[j] / d);\n                if (q < -127.0) q = -127.0;",
     "q = round_half_away((double)w[j] / (amax / 127.0));\n                if (q < -127.0) q = -127.0;"),
    ("quantizer: /128",
     "double_to_fp16_bits(amax / 127.0, &dbits)",
     "double_to_fp16_bits(amax / 128.0, &dbits)"),
    ("quantizer: q4_0 scale sign",
     "double_to_fp16_bits(m / -8.0, &dbits)",
     "double_to_fp16_bits(m / 8.0, &dbits)"),
    ("quantizer: q4_0 nibbles swapped",
     "if (j < 16) blk[2 + j] |= (uint8_t)qi;\n            else blk[2 + j - 16] |= (uint8_t)(qi << 4);",
     "if (j < 16) blk[2 + j] |= (uint8_t)(qi << 4);\n            else blk[2 + j - 16] |= (uint8_t)qi;"),
    ("quantizer: binary16 ties away from zero",
     "if (rest > 0.5 || (rest == 0.5 && fmod(kf, 2.0) == 1.0)) kf += 1.0;",
     "if (rest >= 0.5) kf += 1.0;"),
    ("quantizer: clamps at -128",
     "if (q < -127.0) q = -127.0;",
     "if (q < -128.0) q = -128.0;"),
    # the activation quantization (x to int8)
    ("x int8: ties to even",
     "float r = roundf(t);              /* ties away from zero */",
     "float r = rintf(t);"),
    ("x int8: scale /128",
     "volatile float s = amax / 127.0f;",
     "volatile float s = amax / 128.0f;"),
    ("x int8: scale of the wrong block",
     "double xt = (double)sc[m * (K / 32) + k / 32] * (double)xq[m * K + k];",
     "double xt = (double)sc[m * (K / 32) + k / 64] * (double)xq[m * K + k];"),
    # the gated FFN input
    ("silu: sign of the exponent",
     "return t / (1.0 + exp(-t));",
     "return t / (1.0 + exp(t));"),
    ("swiglu: gate and up swapped in the epilogue",
     "h[n] = oracle_silu(g[n]) * u[n];",
     "h[n] = oracle_silu(u[n]) * g[n];"),
    ("x int8: unquantized x in the product",
     "double xt = (double)sc[m * (K / 32) + k / 32] * (double)xq[m * K + k];",
     "double xt = (double)x[m * K + k];"),
]

# The pins, with the arguments of one case each (the cheap ones).
PINS = [
    (P.test_fp16_decode_exhaustive, {}),
    (P.test_fp16_subnormal_and_extremes, {}),
    (P.test_q4_0_all_nine_times_ones_is_K_d, {"K": 96}),
    (P.test_q4_0_per_block_scales_and_offsets, {}),
    (P.test_int8_closed_forms, {"fmt": Q8_0, "be": 32}),
    (P.test_int8_closed_forms, {"fmt": I8_B64, "be": 64}),
    (P.test_q6_k_closed_forms, {}),
    (P.test_q4_0_element_order, {}),
    (P.test_int8_element_order, {"fmt": Q8_0, "be": 32}),
    (P.test_q6_k_element_order, {}),
    (P.test_q6_k_single_element_positions, {}),
    (P.test_exact_integer_product_vs_numpy, {"fmt": Q4_0}),
    (P.test_exact_integer_product_vs_numpy, {"fmt": Q8_0}),
    (P.test_exact_integer_product_vs_numpy, {"fmt": Q6_K}),
    (P.test_brute_force_tiny, {"fmt": Q4_0}),
    (P.test_power_of_two_scaling_exact, {"fmt": Q4_0}),
    (P.test_q8_sign_flip_negates, {}),
    (QP.test_fp16_rounding_matches_numpy, {}),
    (QP.test_q8_hand_worked_block, {}),
    (QP.test_q4_0_hand_worked_blocks, {}),
    (QP.test_zero_block_and_tiny_scales, {}),
    (QP.test_rejects, {}),
    (QP.test_each_code_is_the_nearest, {"fmt": Q4_0, "be": 32}),
    (QP.test_each_code_is_the_nearest, {"fmt": Q8_0, "be": 32}),
    (QP.test_round_trip_error_bound, {"fmt": I8_B64, "be": 64}),
    (SP.test_silu_closed_forms, {}),
    (SP.test_swiglu_hand_built_blocks, {}),
    (XP.test_exact_multiples_reduce_to_the_fp32_product, {"fmt": Q8_0}),
    (XP.test_codes_within_half_a_step, {}),
    (XP.test_ties_go_away_from_zero, {}),
    (XP.test_zero_block_and_scaling_and_sign, {}),
    (XP.test_within_the_quantization_bound_of_the_exact_product, {"fmt": Q4_0}),
]


def failing_pins(lib):
    """Names of the pins that fail with the oracle routed to `lib`."""
    failed = []
    with oracle.using(lib):
        for fn, kw in PINS:
            try:
                fn(**kw)
            except (Exception, pytest.fail.Exception):  # an assertion, a failed
                failed.append(fn.__name__)                   # pytest.raises, an error
    return failed


def test_unmodified_source_passes_every_pin(tmp_path):
    lib = oracle.load_library(oracle.build_variant(oracle.source(), tmp_path / "same.so"))
    assert failing_pins(lib) == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = oracle.source()
    assert src.count(old) == 1, "mutation site not found uniquely: %r" % old
    lib = oracle.load_library(oracle.build_variant(src.replace(old, new), tmp_path / "m.so"))
    assert failing_pins(lib), "no pin caught: " + name
    # the real oracle is back in place afterwards
    assert oracle.fp16_to_double(0x3C00) == 1.0 and np.isfinite(oracle.fp16_to_double(0x7BFF))
