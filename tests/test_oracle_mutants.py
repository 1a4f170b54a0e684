"""Plant one plausible mistake at a time in a copy of the oracle (on the CPU)
and check that some pin rejects it -- evidence that the pins would notice a
dropped term, a wrong sign or index, a swapped operand or a wrong rounding."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import oracle  # noqa: E402
from oracle_pins import ALL_PINS  # noqa: E402

MUTANTS = [
    ("nibble_order_decode", "int lo = blk[2 + j] & 0x0f, hi = blk[2 + j] >> 4;\n                out",
     "int hi = blk[2 + j] & 0x0f, lo = blk[2 + j] >> 4;\n                out"),
    ("nibble_order_encode", "blk[2 + j] = (uint8_t)(q[j] | (q[j + 16] << 4));",
     "blk[2 + j] = (uint8_t)(q[j + 16] | (q[j] << 4));"),
    ("round_half_even", "roundf(x[i] / d)", "nearbyintf(x[i] / d)"),
    ("divide_by_fp32_scale_q8_0", "float q = (d == 0.0f) ? 0.0f : clampf(roundf(x[i] / d), -127.0f, 127.0f);\n        blk[2 + i]",
     "float q = (d == 0.0f) ? 0.0f : clampf(roundf(x[i] / (amax / 127.0f)), -127.0f, 127.0f);\n        blk[2 + i]"),
    ("q4_0_dropped_offset", "out[b * QK + j] = (double)(lo - 8) * d;", "out[b * QK + j] = (double)lo * d;"),
    ("q4_0_scale_sign", "m / -8.0f", "m / 8.0f"),
    ("q4_0_tie_last", "if (fabsf(x[i]) > fabsf(m)) m = x[i];", "if (fabsf(x[i]) >= fabsf(m)) m = x[i];"),
    ("fp16_exponent_off_by_one", "ldexp((double)(m + 1024), e - 25)", "ldexp((double)(m + 1024), e - 24)"),
    ("fp16_round_truncate", "double n = nearbyint(ldexp(a, -ulp_exp));", "double n = floor(ldexp(a, -ulp_exp));"),
    ("q8_1_sum_without_scale", "ref_fp16_from_float(d * (float)sum)", "ref_fp16_from_float((float)sum)"),
    ("gemv_selected_row_index", "decode_row(wfmt, W + n * wrb, K, w);\n        for (int64_t m = 0; m < M; m++) {\n            double s = 0.0, a = 0.0;",
     "decode_row(wfmt, W + j * wrb, K, w);\n        for (int64_t m = 0; m < M; m++) {\n            double s = 0.0, a = 0.0;"),
    ("gemv_x_row_transposed", "const double *x = xd + m * K;", "const double *x = xd + (M - 1 - m) * K;"),
    ("abs_sum_signed", "a += fabs(w[k] * x[k]);", "a += w[k] * x[k];"),
    ("block_dots_no_offset", "s += (int64_t)(lo - 8) * (int8_t)xb[4 + j];", "s += (int64_t)lo * (int8_t)xb[4 + j];"),
    ("swiglu_sign", "h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];", "h[i] = g[i] / (1.0 + exp(g[i])) * u[i];"),
    ("repack_codes_offset", "memcpy(tile + 16 * s, blk + 2, 16);\n                memcpy(tile + 512 + 2 * s, blk, 2);",
     "memcpy(tile + 16 * s, blk, 16);\n                memcpy(tile + 512 + 2 * s, blk, 2);"),
    ("bf16_decode_shift", "uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    ("rmsnorm_sum_not_mean", "sqrt(s / (double)K + (double)eps)", "sqrt(s + (double)eps)"),
    ("rmsnorm_eps_outside_root", "sqrt(s / (double)K + (double)eps)", "sqrt(s / (double)K) + (double)eps"),
    ("rmsnorm_gamma_ignored", "if (gamma) v = v * gamma[k];", "if (gamma) v = v;"),
    ("q8_0_scale_over_128", "amax / 127.0f);\n    float d = fp16_to_float(dh);\n    wr_u16(blk, dh);",
     "amax / 128.0f);\n    float d = fp16_to_float(dh);\n    wr_u16(blk, dh);"),
    ("q8_1_scale_over_128", "amax / 127.0f);\n    float d = fp16_to_float(dh);\n    int sum = 0;",
     "amax / 128.0f);\n    float d = fp16_to_float(dh);\n    int sum = 0;"),
    ("q8_0_codes_read_unsigned", "out[b * QK + i] = (double)(int8_t)blk[2 + i] * d;",
     "out[b * QK + i] = (double)blk[2 + i] * d;"),
    ("q8_0_dequant_unscaled", "out[b * QK + i] = (double)(int8_t)blk[2 + i] * d;",
     "out[b * QK + i] = (double)(int8_t)blk[2 + i];"),
    ("q8_1_dequant_uses_s", "double d = ref_fp16_to_double(rd_u16(blk));\n            for (int i = 0; i < QK; i++) out[b * QK + i] = (double)(int8_t)blk[4 + i] * d;",
     "double d = ref_fp16_to_double(rd_u16(blk + 2));\n            for (int i = 0; i < QK; i++) out[b * QK + i] = (double)(int8_t)blk[4 + i] * d;"),
    ("q4_0_clamp_at_16", "clampf(roundf(x[i] / d) + 8.0f, 0.0f, 15.0f)", "clampf(roundf(x[i] / d) + 8.0f, 0.0f, 16.0f)"),
    ("block_dots_x_unsigned", "s += (int64_t)(lo - 8) * (int8_t)xb[4 + j];", "s += (int64_t)(lo - 8) * xb[4 + j];"),
    ("block_dots_high_nibble_wrong_x", "s += (int64_t)(hi - 8) * (int8_t)xb[4 + j + 16];",
     "s += (int64_t)(hi - 8) * (int8_t)xb[4 + j];"),
    ("repack_q8_0_halves_swapped", "memcpy(tile + 16 * s, blk + 2, 16);\n                memcpy(tile + 512 + 16 * s, blk + 18, 16);",
     "memcpy(tile + 16 * s, blk + 18, 16);\n                memcpy(tile + 512 + 16 * s, blk + 2, 16);"),
    ("repack_q8_0_scale_stride", "memcpy(tile + 1024 + 2 * s, blk, 2);", "memcpy(tile + 1024 + s, blk, 2);"),
    ("repack_row_stride_dropped",
     "uint8_t *tile = packed + (n * T + b / 32) * tb;\n            int64_t s = b % 32;\n            if (fmt == FMT_Q4_0) {\n                const uint8_t",
     "uint8_t *tile = packed + (n + b / 32) * tb;\n            int64_t s = b % 32;\n            if (fmt == FMT_Q4_0) {\n                const uint8_t"),
    ("swiglu_u_dropped", "h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];", "h[i] = g[i] / (1.0 + exp(-g[i]));"),
    ("fp16_overflow_threshold", "if (a >= 65520.0)", "if (a > 65504.0)"),
    ("fp16_subnormal_exponent", "v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    ("fp16_ties_away", "double n = nearbyint(ldexp(a, -ulp_exp));", "double n = round(ldexp(a, -ulp_exp));"),
    ("gemv_k_shifted", "s += w[k] * x[k];", "s += w[k] * x[(k + 1) % K];"),
    ("rmsnorm_divides", "float v = xr[k] * rr;", "float v = xr[k] / rr;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_some_pin_rejects_mutant(tmp_path, name, old, new):
    src = open(oracle.SOURCE).read()
    want = 3 if name == "round_half_even" else 1     # every encoder rounds the same way
    assert src.count(old) == want, f"mutation site for {name} not found as expected"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(path), str(tmp_path / f"lib{name}.so"))
    o = oracle.Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin rejects mutant {name}"
