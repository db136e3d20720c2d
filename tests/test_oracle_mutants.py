"""Planted mistakes: each mutant is a copy of the oracle's C source with one
plausible error (a wrong rounding mode, swapped nibbles, a dropped clamp, a
wrong divisor, an off-by-one offset, a reversed operand, a truncating
conversion, a wrong exponent bias, a wrong group stride, a transposed scale
store, a scale taken from the wrong group; for the asymmetric quantizer a
range that leaves out 0, a wrong divisor, a wrong-signed or truncated zero
point, the symmetric +8 offset, zero points ignored by the dequantizer; for the
fp16 dequantized weight a swapped zero point, a truncating rounding, a scale
of the wrong group, a wrong offset).  The pin suite must reject every
one of them; a mutant that passes all pins means the pins are too weak."""
from __future__ import annotations

import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "w4a16_oracle.c")

MUTANTS = {
    "round_half_away": ("float rq = nearbyintf(r);", "float rq = roundf(r);"),
    "swapped_nibbles": ("(uint8_t)((hi << 4) | lo)", "(uint8_t)((lo << 4) | hi)"),
    "dropped_clamp": ("if (s < 1e-8f)", "if (s < 0.0f)"),
    "divide_by_8": ("float s = amax / 7.0f;", "float s = amax / 8.0f;"),
    "offset_7": ("int z = zrow ? zrow[k / group] : 8;", "int z = zrow ? zrow[k / group] : 7;"),
    "reversed_x": ("acc += orc_half_to_double(x[m * K + k]) * wd[k];",
                   "acc += orc_half_to_double(x[m * K + (K - 1 - k)]) * wd[k];"),
    "truncating_f2h": ("double m = rint(ldexp(a, 10 - e)) - 1024.0;",
                       "double m = floor(ldexp(a, 10 - e)) - 1024.0;"),
    "exponent_bias": ("v = ldexp(1024.0 + (double)m, e - 25);",
                      "v = ldexp(1024.0 + (double)m, e - 24);"),
    "group_stride": ("const uint16_t *wg = W + n * K + g * group;",
                     "const uint16_t *wg = W + n * K + g;"),
    "scale_transposed": ("scales[n * ngroups + g] = quantize_group",
                         "scales[g * N + n] = quantize_group"),
    "scale_group_zero": ("out[k] = (double)(nib - z) * orc_half_to_double(srow[k / group]);",
                         "out[k] = (double)(nib - z) * orc_half_to_double(srow[0]);"),
    "amax_signed": ("float a = fabsf((float)orc_half_to_double(w16[i]));",
                    "float a = (float)orc_half_to_double(w16[i]);"),
    "asym_range_without_zero": ("float mn = 0.0f, mx = 0.0f;",
                                "float mn = INFINITY, mx = -INFINITY;"),
    "asym_divide_by_16": ("float s = (mx - mn) / 15.0f;", "float s = (mx - mn) / 16.0f;"),
    "asym_zero_sign": ("float z = -nearbyintf(mn / s);", "float z = nearbyintf(-mn / s) + 1.0f;"),
    "asym_zero_truncated": ("float z = -nearbyintf(mn / s);", "float z = -truncf(mn / s);"),
    "asym_stored_plus_8": ("(uint8_t)(((q[i + 1] & 0x0f) << 4) | (q[i] & 0x0f));",
                           "(uint8_t)((((q[i + 1] + 8) & 0x0f) << 4) | ((q[i] + 8) & 0x0f));"),
    "zeros_ignored": ("int z = zrow ? zrow[k / group] : 8;", "int z = 8;"),
    "q4_0_nibbles_swapped": ("out[n * K + b * 32 + 2 * i] = (double)((blk[2 + i] & 0x0f) - 8) * d;",
                             "out[n * K + b * 32 + 2 * i] = (double)(((blk[2 + i] >> 4) & 0x0f) - 8) * d;"),
    "q4_0_scale_big_endian": ("blk[0] = (uint8_t)(d & 0xff);        /* little-endian fp16 */",
                              "blk[0] = (uint8_t)(d >> 8);"),
    "w8_divide_by_128": ("float s = amax / 127.0f;   /* 2^(b-1) - 1 = 127 */",
                         "float s = amax / 128.0f;"),
    "w8_offset_127": ("out[k] = (double)((int)qrow[k] - 128) * s;",
                      "out[k] = (double)((int)qrow[k] - 127) * s;"),
    "awq_alpha_by_row": ("(float)orc_half_to_double(alpha[k]);", "(float)orc_half_to_double(alpha[m]);"),
    "f16_dequant_zero_swapped": ("float v = (float)(nib - z) * s;", "float v = (float)(z - nib) * s;"),
    "f16_dequant_truncating": ("out[n * K + k] = orc_float_to_half(v);",
                               "out[n * K + k] = orc_float_to_half(v * (1.0f - 1.0f / 4096.0f));"),
    "f16_dequant_scale_group_zero": ("float s = (float)orc_half_to_double(scales[n * (K / group) + k / group]);",
                                     "float s = (float)orc_half_to_double(scales[n * (K / group)]);"),
    "f16_dequant_offset_7": ("int z = zeros ? zeros[n * (K / group) + k / group] : 8;",
                             "int z = zeros ? zeros[n * (K / group) + k / group] : 7;"),
    "awq_truncating": ("out[m * K + k] = orc_float_to_half(p);",
                       "out[m * K + k] = orc_float_to_half(p * (1.0f - 1.0f / 4096.0f));"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    with open(SRC, encoding="utf-8") as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutant_src = tmp_path / f"oracle_{name}.c"
    mutant_src.write_text(src.replace(old, new), encoding="utf-8")
    lib = oracle.build(str(mutant_src), out=str(tmp_path / f"liboracle_{name}.so"))
    orc = oracle.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
