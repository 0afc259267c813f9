"""Planted mistakes in the oracle must be caught by its pins.

Each case copies the oracle's C source, makes one plausible mistake in it (a
wrong exponent bias, ties away from zero, a dropped rank, a wrong scale index,
a missing absolute value, ...), builds the copy and runs the pins against it:
at least one pin has to fail. The real oracle is untouched.
"""
import os

import pytest

import oracle as orc
from oracle import build as obuild
from oracle_pins import PINS

MUTANTS = [
    ("decode_bias", "ldexp((double)(8 + m), e - 10)", "ldexp((double)(8 + m), e - 9)"),
    ("ties_away", "m = nearbyint(ldexp(a, 3 - e));", "m = round(ldexp(a, 3 - e));"),
    ("sub_ties_away", "m = nearbyint(a * 0x1p9);", "m = round(a * 0x1p9);"),
    ("sat_to_nan", "return sign | 0x7E;", "return 0x7F;"),
    ("sub_scale", "m = nearbyint(a * 0x1p9);", "m = nearbyint(a * 0x1p8);"),
    ("max_240", "return fmt == ORC_E5M2 ? 57344.0f : 448.0f;",
     "return fmt == ORC_E5M2 ? 57344.0f : 240.0f;"),
    ("divide_not_reciprocal", "float y = v[i] * inv;", "float y = v[i] / s;"),
    ("degenerate_sign", "codes[i] = signbit(v[i]) ? 0x80 : 0x00;", "codes[i] = 0x00;"),
    ("no_fabs", "amax = fmaxf(amax, fabsf(v[i]));", "amax = fmaxf(amax, v[i]);"),
    ("scale_index", "float s = scales[i / (size_t)block];", "float s = scales[(i + 1) / (size_t)block];"),
    ("drop_last_rank",
     "        for (r = 1; r < nranks; r++)\n            sum = sum + dequant_elem(codes[r], scales[r], block, i);",
     "        for (r = 1; r < nranks - 1; r++)\n            sum = sum + dequant_elem(codes[r], scales[r], block, i);"),
    ("zero_start",
     "        float sum = dequant_elem(codes[0], scales[0], block, i);",
     "        float sum = 0.0f + dequant_elem(codes[0], scales[0], block, i);"),
    ("reverse_order_exact",
     "                float sum = load_elem(in[0], dtype, i);\n                for (r = 1; r < nranks; r++)\n                    sum = sum + load_elem(in[r], dtype, i);\n                store_elem(out[dst], dtype, i, sum);",
     "                float sum = load_elem(in[nranks - 1], dtype, i);\n                for (r = nranks - 2; r >= 0; r--)\n                    sum = sum + load_elem(in[r], dtype, i);\n                store_elem(out[dst], dtype, i, sum);"),
    ("bf16_truncate", "u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0;"),
    ("bf16_ties_up", "u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0x8000u;"),
    ("tree_no_requant",
     "                       dequant_elem(shard_codes, shard_scales, block, i));",
     "                       reduced[i]);"),
    ("tail_block_dropped",
     "    float buf[128];\n    size_t b, nb, lo, len, i;\n    if (check_dtype(dtype) || check_block(block))\n        return check_dtype(dtype) ? ORC_ERR_ARG : ORC_ERR_UNSUPPORTED;\n    nb = (n + (size_t)block - 1) / (size_t)block;",
     "    float buf[128];\n    size_t b, nb, lo, len, i;\n    if (check_dtype(dtype) || check_block(block))\n        return check_dtype(dtype) ? ORC_ERR_ARG : ORC_ERR_UNSUPPORTED;\n    nb = n / (size_t)block;"),
    ("shard_len_unrounded",
     "        per = (per + (size_t)block - 1) / (size_t)block * (size_t)block;",
     "        per = per;"),
    ("subnormal_sign_lost",
     "         * code (exponent 1, mantissa 0) is also 8. */\n        m = nearbyint(a * 0x1p9);\n        return sign | (uint8_t)m;",
     "         * code (exponent 1, mantissa 0) is also 8. */\n        m = nearbyint(a * 0x1p9);\n        return (uint8_t)m;"),
    ("rs_wrong_offset", "            store_elem(out[owner], dtype, i - lo, sum);",
     "            store_elem(out[owner], dtype, i - lo + (owner > 0), sum);"),
    ("ag_own_contribution",
     "                float v = block ? dequant_elem(wire_codes[r], wire_scales[r], block, i)\n                                : load_elem(in[r], dtype, i);",
     "                float v = block ? dequant_elem(wire_codes[dst], wire_scales[dst], block, i)\n                                : load_elem(in[dst], dtype, i);"),
    ("a2a_transposed",
     "                store_elem(out[j], dtype, (size_t)r * c + i, v);",
     "                store_elem(out[r], dtype, (size_t)j * c + i, v);"),
    ("e5m2_bias", "ldexp((double)(4 + m), e - 17)", "ldexp((double)(4 + m), e - 16)"),
    ("e5m2_max", "return fmt == ORC_E5M2 ? 57344.0f : 448.0f;",
     "return fmt == ORC_E5M2 ? 49152.0f : 448.0f;"),
    ("e5m2_ties_away", "m = nearbyint(ldexp(a, 2 - e));", "m = round(ldexp(a, 2 - e));"),
    ("e5m2_inf_as_nan", "        return m ? NAN : (sign ? -INFINITY : INFINITY);",
     "        return NAN;"),
    ("e5m2_saturates_to_inf", "        return sign | 0x7B;", "        return sign | 0x7C;"),
    ("variant_block_fixed", "        len = (n - lo < (size_t)block) ? n - lo : (size_t)block;\n        for (i = 0; i < len; i++)\n            buf[i] = load_elem(in, dtype, lo + i);\n        scales[b] = quantize_block_fmt(buf, len, codes + lo, fmt);",
     "        len = (n - lo < (size_t)block) ? n - lo : (size_t)block;\n        for (i = 0; i < len; i++)\n            buf[i] = load_elem(in, dtype, lo + i);\n        scales[b] = quantize_block_fmt(buf, len, codes + lo, block == 256 ? 0 : fmt);"),
    ("fmt_reduce_drop_last_rank",
     "        for (r = 1; r < nranks; r++)\n            sum = sum + dequant_elem_fmt(codes[r], scales[r], block, i, fmt);",
     "        for (r = 1; r < nranks - 1; r++)\n            sum = sum + dequant_elem_fmt(codes[r], scales[r], block, i, fmt);"),
    ("fmt_reduce_reversed",
     "        float sum = dequant_elem_fmt(codes[0], scales[0], block, i, fmt);\n        for (r = 1; r < nranks; r++)\n            sum = sum + dequant_elem_fmt(codes[r], scales[r], block, i, fmt);",
     "        float sum = dequant_elem_fmt(codes[nranks - 1], scales[nranks - 1], block, i, fmt);\n        for (r = nranks - 2; r >= 0; r--)\n            sum = sum + dequant_elem_fmt(codes[r], scales[r], block, i, fmt);"),
    ("tree_requant_bf16_sum",
     "                sum = sum + dequant_elem(wire_codes[r], wire_scales[r], block, i);\n            reduced[i] = sum;",
     "                sum = sum + dequant_elem(wire_codes[r], wire_scales[r], block, i);\n            reduced[i] = dtype == ORC_BF16 ? orc_bf16_to_f32(orc_f32_to_bf16(sum)) : sum;"),
    ("a2a_global_blocks",
     "                st = orc_quantize(elem_ptr(in[r], dtype, (size_t)j * c), dtype, c, block,\n                                  wire_codes[r] + (size_t)j * c,\n                                  wire_scales[r] + (size_t)j * nbc);",
     "                st = j ? 0 : orc_quantize(in[r], dtype, c * (size_t)nranks, block,\n                                          wire_codes[r], wire_scales[r]);"),
]


@pytest.fixture(scope="module")
def source():
    with open(obuild.SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, source, name, old, new):
    assert source.count(old) == 1, "mutation site not found exactly once: %s" % name
    path = obuild.build_source(source.replace(old, new),
                               os.path.join(str(tmp_path), "mutant_%s.so" % name))
    caught = []
    with orc.using(path):
        for pin in PINS:
            try:
                pin(orc)
            except (AssertionError, ValueError) as e:
                caught.append((pin.__name__, repr(e)[:120]))
                break
    assert caught, "no pin caught the planted mistake %r" % name
