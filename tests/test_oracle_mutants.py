"""Every plausible mistake planted in the oracle must fail at least one pin.

Each mutant is a copy of oracle/fia_oracle.c with one textual change (a dropped
term, a wrong sign, a wrong index, a swapped operand), compiled on the CPU and
run through every pin in oracle_pins.  A mutant that passes all pins would show
that the pins do not constrain that part of the oracle.
"""
import os

import pytest

import oracle
import oracle_pins

MUTANTS = [
    ("gqa_mapping", "const int hk = h / G;                               /* R1 */",
     "const int hk = h % Nkv;"),
    ("dropped_scale", "s[t] = scale * dot;", "s[t] = dot;"),
    ("sink_missing_from_sum", "        l += exp(*sink - m);", "        l += 0.0;"),
    ("sink_missing_from_max", "    if (sink && *sink > m)\n        m = *sink;", "    if (0)\n        m = *sink;"),
    ("unnormalised_out", "out[d] = acc / l;", "out[d] = acc;"),
    ("rau_prev_sum_dropped", "prev_sum[r] * exp(mp - m)", "exp(mp - m)"),
    ("rau_cur_sum_dropped", "cur_sum[r] * exp(mc - m)", "exp(mc - m)"),
    ("rau_max_prev_only", "const double m = mp > mc ? mp : mc;", "const double m = mp;"),
    ("dequant_offset_sign", "float centred = xf - offset;", "float centred = xf + offset;"),
    ("dequant_k_uses_v_scale", "aq_scale[(0 * Nkv + hk) * D + d]", "aq_scale[(1 * Nkv + hk) * D + d]"),
    ("dequant_v_uses_k_offset", "aq_offset[(1 * Nkv + hk) * D + d]", "aq_offset[(0 * Nkv + hk) * D + d]"),
    ("block_row_off_by_one", "t % block_size) * D;", "(t + 1) % block_size) * D;"),
    ("causal_off_by_one", "const int64_t last = qi + (Lkv - Lq);", "const int64_t last = qi + (Lkv - Lq) - 1;"),
    ("causal_left_up", "const int64_t last = qi + (Lkv - Lq);", "const int64_t last = qi;"),
    ("f16_exponent_bias", "expo - 25", "expo - 24"),
    ("f16_subnormal", "ldexp((double)frac, -24)", "ldexp((double)frac, -25)"),
    ("empty_row_max", "*smax = -INFINITY;\n        *ssum = 0.0;\n        return;",
     "*smax = 0.0;\n        *ssum = 0.0;\n        return;"),
    ("gather_in_block_row", "const int64_t in_block = t - logical * block_size;",
     "const int64_t in_block = (t + 1) % block_size;"),
    ("dequant_array_offset_ignored", "out[i] = oracle_dequant_i8(x[i], offset[i], scale[i]);",
     "out[i] = oracle_dequant_i8(x[i], 0.0f, scale[i]);"),
    ("mask_ignored", "if (mask && mask[(int64_t)b * mask_stride + t] != 0)",
     "if (0 && mask && mask[(int64_t)b * mask_stride + t] != 0)"),
    ("mask_polarity", "mask[(int64_t)b * mask_stride + t] != 0)", "mask[(int64_t)b * mask_stride + t] == 0)"),
    ("mask_batch_row", "mask[(int64_t)b * mask_stride + t]", "mask[t]"),
    ("decode_band_lower_off_by_one", "if (t < qp - pre_tokens ||", "if (t <= qp - pre_tokens ||"),
    ("decode_band_upper_ignored", "|| t > qp + next_tokens)", "|| t > qp + 1000000)"),
    ("decode_positions_off_by_one", "const int64_t qp = L - q_len + pos;", "const int64_t qp = L - q_len + pos + 1;"),
    ("decode_positions_all_last", "const int64_t qp = L - q_len + pos;", "const int64_t qp = L - 1;"),
    ("decode_positions_batch_index", "const int b = (int)(bi / q_len), h = (int)(r % Nq);",
     "const int b = (int)(bi % q_len), h = (int)(r % Nq);"),
    ("post_quant_ties_away", "double q = nearbyint(v);", "double q = round(v);"),
    ("post_quant_truncates", "double q = nearbyint(v);", "double q = trunc(v);"),
    ("post_quant_no_upper_saturation", "if (q > 127.0)\n                q = 127.0;",
     "if (q > 255.0)\n                q = 127.0;"),
    ("post_quant_low_clamp", "q = -128.0;", "q = -127.0;"),
    ("post_quant_channel_by_row", "const int64_t pc = per_channel ? c : 0;",
     "const int64_t pc = per_channel ? r : 0;"),
    ("post_quant_offset_sign", "x[i] * (double)scale2[pc] + (offset2", "x[i] * (double)scale2[pc] - (offset2"),
    ("band_lower_off_by_one", "int64_t lo = qi + (Lkv - Lq) - pre_tokens,", "int64_t lo = qi + (Lkv - Lq) - pre_tokens + 1,"),
    ("band_not_shifted", "int64_t lo = qi + (Lkv - Lq) - pre_tokens, hi = qi + (Lkv - Lq) + next_tokens;",
     "int64_t lo = qi - pre_tokens, hi = qi + next_tokens;"),
    ("band_next_ignored", "hi = qi + (Lkv - Lq) + next_tokens;", "hi = qi + (Lkv - Lq);"),
    ("band_first_key_dropped", "((cu_kv[b] + first + j) * Nkv + hk) * D + d", "((cu_kv[b] + j) * Nkv + hk) * D + d"),
    ("prefill_kv_head_index", "const int64_t src = ((cu_kv[b] + first + j) * Nkv + hk) * D + d;",
     "const int64_t src = ((cu_kv[b] + first + j) * Nkv + (h % Nkv)) * D + d;"),
]


def _failures(O):
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(O)
        except Exception:  # an assertion or a rejected call: the pin caught it
            failed.append(pin.__name__)
    return failed


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(oracle.SOURCE).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    path = os.path.join(tmp_path, f"mutant_{name}.c")
    with open(path, "w") as f:
        f.write(mutated)
    lib = oracle.compile_source(path, os.path.join(tmp_path, f"libmutant_{name}.so"))
    failed = _failures(oracle.Oracle(lib))
    assert failed, f"mutant {name} passed every pin"


def test_unmutated_oracle_passes_every_pin():
    assert _failures(oracle.default()) == []
