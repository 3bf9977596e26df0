"""Plant plausible mistakes in a copy of the oracle source, on the CPU, and
check that at least one pin fails for each: the pins discriminate."""
import pytest

import oracle as oracle_mod
from oracle_pins import ALL_PINS

# (name, exact text in na_oracle.c, replacement, occurrences to replace)
MUTANTS = [
    ("rotation_sign", "x[i] = (x0 * c - x1 * s) * scale;", "x[i] = (x0 * c + x1 * s) * scale;", 1),
    ("cos_sin_swapped", "double c = cos(angle), s = sin(angle);",
     "double c = sin(angle), s = cos(angle);", 1),
    ("interleaved_pairing", "double x0 = x[i], x1 = x[i + half];",
     "double x0 = x[i], x1 = x[(i ^ 1) % (2 * half)];", 1),
    ("frequency_exponent_dropped_2", "inv_freq[i] = 1.0 / pow(base, 2.0 * (double)i / (double)rd);",
     "inv_freq[i] = 1.0 / pow(base, (double)i / (double)rd);", 1),
    ("yarn_mix_swapped", "inv_freq[i] = interp * (1.0 - extrapolation) + extrap * extrapolation;",
     "inv_freq[i] = extrap * (1.0 - extrapolation) + interp * extrapolation;", 1),
    ("yarn_low_ceil", "double lo = floor(", "double lo = ceil(", 1),
    ("yarn_factor_multiplies", "double interp = extrap / factor;", "double interp = extrap * factor;", 1),
    ("causal_excludes_self", "capacity, d), pos + 1,\n", "capacity, d), pos,\n", 1),
    ("gqa_modulo_mapping", "int kvh = h / group;", "int kvh = h % KV;", 2),
    ("softmax_unnormalised", "double p = scores[j] / sum;", "double p = scores[j];", 1),
    ("score_scale_dropped", "        s *= scale;\n", "", 1),
    ("rms_sum_not_mean", "double inv = 1.0 / sqrt(ss / (double)d + eps);\n    for (int i = 0; i < d; i++)\n        x[i] = x[i] * inv",
     "double inv = 1.0 / sqrt(ss + eps);\n    for (int i = 0; i < d; i++)\n        x[i] = x[i] * inv", 1),
    ("vnorm_eps_dropped", "double inv = 1.0 / sqrt(ss / (double)d + eps);\n    for (int i = 0; i < d; i++)\n        x[i] *= inv;",
     "double inv = 1.0 / sqrt(ss / (double)d);\n    for (int i = 0; i < d; i++)\n        x[i] *= inv;", 1),
    ("zero_centred_swapped", "(zero_centered ? 1.0 + w[i] : w[i])", "(zero_centered ? w[i] : 1.0 + w[i])", 1),
    ("gate_sign", "o[i] *= 1.0 / (1.0 + exp(-g[i]));", "o[i] *= 1.0 / (1.0 + exp(g[i]));", 1),
    ("position_ignores_prior", "int pos = cache_lens[b] + (t - cu_seqlens[b]);\n            if (pos < 0 ||",
     "int pos = (t - cu_seqlens[b]);\n            if (pos < 0 ||", 1),
    ("rope_scale_ignored", "x[i + half] = (x0 * s + x1 * c) * scale;", "x[i + half] = (x0 * s + x1 * c);", 1),
    ("k_not_normed", "oracle_rmsnorm_head(kx, k_norm_w, d, eps, zc);", "(void)zc;", 1),
    ("v_norm_on_k", "oracle_vnorm_head(vx, d, eps);", "oracle_vnorm_head(kx, d, eps);", 1),
    ("probs_before_shift_lost", "scores[j] = exp(scores[j] - m);", "scores[j] = exp(scores[j] - m) + 1e-3;", 1),
    ("importance_mean_not_sum", "*dst = accumulate ? *dst + s : s;", "*dst = accumulate ? *dst + s / H : s / H;", 1),
    ("importance_first_head_only", "for (int h = 0; h < H; h++)\n                s += probs[", "for (int h = 0; h < 1; h++)\n                s += probs[", 1),
    ("softcap_missing_divide", "s = softcap * tanh(s / softcap);", "s = softcap * tanh(s);", 1),
    ("decode_window_off_by_one", "window > 0 ? n - window : 0", "window > 0 ? n - window + 1 : 0", 1),
    ("prefill_window_off_by_one", "window > 0 ? pos + 1 - window : 0", "window > 0 ? pos - window : 0", 1),
    ("importance_overwrites", "*dst = accumulate ? *dst + s : s;", "*dst = s;", 1),
    ("yarn_attn_factor_log10", "return 0.1 * log(factor) + 1.0;", "return 0.1 * log10(factor) + 1.0;", 1),
    ("yarn_attn_factor_one_dropped", "return 0.1 * log(factor) + 1.0;", "return 0.1 * log(factor);", 1),
    ("yarn_attn_factor_always_default", "if (attn_factor > 0.0)\n        return attn_factor;",
     "if (attn_factor > 0.0)\n        return 1.0;", 1),
    ("ring_slot_off_by_one", "return (int)(pos % (int64_t)capacity);",
     "return (int)((pos + 1) % (int64_t)capacity);", 1),
    ("ring_capacity_check_ignores_chunk", "(int64_t)capacity < (int64_t)window + (last - pos)",
     "(int64_t)capacity < (int64_t)window", 1),
]


def _source():
    with open(oracle_mod.SOURCE) as fh:
        return fh.read()


@pytest.mark.parametrize("name,old,new,count", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new, count):
    src = _source()
    assert src.count(old) == count, f"anchor for {name} occurs {src.count(old)} times"
    mutant = oracle_mod.build_variant(src.replace(old, new), name)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
