"""Each pin must catch a plausible slip in the oracle.

Every case below plants one mistake in a copy of oracle/moe_oracle.c on the CPU
(a dropped term, a wrong sign, index or operand, a swapped nibble or byte),
builds the copy on its own, and runs the oracle's pins (tests/test_oracle.py)
against it: the pins must fail.  A clean copy must pass them, which shows the
copy is what the pins load.  Nothing here touches the GPU or the oracle in the
tree.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle")
PINS = os.path.join(ROOT, "tests", "test_oracle.py")

# name -> (text in moe_oracle.c, replacement, which occurrence)
MUTANTS = {
    # routing: SelectedSoftmax ("New Community Model: ZONOS3-Mini (Zyphra) - #1271",
    # §Framework change)
    "bias_left_out_of_ranking": (
        "score[e] = l[e] + (bias ? (double)bias[e] : 0.0);", "score[e] = l[e];", 0),
    "softmax_of_biased_scores": (
        "/* 4. weights: softmax", "l = score; /* 4. weights: softmax", 0),
    "ties_to_higher_index": ("score[e] > score[best]", "score[e] >= score[best]", 0),
    "ranked_ascending": ("score[e] > score[best]", "score[e] < score[best]", 0),
    "softmax_denominator_skips_first": (
        "for (int j = 0; j < k; ++j) den += exp(", "for (int j = 1; j < k; ++j) den += exp(", 0),
    "margin_sign_flipped": ("margin[t] = kth - next;", "margin[t] = next - kth;", 0),
    # the set-weights helper (softmax of a given set's logits), a second copy
    # of step 4 that the near-tie re-evaluation uses
    "set_weights_denominator_skips_first": (
        "for (int j = 0; j < k; ++j) den += exp(", "for (int j = 1; j < k; ++j) den += exp(", 1),
    "set_weights_all_from_first_slot": (
        "topk_w[(size_t)t * k + j] = exp(l[topk_idx[(size_t)t * k + j]] - m) / den;\n    }\n    return 0;",
        "topk_w[(size_t)t * k + j] = exp(l[topk_idx[(size_t)t * k]] - m) / den;\n    }\n    return 0;", 0),
    # router projection
    "router_row_off_by_one": (
        "decode_row(c->w_r, c->x_dt, (size_t)e, c->d, wr);",
        "decode_row(c->w_r, c->x_dt, (size_t)((e + 1) % c->E), c->d, wr);", 0),
    # other scoring modes (same section: activation before ranking)
    "softmax_mode_uses_sigmoid": ("if (mode == 1) {", "if (mode == 3) {", 0),
    "sigmoid_sign_flipped": ("1.0 / (1.0 + exp(-l[e]))", "1.0 / (1.0 + exp(l[e]))", 0),
    "scored_modes_rank_raw_logits": (
        "score[e] = prob[e] + (bias", "score[e] = l[e] + (bias", 0),
    "scored_modes_weigh_by_biased_score": (
        "topk_w[(size_t)t * k + j] = prob[best];", "topk_w[(size_t)t * k + j] = score[best];", 0),
    # grouping: histogram, exclusive scan, stable permutation
    "grouping_not_stable": (
        "for (size_t i = 0; i < n; ++i) {\n            if (topk_idx[i] != e) continue;",
        "for (size_t i2 = 0; i2 < n; ++i2) {\n            size_t i = n - 1 - i2;\n"
        "            if (topk_idx[i] != e) continue;", 0),
    "perm_holds_slot_not_token": (
        "perm_tok[pos] = (int32_t)(i / (size_t)k);", "perm_tok[pos] = (int32_t)i;", 0),
    # SwiGLU experts ("zonos2.cpp internals", §Recommended: F16 spine + K-quant experts)
    "silu_drops_z_factor": (
        "h[f] = g / (1.0 + exp(-g)) * u;", "h[f] = 1.0 / (1.0 + exp(-g)) * u;", 0),
    "silu_sign_flipped": ("h[f] = g / (1.0 + exp(-g)) * u;", "h[f] = g / (1.0 + exp(g)) * u;", 0),
    "gate_and_up_swapped": ("h[f] = g / (1.0 + exp(-g)) * u;", "h[f] = u / (1.0 + exp(-u)) * g;", 0),
    "gate_rows_transposed": (
        "decode_row(c->w_gate, c->w_dt, (size_t)e * F + f, d, row);",
        "decode_row(c->w_gate, c->w_dt, (size_t)f * c->E + e, d, row);", 0),
    "combine_weight_dropped": ("o[i] += wt * y;", "o[i] += y;", 0),
    "combine_weight_of_first_slot": (
        "double wt = c->w[(size_t)t * c->k + j];", "double wt = c->w[(size_t)t * c->k];", 0),
    # storage formats: Q8_0 ("zonos2.cpp internals", §Quantization) and the
    # affine 4-bit groups ("Zyphra-ZONOS2-4bit", §How this was quantized)
    "q8_scale_ignored": (
        "out[b * 32 + i] = scale * (double)(int8_t)blk[2 + i];",
        "out[b * 32 + i] = (double)(int8_t)blk[2 + i];", 0),
    "q8_codes_unsigned": ("(double)(int8_t)blk[2 + i]", "(double)blk[2 + i]", 0),
    "q8_scale_bytes_swapped": (
        "(uint16_t)(blk[0] | (blk[1] << 8))", "(uint16_t)(blk[1] | (blk[0] << 8))", 0),
    "f16_exponent_bias_off_by_one": ("expo - 25", "expo - 24", 0),
    "f16_subnormal_scale_off": ("ldexp((double)mant, -24)", "ldexp((double)mant, -25)", 0),
    "q4_nibbles_swapped": (
        "scale * (double)(blk[4 + j] & 15) + bias;\n"
        "                out[b * 64 + 2 * j + 1] = scale * (double)(blk[4 + j] >> 4) + bias;",
        "scale * (double)(blk[4 + j] >> 4) + bias;\n"
        "                out[b * 64 + 2 * j + 1] = scale * (double)(blk[4 + j] & 15) + bias;", 0),
    "q4_bias_scaled": (
        "scale * (double)(blk[4 + j] & 15) + bias;", "scale * ((double)(blk[4 + j] & 15) + bias);", 0),
    "q4_bias_dropped": ("double bias = f16_bits_to_double((uint16_t)(blk[2] | (blk[3] << 8)));",
                        "double bias = 0.0 * (blk[2] | blk[3]);", 0),
    # Q4_K super-blocks ("zonos2.cpp internals", §Recommended: F16 spine + K-quant experts)
    "q4k_high_scale_bits_from_mins": (
        "sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);", "sc = (s[j + 4] & 15) | ((s[j] >> 6) << 4);", 0),
    "q4k_min_nibble_low": ("m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);",
                           "m = (s[j + 4] & 15) | ((s[j] >> 6) << 4);", 0),
    "q4k_sub_block_nibbles_swapped": ("const int q = (j % 2) ? (run[i] >> 4) : (run[i] & 15);",
                                      "const int q = (j % 2) ? (run[i] & 15) : (run[i] >> 4);", 0),
    "q4k_min_added": ("d * (double)sc * (double)q - dmin * (double)m;",
                      "d * (double)sc * (double)q + dmin * (double)m;", 0),
    "q4k_d_dmin_swapped": ("const double dmin = f16_bits_to_double((uint16_t)(blk[2] | (blk[3] << 8)));",
                           "const double dmin = f16_bits_to_double((uint16_t)(blk[0] | (blk[1] << 8)));", 0),
    # Q6_K super-blocks ("zonos2.cpp internals", §Recommended: F16 spine + K-quant experts)
    "q6k_top_bits_shift": ("const int hi = (qh[32 * h + l] >> (2 * g)) & 3;",
                           "const int hi = (qh[32 * h + l] >> g) & 3;", 0),
    "q6k_scale_per_32": ("(double)sc[v / 16]", "(double)sc[v / 32]", 0),
    "q6k_no_offset": ("(double)(q - 32)", "(double)q", 0),
    "q6k_nibble_halves_swapped": ("const int lo = g < 2 ? (lo_byte & 15) : (lo_byte >> 4);",
                                  "const int lo = g < 2 ? (lo_byte >> 4) : (lo_byte & 15);", 0),
    "q6k_ql_run_offset": ("ql[64 * h + l + 32 * (g % 2)]", "ql[64 * h + l + 32 * (g / 2)]", 0),
    # fp8 (E4M3) rows ("zonos2" sglang-omni cookbook, §Benchmark Results: fp8 serving)
    "fp8_exponent_bias_8": ("v = ldexp((double)(8 + mant), expo - 10);",
                            "v = ldexp((double)(8 + mant), expo - 11);", 0),
    "fp8_subnormal_as_normal": ("v = ldexp((double)mant, -9);", "v = ldexp((double)(8 + mant), -10);", 0),
    "fp8_sign_dropped": ("    return sign ? -v : v;\n}\n\n/* Decode row", "    return v;\n}\n\n/* Decode row", 0),
    "fp8_scale_ignored": ("out[c] = (double)scale * e4m3_to_double(p[4 + c]);",
                          "out[c] = e4m3_to_double(p[4 + c]);", 0),
    "fp8_two_mantissa_bits": ("mant = b & 7;", "mant = b & 3;", 0),
    # bf16 storage
    "bf16_low_half": ("uint32_t u = (uint32_t)h << 16;", "uint32_t u = (uint32_t)h << 15;", 0),
}


def _mutate(src, old, new, nth):
    at = -1
    for _ in range(nth + 1):
        at = src.find(old, at + 1)
        assert at >= 0, f"mutation anchor not found: {old!r}"
    return src[:at] + new + src[at + len(old):]


def _copy(dst, name):
    os.makedirs(os.path.join(dst, "oracle"))
    for f in ("__init__.py", "moe_oracle.h"):
        shutil.copy(os.path.join(ORACLE, f), os.path.join(dst, "oracle", f))
    src = open(os.path.join(ORACLE, "moe_oracle.c")).read()
    if name is not None:
        src = _mutate(src, *MUTANTS[name])
    with open(os.path.join(dst, "oracle", "moe_oracle.c"), "w") as f:
        f.write(src)


def _run_pins(dst):
    # The copy comes first on the path; the package and the pins come from the tree.
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([dst, ROOT]))
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu"], cwd=dst, env=env, capture_output=True, text=True,
                       timeout=600)
    return r.returncode, r.stdout[-1500:] + r.stderr[-1500:]


def _loaded_from(dst):
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([dst, ROOT]))
    r = subprocess.run([sys.executable, "-c", "import oracle; print(oracle.__file__)"], cwd=dst,
                       env=env, capture_output=True, text=True, timeout=120, check=True)
    return os.path.realpath(r.stdout.strip())


def test_every_planted_slip_fails_a_pin(tmp_path):
    clean = str(tmp_path / "clean")
    _copy(clean, None)
    assert _loaded_from(clean).startswith(os.path.realpath(clean))
    rc, log = _run_pins(clean)
    assert rc == 0, "clean copy fails its pins:\n" + log

    def one(name):
        dst = str(tmp_path / name)
        _copy(dst, name)
        return name, _run_pins(dst)

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as pool:
        results = list(pool.map(one, sorted(MUTANTS)))
    survivors = [name for name, (rc, _) in results if rc == 0]
    assert not survivors, f"slips no pin catches: {survivors}"
