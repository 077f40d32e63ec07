"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (a wrong
exponent bias, a dropped term, a flipped sign, a transposed index, the wrong
tie rule, ...), builds that copy, swaps it in for the oracle's library and
runs the pins that should catch it: at least one must fail.  The planted
mistakes stay in bounds, so a mutant can give wrong numbers but not fault."""
from __future__ import annotations

import ctypes
import os
import subprocess

import pytest

import oracle
import synth
from tests import test_oracle as T

SRC = os.path.join(os.path.dirname(os.path.abspath(oracle.__file__)), "moe_oracle.c")

FP8, NVFP4 = synth.FMT_FP8, synth.FMT_NVFP4

# (name, text in the oracle, its planted replacement, pins expected to catch it)
MUTANTS = [
    ("e4m3 exponent bias 8",
     "v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);",
     [T.test_e4m3_all_codes_match_torch]),
    ("e4m3 subnormal step 2^-10",
     "v = ldexp((double)m / 8.0, -6);", "v = ldexp((double)m / 8.0, -7);",
     [T.test_e4m3_all_codes_match_torch]),
    ("e2m1 subnormal 1.0",
     "(e == 0) ? 0.5 * (double)m", "(e == 0) ? 1.0 * (double)m",
     [T.test_e2m1_matches_ocp_table]),
    ("bf16 ties away from zero",
     "double r = nearbyint(a / q);", "double r = round(a / q);",
     [T.test_bf16_rne_closed_form_cases, T.test_bf16_rne_matches_torch_on_float32_values]),
    ("router drops the last input",
     "for (int c = 0; c < H; ++c)\n                acc += oracle_bf16_value(x[(size_t)t * H + c]) *",
     "for (int c = 0; c < H - 1; ++c)\n                acc += oracle_bf16_value(x[(size_t)t * H + c]) *",
     [T.test_router_logits_match_torch_matmul, T.test_router_logits_closed_form]),
    ("top-k ties to the higher id",
     "if (best < 0 || l[e] > l[best])", "if (best < 0 || l[e] >= l[best])",
     [T.test_topk_ties_take_lower_id_brute_force]),
    ("top-k weights not renormalised",
     "w[(size_t)t * k + j] = p[ids[(size_t)t * k + j]] / sel;",
     "w[(size_t)t * k + j] = p[ids[(size_t)t * k + j]];",
     [T.test_topk_softmax_matches_torch]),
    ("alignment rank counts later slots",
     "/* stage 3 */\n    for (int i = 0; i < n; ++i) {",
     "/* stage 3 */\n    for (int i = n - 1; i >= 0; --i) {",
     [T.test_align_arbitrary_ids_with_repeats_brute_force,
      T.test_align_every_routing_of_three_tokens_brute_force]),
    ("alignment without block padding",
     "padded[e] = (counts[e] + BS - 1) / BS * BS;", "padded[e] = counts[e];",
     [T.test_align_every_routing_of_three_tokens_brute_force,
      T.test_align_arbitrary_ids_with_repeats_brute_force]),
    ("nvfp4 high nibble first",
     "(i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF)",
     "(i & 1) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4)",
     [T.test_dequant_nvfp4_matches_table_and_torch]),
    ("fp8 block scales transposed",
     "* (double)s[(o / 128) * sc + i / 128];", "* (double)s[(i / 128) * sr + o / 128];",
     [T.test_dequant_fp8_matches_torch]),
    ("silu with the wrong sign",
     "static double silu(double z) { return z / (1.0 + exp(-z)); }",
     "static double silu(double z) { return z / (1.0 + exp(z)); }",
     [lambda: T.test_grouped_stages_match_torch(FP8, False)]),
    ("shared expert left out of the blend",
     "            if (y_sh)\n                acc +=", "            if (0)\n                acc +=",
     [lambda: T.test_layer_matches_torch(NVFP4, True)]),
    ("blend skips slot 0",
     "for (int j = 0; j < top_k; ++j) {\n                int32_t p = token_to_perm",
     "for (int j = 1; j < top_k; ++j) {\n                int32_t p = token_to_perm",
     [T.test_blend_skips_bad_slots_and_is_weighted_sum]),
    ("gate with the wrong sign",
     "g[t] = 1.0 / (1.0 + exp(-z));", "g[t] = 1.0 / (1.0 + exp(z));",
     [T.test_shared_gate_special_values_and_symmetry]),
    ("gate on the whole sum",
     "acc += (gate ? gate[t] : 1.0) * y_sh[(size_t)t * H + c];",
     "acc = (gate ? gate[t] : 1.0) * (acc + y_sh[(size_t)t * H + c]);",
     [T.test_blend_gate_scales_only_the_shared_term]),
]


def _build_mutant(tmp_path, old: str, new: str) -> ctypes.CDLL:
    text = open(SRC).read()
    assert text.count(old) == 1, old
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-o",
                    str(so), str(src), "-lm"], check=True, capture_output=True)
    lib = ctypes.CDLL(str(so))
    oracle._declare(lib)
    return lib


@pytest.mark.parametrize("name,old,new,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, monkeypatch, name, old, new, pins):
    monkeypatch.setattr(oracle, "_lib", _build_mutant(tmp_path, old, new))
    caught = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin caught: {name}"
