"""Plant plausible mistakes in a copy of the oracle and check the pins catch them.

Each mutant is the oracle source with one textual change (a flipped tie rule,
a dropped term, swapped operands, a wrong sign, an unstable sort ...), built
with gcc into a temporary directory.  The pins of ``test_oracle_pins`` are then
run against the mutant; at least one of them must fail.  Nothing here touches
a GPU.
"""
import os
import shutil

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")

MUTANTS = {
    "tie_to_higher_id": [("if (best < 0 || l[e] > l[best]) best = e;",
                          "if (best < 0 || l[e] >= l[best]) best = e;")],
    "no_renormalise": [("w[(size_t)t * k + j] = ex[j] / s;", "w[(size_t)t * k + j] = ex[j];")],
    "swap_up_gate": [("const uint16_t *up_row = w1e + (size_t)n * H;",
                      "const uint16_t *up_row = w1e + (size_t)(I + n) * H;"),
                     ("const uint16_t *gate_row = w1e + (size_t)(I + n) * H;",
                      "const uint16_t *gate_row = w1e + (size_t)n * H;")],
    "silu_wrong_sign": [("float silu_g = g / (1.0f + expf(-g));", "float silu_g = g / (1.0f + expf(g));")],
    "round_half_up": [("if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u)))", "if (lo >= 0x8000u)")],
    "w2_transposed": [("acc = acc + bf16_to_float(h[n]) * bf16_to_float(w2_row[n]);",
                       "acc = acc + bf16_to_float(h[n]) * bf16_to_float(w2e[(size_t)n * H + c]);")],
    "combine_drops_weight": [("acc = acc + w[j] * y[(size_t)j * H + c];",
                              "acc = acc + y[(size_t)j * H + c];")],
    "fc1_drops_last_term": [("        for (int c = 0; c < H; ++c) {\n            float xv = bf16_to_float(x_row[c]);",
                             "        for (int c = 0; c < H - 1; ++c) {\n            float xv = bf16_to_float(x_row[c]);")],
    "sort_unstable": [("int p = next[e - off]++;",
                       "int p = m_indptr[e - off + 1] - 1 - (next[e - off]++ - m_indptr[e - off]);")],
    "sort_offsets_off_by_one": [("for (int i = 0; i < L; ++i) m_indptr[i + 1] = m_indptr[i] + cnt[i];",
                                 "for (int i = 0; i < L; ++i) m_indptr[i + 1] = m_indptr[i] + cnt[i] + (i == 0);")],
    "step_clamps_gate_below": [("    if (g > limit) g = limit;\n",
                                "    if (g > limit) g = limit;\n    if (g < -limit) g = -limit;\n")],
    "step_up_clamped_above_only": [("    if (u < -limit) u = -limit;\n", "")],
    "step_limit_by_global_id": [("limit_of(clamp, e - off), h, y + (size_t)j * H);",
                                 "limit_of(clamp, e), h, y + (size_t)j * H);")],
    "dgrad_row_off_by_one": [("const uint16_t *gr = G + (size_t)p * N;",
                              "const uint16_t *gr = G + (size_t)(p > 0 ? p - 1 : p) * N;")],
    "dgrad_drops_last_term": [("            for (int n = 0; n < N; ++n)\n                acc = acc + bf16_to_float(gr[n]) *",
                               "            for (int n = 0; n < N - 1; ++n)\n                acc = acc + bf16_to_float(gr[n]) *")],
    "wgrad_takes_next_row": [("for (int p = start; p < end; ++p)",
                              "for (int p = start; p < end + (end < offs[E - 1]); ++p)")],
    "bgmv_wrong_lora": [("(((size_t)lora[t] * E + eid[p]) * R) * (size_t)H;",
                         "(((size_t)(num_loras - 1 - lora[t]) * E + eid[p]) * R) * (size_t)H;")],
    "bgmv_drops_weight": [("acc = acc + w[p] * v;", "acc = acc + v;")],
    "e4m3_no_saturation": [("    if (a >= 448.0f) return (uint8_t)(s | 0x7E);\n", "    if (a >= 480.0f) return (uint8_t)(s | 0x7F);\n")],
    "e4m3_truncates": [("    float q = nearbyintf(ldexpf(fr, 4)); /* mant * 8 = fr * 16 */",
                        "    float q = floorf(ldexpf(fr, 4));")],
    "fp8_h_not_requantised_by_a2": [("        hq[n] = float_to_e4m3(swiglu_step(g, u, limit) / a2);",
                                     "        hq[n] = float_to_e4m3(swiglu_step(g, u, limit));")],
    "finalize_skips_slot0": [("            for (int j = 0; j < k; ++j) {\n                int p = exp_to_perm[(size_t)t * k + j];",
                              "            for (int j = 1; j < k; ++j) {\n                int p = exp_to_perm[(size_t)t * k + j];")],
}

PIN_CALLS = [
    ("route_hand_worked", lambda: pins.test_route_hand_worked()),
    ("route_bruteforce", lambda: pins.test_route_bruteforce_with_ties(5)),
    ("route_weights", lambda: pins.test_route_weights_vs_fp64_softmax_topk_renorm(8, 2)),
    ("sort_hand_worked", lambda: pins.test_sort_hand_worked()),
    ("sort_argsort", lambda: pins.test_sort_vs_stable_argsort(64, 8, 128, 32, 40, False)),
    ("layer_fp64", lambda: pins.test_layer_bruteforce_fp64_tiny()),
    ("dense_mlp", lambda: pins.test_e1_k1_equals_dense_swiglu_mlp(9, 64, 64)),
    ("stages_compose", lambda: pins.test_stage_functions_compose_to_layer()),
    ("grouped_gemm", lambda: pins.test_grouped_gemm_vs_torch_per_group()),
    ("rounding", lambda: pins.test_bf16_rounding_matches_torch()),
    ("step_hand_worked", lambda: pins.test_swiglu_step_hand_worked()),
    ("step_fp64", lambda: pins.test_swiglu_step_fp64_bruteforce_tiny()),
    ("dgrad_torch", lambda: pins.test_grouped_gemm_dgrad_vs_torch_per_group()),
    ("wgrad_torch", lambda: pins.test_grouped_gemm_wgrad_vs_torch_per_group_and_empty_groups_zero()),
    ("gg_adjoint", lambda: pins.test_grouped_gemm_adjoint_identity()),
    ("bgmv_torch", lambda: pins.test_bgmv_vs_torch_per_pair(False)),
    ("bgmv_invariants", lambda: pins.test_bgmv_rank_padding_linearity_and_zero_b()),
    ("e4m3_torch", lambda: pins.test_e4m3_codes_exhaustive_against_torch()),
    ("e4m3_round", lambda: pins.test_e4m3_rounding_ties_and_saturation()),
    ("fp8_fp64", lambda: pins.test_fp8_layer_fp64_tiny()),
    ("step_per_expert", lambda: pins.test_swiglu_step_infinite_limit_is_plain_swiglu_and_limits_are_per_local_expert()),
]


def _build_mutant(tmp_path, name):
    src = open(SRC).read()
    for old, new in MUTANTS[name]:
        assert src.count(old) == 1, f"mutation anchor for {name} not unique: {old!r}"
        src = src.replace(old, new)
    path = os.path.join(str(tmp_path), f"{name}.c")
    open(path, "w").write(src)
    out = os.path.join(str(tmp_path), f"lib_{name}.so")
    oracle.build(force=True, src=path, out=out)
    return oracle.load(out)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path, monkeypatch):
    lib = _build_mutant(tmp_path, name)
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = []
    for pin, call in PIN_CALLS:
        try:
            call()
        except AssertionError:
            caught.append(pin)
    assert caught, f"mutant {name} passed every pin"


def test_unmutated_copy_passes_all_pins(tmp_path, monkeypatch):
    path = os.path.join(str(tmp_path), "same.c")
    shutil.copy(SRC, path)
    out = os.path.join(str(tmp_path), "lib_same.so")
    oracle.build(force=True, src=path, out=out)
    monkeypatch.setattr(oracle, "_lib", oracle.load(out))
    for _, call in PIN_CALLS:
        call()
