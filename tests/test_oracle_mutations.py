"""Planted mistakes in the oracle must be caught by its pins.

Each mutant is a copy of the oracle's C++ source with one plausible mistake
planted by a text edit (a swapped operand, a wrong tie-break, a renormalised
mask, single-precision accumulation, the wrong FP8 variant's maximum, ...).
The copy is compiled into a library of its own and every pin runs against
it; at least one pin has to fail.  Mistakes are planted on the CPU, in the
oracle, never in the CUDA path.
"""

import concurrent.futures
import json
import os

import numpy as np
import pytest

from oracle import build as obuild
from oracle import moe_oracle as mo
import tests.test_oracle_fp4 as fp4_pins
import tests.test_oracle_fp8 as fp8_pins
import tests.test_oracle_pins as pins
import tests.test_oracle_router as router_pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cases(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)["cases"]


def _all_pins():
    """Run every pin once; return the number that fail."""
    checks = []
    for c in _cases("topk_cases.json"):
        checks.append(lambda c=c: pins.test_golden_topk(c))
    for c in _cases("softmax_cases.json"):
        checks.append(lambda c=c: pins.test_golden_softmax(c))
    for c in _cases("ffn_cases.json"):
        checks.append(lambda c=c: pins.test_golden_ffn(c))
    for c in _cases("combine_cases.json"):
        checks.append(lambda c=c: pins.test_golden_combine(c))
    checks += [
        pins.test_topk_brute_force_with_ties,
        pins.test_softmax_matches_full_softmax_renormalised,
        lambda: pins.test_histogram_offsets_permutation(33, 16, 6, 0.25),
        lambda: pins.test_histogram_offsets_permutation(64, 12, 12, 0.5),
        pins.test_scatter_then_gather_is_identity,
        pins.test_single_expert_is_dense_swiglu,
        pins.test_k_equals_E_is_full_softmax_mixture,
        pins.test_all_masked_gives_plus_zero,
        pins.test_masked_expert_never_touched,
        pins.test_silu_closed_forms,
        fp8_pins.test_e4m3_round_matches_torch_cast,
        fp8_pins.test_negative_values_that_round_to_zero_keep_their_sign,
        fp8_pins.test_e4m3_ties_go_to_even_and_saturate,
        fp8_pins.test_code_layout_and_round_trip,
        fp8_pins.test_per_channel_scaling_properties,
        fp8_pins.test_quantized_bank_ffn_is_the_dequantized_ffn,
        fp8_pins.test_bf16_rounding_matches_torch_cast,
        fp8_pins.test_w8a8_path_is_the_dense_ffn_on_quantized_operands,
        fp4_pins.test_e2m1_code_table,
        fp4_pins.test_e2m1_rounding_against_brute_force,
        fp4_pins.test_fp4_quantizer_hand_worked_row,
        fp4_pins.test_fp4_quantizer_picks_the_nearest_value_of_each_block,
        fp4_pins.test_fp4_bank_ffn_is_the_dequantized_ffn,
        fp4_pins.test_w4a4_path_is_the_dense_ffn_on_quantized_operands,
        router_pins.test_hand_worked_router_case,
        router_pins.test_one_hot_router_rows_select_input_columns,
        router_pins.test_router_is_linear_and_permutation_equivariant,
    ]
    failures = 0
    for check in checks:
        try:
            with np.errstate(all="ignore"):
                check()
        except (AssertionError, ValueError, IndexError):
            failures += 1
    return failures


# (name, [(text in the oracle source, replacement), ...]); each text must occur exactly once
MUTANTS = [
    ("topk_ties_to_higher_id",
     [("return row[a] > row[b]; });", "return row[a] > row[b] || (row[a] == row[b] && a > b); });")]),
    ("softmax_over_all_experts",
     [("for (int s = 0; s < k; ++s) sum += std::exp", "for (int s = 0; s < E; ++s) sum += std::exp")]),
    ("swapped_gate_and_up", [("silu(g[r]) * u[r]", "silu(u[r]) * g[r]")]),
    ("down_read_with_gate_shape",
     [("static_cast<size_t>(e - e0) * d, d, f, wd.data());", "static_cast<size_t>(e - e0) * d, f, d, wd.data());")]),
    ("silu_is_sigmoid", [("return a / (1.0 + std::exp(-a));", "return 1.0 / (1.0 + std::exp(-a));")]),
    ("single_precision_accumulation", [("double sa[NR], sb[NR];", "float sa[NR], sb[NR];")]),
    ("combine_renormalised_over_unmasked",
     [("const double ws = w[t * k + s];",
       "double wsum = 0.0;\n            for (int q = 0; q < k; ++q) if (row_of_route[t * k + q] >= 0) wsum += "
       "w[t * k + q];\n            const double ws = w[t * k + s] / wsum;")]),
    ("combine_starts_at_minus_zero", [("for (int c = 0; c < d; ++c) o[c] = 0.0;", "for (int c = 0; c < d; ++c) o[c] = -0.0;")]),
    ("combine_multiplies_masked_slots",
     [("if (row < 0) continue;", "if (row < 0 && n_rows == 0) continue;"),
      ("const double ws = w[t * k + s];", "const double ws = row < 0 ? 0.0 : w[t * k + s];"),
      ("ws * y[row * d + c]", "ws * y[(row < 0 ? 0 : row) * d + c]")]),
    ("permutation_reversed_within_expert",
     [("return ids[a] < ids[b]; });", "return ids[a] < ids[b] || (ids[a] == ids[b] && a > b); });")]),
    ("inclusive_prefix",
     [("offsets[e + 1] = offsets[e] + counts[e];",
       "offsets[e + 1] = offsets[e] + counts[e];\n    for (int e = 0; e < E; ++e) offsets[e] = offsets[e + 1];")]),
    ("histogram_counts_masked_routes",
     [("        if (mask && mask[r]) continue;\n        if (ids[r] < 0", "        if (ids[r] < 0")]),
    ("gather_uses_slot_not_token", [("route_of_row[i] / k);", "route_of_row[i] % k);")]),
    ("e4m3_ties_away_from_zero", [("std::nearbyint(a / quantum) * quantum;\n    r = std::min(r, 448.0);",
                                   "std::round(a / quantum) * quantum;\n    r = std::min(r, 448.0);")]),
    ("e4m3_subnormal_binade_off_by_one", [("std::max(ex - 1, -6);", "std::max(ex - 1, -7);")]),
    ("fp8_scale_of_the_fnuz_variant", [("amax / 448.0f", "amax / 240.0f")]),
    ("bf16_with_seven_significant_bits", [("std::ldexp(1.0, binade - 7);", "std::ldexp(1.0, binade - 6);")]),
    ("e2m1_ties_away_from_zero", [("std::nearbyint(a / quantum) * quantum;\n    r = std::min(r, 6.0);",
                                   "std::round(a / quantum) * quantum;\n    r = std::min(r, 6.0);")]),
    ("fp4_block_scale_from_max_over_4", [("bmax / 6.0f / s", "bmax / 4.0f / s")]),
    ("fp4_row_scale_without_the_e2m1_max", [("amax / 2688.0f", "amax / 448.0f")]),
    ("fp4_nibbles_swapped", [("q << (4 * (i & 1))", "q << (4 * (1 - (i & 1)))")]),
    ("fp4_blocks_of_8_when_decoding", [("e4m3_value(bs[c / 16])", "e4m3_value(bs[c / 8])")]),
    ("router_reads_wr_transposed",
     [("element(wr, wdtype, static_cast<size_t>(e) * d + c)", "element(wr, wdtype, static_cast<size_t>(c) * E + e)")]),
]


def _mutated_source(edits):
    with open(obuild.SRC) as fh:
        src = fh.read()
    for old, new in edits:
        assert src.count(old) == 1, f"mutation anchor not unique or missing: {old!r}"
        src = src.replace(old, new)
    return src


@pytest.fixture(scope="module")
def mutant_libs(tmp_path_factory):
    root = tmp_path_factory.mktemp("oracle_mutants")
    with concurrent.futures.ThreadPoolExecutor(max_workers=8) as ex:
        futs = {name: ex.submit(obuild.build, str(root / f"lib_{name}.so"), _mutated_source(edits))
                for name, edits in MUTANTS}
        return {name: f.result() for name, f in futs.items()}


def test_unmutated_oracle_passes_every_pin():
    assert _all_pins() == 0


def test_unmutated_rebuild_passes_every_pin(tmp_path):
    """A copy of the unmodified source built like a mutant passes (the harness itself plants nothing)."""
    with mo.use_library(obuild.build(str(tmp_path / "lib_copy.so"), _mutated_source([]))):
        assert _all_pins() == 0


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_mutant_is_caught(mutant_libs, name):
    with mo.use_library(mutant_libs[name]):
        assert _all_pins() > 0
