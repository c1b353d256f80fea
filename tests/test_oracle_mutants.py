"""The oracle's pins have teeth: a plausible mistake planted in a copy of the
oracle source (compiled on the CPU into a temporary library) must make at
least one pin fail.  Only in-bounds mistakes are planted."""
import os
import subprocess
import tempfile

import pytest

import oracle
import test_oracle_combine as combine_pins
import test_oracle_pins as pins
import test_oracle_plan_variants as skip_pins
import test_oracle_stage as stage_pins
from golden_io import read_sections

SRC = os.path.join(os.path.dirname(oracle.__file__), "ultraep_oracle.c")

MUTANTS = {
    "hot tie to highest rank": ("if (L[r] > L[hot]) hot = r;", "if (L[r] >= L[hot]) hot = r;"),
    "instance tie to highest expert": ("(quota[p] == quota[src_p] && e < src_e)",
                                       "(quota[p] == quota[src_p] && e > src_e)"),
    "cold tie to highest rank": ("if (cold < 0 || L[c] < L[cold]) cold = c;",
                                 "if (cold < 0 || L[c] <= L[cold]) cold = c;"),
    "move the whole gap": ("int64_t half = (L[hot] - L[cold]) / 2;",
                           "int64_t half = (L[hot] - L[cold]);"),
    "halve rounding up": ("int64_t half = (L[hot] - L[cold]) / 2;",
                          "int64_t half = (L[hot] - L[cold] + 1) / 2;"),
    "ignore the instance quota": ("int64_t q = quota[src_p] < half ? quota[src_p] : half;",
                                  "int64_t q = half;"),
    "highest free slot first": (
        "for (int32_t j = 0; j < S && dst_p < 0; j++)\n            if (slot_expert[cold * S + j] < 0) {",
        "for (int32_t j = S - 1; j >= 0 && dst_p < 0; j--)\n            if (slot_expert[cold * S + j] < 0) {"),
    "holders not eligible": ("if (slot_expert[c * S + j] == src_e) holds = 1;",
                             "if (slot_expert[c * S + j] == src_e) holds = 0;"),
    "home rank not eligible": ("int holds = (src_e / H == c);", "int holds = 0;"),
    "replicas listed by descending p": (
        "for (int32_t p = 0; p < P; p++) {\n            int32_t j = p % W;",
        "for (int32_t p = P - 1; p >= 0; p--) {\n            int32_t j = p % W;"),
    "cap allows one extra move": ("if (moves == max_iters)", "if (moves > max_iters)"),
    "count drops the last choice": ("for (int32_t j = 0; j < k; j++) {\n            int32_t e = ids[t * k + j];",
                                    "for (int32_t j = 0; j < k - (k > 1); j++) {\n            int32_t e = ids[t * k + j];"),
    "source ranks by floor": ("int64_t Tr = (T + R - 1) / R;", "int64_t Tr = (T / R) + 1;"),
    "instance rows not in slot order": ("int64_t row = inst_offset[p] + fill[p]++;",
                                        "int64_t row = inst_offset[p + 1] - 1 - fill[p]++;"),
    "permute reads the row's own index": ("int64_t t = src_slot[row] / k;", "int64_t t = row / k;"),
    "missing slot not zeroed": ("(row < 0) ? 0 : grouped[row * Hd + h]",
                                "(row < 0) ? grouped[h] : grouped[row * Hd + h]"),
    "combine sums in descending j": (
        "for (int32_t j = 0; j < k; j++) {\n                int64_t row = dst_row[t * k + j];",
        "for (int32_t j = k - 1; j >= 0; j--) {\n                int64_t row = dst_row[t * k + j];"),
    "combine rounds toward zero": (
        "if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;",
        "if (lower > 0xFFFFu) upper += 1u;"),
    "combine rounds ties up": (
        "if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;",
        "if (lower >= 0x8000u) upper += 1u;"),
    "combine keeps NaN payloads": ("!= 0) return 0x7FC0u;", "!= 0) return (uint16_t)(u >> 16);"),
    "combine reads row 0 for missing slots": ("if (row < 0) continue;", "if (row < 0) row = 0;"),
    "combine accumulates in double": ("float sum = 0.0f;", "double sum = 0.0;"),
    "combine multiplies after the sum": ("sum = sum + prod;", "sum = sum + x;"),
    "skip tries the coldest rank first": (
        "if (!rank_tried[r] && (hot < 0 || L[r] > L[hot])) hot = r;",
        "if (!rank_tried[r] && (hot < 0 || L[r] < L[hot])) hot = r;"),
    "skip gives up after the hottest rank": ("int32_t n_ranks = (flags & ORACLE_PLAN_SKIP) ? R : 1;",
                                             "int32_t n_ranks = (flags & ORACLE_PLAN_SKIP) ? 1 : 1;"),
    "skip gives up after one instance": ("int32_t n_insts = (flags & ORACLE_PLAN_SKIP) ? W : 1;",
                                         "int32_t n_insts = (flags & ORACLE_PLAN_SKIP) ? 1 : 1;"),
    "skip tries the smallest instance first": (
        "if (src_p < 0 || quota[p] > quota[src_p] ||\n                        (quota[p] == quota[src_p] && e < src_e)) {",
        "if (src_p < 0 || quota[p] < quota[src_p] ||\n                        (quota[p] == quota[src_p] && e < src_e)) {"),
    "release never frees a slot": ("if ((flags & ORACLE_PLAN_RELEASE) && src_p % W >= H && quota[src_p] == 0)",
                                   "if ((flags & ORACLE_PLAN_RELEASE) && src_p % W >= H && quota[src_p] < 0)"),
    "release frees replicas that still hold quota": (
        "if ((flags & ORACLE_PLAN_RELEASE) && src_p % W >= H && quota[src_p] == 0)",
        "if ((flags & ORACLE_PLAN_RELEASE) && src_p % W >= H && quota[src_p] >= 0)"),
    "stage ignores what a slot holds": ("if (prev != NULL && prev[x] == e) continue;",
                                        "if (prev != NULL && prev[x] == e + E) continue;"),
    "stage clears empty slots": (
        "if (e == -1) continue;",
        "if (e == -1) { memset(slot_w + x * expert_bytes, 0, (size_t)expert_bytes); continue; }"),
    "stage copies the next expert": ("expert_w + (int64_t)e * expert_bytes",
                                     "expert_w + (int64_t)((e + 1) % E) * expert_bytes"),
}


def battery():
    hand = read_sections("plan_hand_examples.txt")
    for name in sorted(hand):
        pins.test_plan_hand_examples(name)
        if "ids" in hand[name]:
            pins.test_reroute_hand_examples(name)
    for args in [(37, 3, 4, 8), (4096, 4, 8, 32), (5, 2, 8, 16)]:
        pins.test_count_is_a_histogram(*args)
    for seed in range(40):
        pins.test_plan_invariants_random(seed)
    for args in [(3, 1, 12), (8, 2, 77)]:
        pins.test_plan_single_hot_expert_levels_ranks(*args)
    pins.test_plan_iteration_cap_random()
    for seed in range(10):
        pins.test_reroute_properties_random(seed)
    for args in [(17, 3, 16), (64, 8, 24)]:
        pins.test_permute_unpermute_are_gathers(*args)
    pins.test_pipeline_round_trip_tiny_workload()
    for name in ("test_exact_binary_fractions", "test_float32_sum_in_ascending_j",
                 "test_bf16_round_to_nearest_even", "test_nan_inf_and_signed_zero",
                 "test_missing_slots_add_nothing_and_zero_weights",
                 "test_rows_follow_dst_row_per_token"):
        getattr(combine_pins, name)()
    combine_pins.test_k1_unit_weight_is_the_identity(0)
    for name in sorted(skip_pins.SKIP):
        skip_pins.test_skip_hand_examples(name)
    for seed in range(8):
        skip_pins.test_skip_prefix_stop_and_bounds(seed, "skip")
        skip_pins.test_skip_prefix_stop_and_bounds(seed, "skip+release")
    stage_pins.test_stage_is_a_gather_of_expert_rows()
    stage_pins.test_empty_invalid_and_unchanged_slots_are_left_alone()


def test_battery_passes_on_the_oracle():
    battery()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    # the first occurrence is the one in the function the mutant names (the
    # skip variant repeats some lines of the base rule further down the file)
    assert src.count(old) >= 1, "mutation site not found"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new, 1))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-shared", "-fPIC",
                    str(mutated), "-o", str(so)], check=True)
    with oracle.using_library(str(so)):
        with pytest.raises(AssertionError):
            battery()
