"""The oracle's pins must catch plausible mistakes in the oracle itself.

Each case below plants one mistake in a temporary copy of oracle/sga_oracle.c
(a flipped tie rule, a NaN that does not stick, an off-by-one padding mask, a
local instead of a global id, a transposed stats layout, acceptance that keeps
counting after a mismatch, a missing bonus-row offset, a wrong count, a dropped
dot-product term, a wrong bf16 widening, a runner-up equal to the winner, the
bonus taken from the wrong row, a wrong E4M3 exponent bias, the fp8 scales
dropped, block boundaries taken from the shard start instead of global ids,
the bonus row's block size ignored or given to the wrong row, an empty block
slot naming the shard's first id, a block count off by one, the smaller of
the two block counts as the slot count, a draft-to-target map that drops the
draft id, the prefill mask ignored, a request in prefill counting its drafts
as rejected), builds it with gcc, points the oracle wrapper
at it, and runs the pin tests of tests/test_oracle_pins.py: at least one pin
must fail for every mutant.  The committed oracle source is never modified.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "sga_oracle.c")

MUTANTS = {
    "ties_keep_last": ("(isnan(cand) || cand > best)", "(isnan(cand) || cand >= best)"),
    "nan_not_sticky": ("return !isnan(best) && (isnan(cand) || cand > best);",
                       "return (isnan(cand) || cand > best);"),
    "mask_off_by_one": ("if (global_id >= org_vocab) return -INFINITY;",
                        "if (global_id > org_vocab) return -INFINITY;"),
    "local_id": ("return (int32_t)(first + best_j);", "return (int32_t)(best_j);"),
    "stats_row_major": ("oracle_stat c = stats[(int64_t)s * rows + r];",
                        "oracle_stat c = stats[(int64_t)r * num_shards + s];"),
    "accept_past_mismatch": ("while (a < k && draft_tokens[c + a] == t[b + a]) ++a;",
                             "for (int j = 0; j < k; ++j) a += draft_tokens[c + j] == t[b + j];"),
    "no_bonus_row_offset": ("int64_t b = (int64_t)c + i;", "int64_t b = (int64_t)c;"),
    "rejected_off_by_one": ("out_num_rejected[i] = k - a;", "out_num_rejected[i] = k - a - 1;"),
    "bonus_from_last_row": ("out_bonus[i] = t[b + a];", "out_bonus[i] = t[b + k];"),
    "dot_drops_last_term": ("for (int64_t k = 0; k < H; ++k) {", "for (int64_t k = 0; k < H - 1; ++k) {"),
    "bf16_widen_shift": ("u = ((uint32_t)b) << 16;", "u = ((uint32_t)b) << 15;"),
    "top2_includes_winner": ("if (j != best_j && c > second) second = c;",
                             "if (c > second) second = c;"),
    "e4m3_bias_off_by_one": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);",
                             "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "fp8_scale_dropped": ("out[j] = scale * acc;", "out[j] = acc;"),
    "blocks_relative_to_shard": ("int64_t lo = (b0 + p) * B, hi = (b0 + p + 1) * B;",
                                 "int64_t lo = shard_start + p * B, hi = shard_start + (p + 1) * B;"),
    "bonus_row_uses_draft_block": ("const int64_t B = is_bonus[r] ? bonus_block : draft_block;",
                                   "const int64_t B = draft_block;"),
    "bonus_row_is_first_row": ("is_bonus[(int64_t)cu_num_draft[i + 1] + i] = 1;",
                               "is_bonus[(int64_t)cu_num_draft[i] + i] = 1;"),
    "empty_slot_id_at_shard_start": ("st.id = (int32_t)(shard_end - 1);",
                                     "st.id = (int32_t)(shard_start);"),
    "block_count_off_by_one": (
        "return (shard_start + shard_width - 1) / block - shard_start / block + 1;",
        "return (shard_start + shard_width) / block - shard_start / block + 1;"),
    "slots_take_the_smaller_count": ("n_draft > n_bonus ? n_draft : n_bonus",
                                     "n_draft < n_bonus ? n_draft : n_bonus"),
    "prefill_mask_ignored": ("if (in_prefill && in_prefill[i]) {", "if (0 && in_prefill) {"),
    "prefill_counts_drafts_rejected": ("      out_num_sampled[i] = 0;\n      out_num_rejected[i] = 0;",
                                       "      out_num_sampled[i] = 0;\n      out_num_rejected[i] = k;"),
    "d2t_drops_the_draft_id": ("out_target_ids[r] = (int32_t)(k + d2t[k]);",
                               "out_target_ids[r] = (int32_t)(d2t[k]);"),
}

PIN_CALLS = [
    lambda: pins.test_argmax_matches_set_brute_force("bf16", 3),
    lambda: pins.test_argmax_matches_set_brute_force("f32", 1),
    pins.test_shard_narrower_than_vector_and_single_ids,
    pins.test_all_padding_shard_reports_its_first_id,
    pins.test_nan_and_inf_only_in_padding_never_win,
    pins.test_plus_minus_zero_tie_keeps_lowest_id_and_its_bits,
    pins.test_nan_payload_and_first_nan_across_shards,
    pins.test_torch_argmax_third_opinion_unpadded,
    pins.test_tiny_workload_planted_rows,
    pins.test_verify_hand_cases,
    pins.test_verify_prefill_hand_cases,
    pins.test_verify_random_variable_k_matches_brute_force,
    pins.test_verify_reduces_stats_across_shards_first,
    pins.test_lmhead_logits_match_numpy_fp64_matmul,
    pins.test_lmhead_one_hot_weight_is_exact_column_pick,
    pins.test_e4m3_decode_matches_torch_float8_for_every_code,
    pins.test_lmhead_fp8_logits_match_numpy_with_scales,
    lambda: pins.test_block_stats_match_grouped_brute_force("bf16"),
    pins.test_block_pieces_follow_global_boundaries_across_shard_edges,
    pins.test_d2t_map_hand_case,
]


def build_mutant(tmp_path, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, old
    c_file = tmp_path / "mutant.c"
    c_file.write_text(src.replace(old, new))
    so = tmp_path / "mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", str(c_file), "-o", str(so), "-lm"],
                   check=True, capture_output=True)
    return oracle.configure(ctypes.CDLL(str(so)))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(tmp_path, monkeypatch, name):
    lib = build_mutant(tmp_path, *MUTANTS[name])
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = 0
    for call in PIN_CALLS:
        try:
            call()
        except (AssertionError, ValueError):
            caught += 1
    assert caught > 0, f"no pin catches the mutant {name}"


def test_unmutated_copy_passes_every_pin(tmp_path, monkeypatch):
    lib = build_mutant(tmp_path, "u = ((uint32_t)b) << 16;", "u = ((uint32_t)b) << 16;")
    monkeypatch.setattr(oracle, "_lib", lib)
    for call in PIN_CALLS:
        call()
