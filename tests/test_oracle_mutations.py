"""The oracle's pins must catch plausible mistakes. Each case below plants one
mistake in a temporary copy of the oracle's C source (on the CPU), builds it, and
checks that at least one pin in tests/test_oracle_pins.py fails against it."""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "hstu_oracle.c")

# (name, text in the oracle, mistaken text)
MUTATIONS = [
    ("transposed_scores", "const double *qi = J->q + ((t0 + i) * J->Nq + h) * D;",
     "const double *qi = J->q + ((t0 + i) * J->Nq + h) * D; (void)0;\n"
     "    const double *qq = qi; (void)qq;"),  # placeholder replaced below
    ("dropped_rab", "x += J->rab[(plane", "x += 0.0 * J->rab[(plane"),
    ("alpha_scales_rab", "x += J->rab[(plane", "x += J->alpha * J->rab[(plane"),
    ("rab_transposed", "(plane * J->max_seqlen + pos) * J->max_seqlen + j]", "(plane * J->max_seqlen + j) * J->max_seqlen + pos]"),
    ("rab_head_ignored", "(J->rab_heads == 1 ? 0 : h)", "(J->rab_heads == 1 ? 0 : 0)"),
    ("silu_sign", "return x / (1.0 + exp(-x));", "return x / (1.0 + exp(x));"),
    ("sigmoid_not_silu", "return x / (1.0 + exp(-x));", "return 1.0 / (1.0 + exp(-x));"),
    ("gqa_modulo", "const int64_t hk = h / G;", "const int64_t hk = h % J->Nk;"),
    ("causal_strict", "if (j <= i && j < H) return 1;", "if (j < i && j < H) return 1;"),
    ("context_off_by_one", "if (i < nc && j < H) return 1;", "if (i <= nc && j < H) return 1;"),
    ("group_not_offset_by_history", "(i - H) / g == (j - H) / g) return 1;", "i / g == j / g) return 1;"),
    ("history_off_by_one", "H = L - nt;", "H = L - nt + 1;"),
    ("targets_see_future_in_group", "j >= H && j <= i && (i - H)", "j >= H && (i - H)"),
    ("dropped_scale", "p *= J->silu_scale;", "p *= 1.0;"),
    ("v_row_of_query", "const double *vj = kv_row(J, b, hk, j, 1);",
     "const double *vj = kv_row(J, b, hk, i, 1);"),
    ("mask_none_causal", "if (mask_type == ORACLE_MASK_NONE || mask_type == ORACLE_MASK_CUSTOM) return 1;",
     "if (mask_type == ORACLE_MASK_CUSTOM) return 1;"),
    ("custom_mask_ignored", "p *= J->mask[", "p *= 1.0 + 0.0 * J->mask["),
    ("custom_mask_before_silu", "    double p = silu(x);", "    if (J->mask_type == ORACLE_MASK_CUSTOM)\n"
     "      x *= J->mask[((b * J->Nq + h) * J->max_seqlen + pos) * J->max_seqlen + j];\n"
     "    double p = silu(x);"),
    # queries with fewer rows than keys (Inputs and Outputs table: seq_offsets_q/k)
    ("delta_position_is_row", "const int64_t pos = L - Lq + i;", "const int64_t pos = i;"),
    ("delta_rab_row_local", "x += J->rab[(plane * J->max_seqlen + pos)",
     "x += J->rab[(plane * J->max_seqlen + i)"),
    ("delta_mask_row_local", "* J->max_seqlen + pos) * J->max_seqlen + j];\n    /* 5.",
     "* J->max_seqlen + i) * J->max_seqlen + j];\n    /* 5."),
    # KV cache pages (Inputs and Outputs table: kv_cache, page_offsets, page_ids, last_page_len)
    ("page_rows_reversed", "const int64_t row = j % J->page_size;",
     "const int64_t row = J->page_size - 1 - j % J->page_size;"),
    ("pages_reversed", "J->page_ids[J->page_offsets[b] + j / J->page_size]",
     "J->page_ids[J->page_offsets[b + 1] - 1 - j / J->page_size]"),
    ("kv_planes_swapped", "(((page * 2 + plane)", "(((page * 2 + 1 - plane)"),
    ("last_page_counted_full", "(pages - 1) * J->page_size + J->last_page_len[b]",
     "pages * J->page_size"),
    ("history_ignored", "  if (!J->kv_cache) return 0;\n  const int64_t pages", "  return 0;\n  const int64_t pages"),
]
# a real transposition: Q row j against K row i (query rows past Lq stay at i: in bounds)
MUTATIONS[0] = ("transposed_scores",
                "const double *kj = kv_row(J, b, hk, j, 0);",
                "const double *kj = kv_row(J, b, hk, i, 0);\n"
                "    qi = J->q + ((t0 + (j < Lq ? j : i)) * J->Nq + h) * D;")


def _pin_checks():
    checks = [pins.test_single_token_closed_forms, pins.test_silu_odd_part_identity,
              pins.test_q_zero_with_rab_closed_form, pins.test_jagged_lengths_match_torch_per_sequence,
              pins.test_count_valid_closed_forms, pins.test_q_zero_without_rab_gives_zero,
              pins.test_causal_rows_ignore_later_keys, pins.test_gqa_equals_replicated_mha,
              lambda: pins.test_q_zero_rab_per_head_and_broadcast_closed_form(1),
              lambda: pins.test_q_zero_rab_per_head_and_broadcast_closed_form(3),
              pins.test_custom_mask_closed_forms,
              pins.test_delta_queries_are_the_last_rows_of_the_full_forward,
              pins.test_delta_custom_mask_rows_follow_positions,
              pins.test_delta_paged_q_zero_closed_form,
              pins.test_count_valid_kv_closed_forms]
    for ps in (4, 8):
        checks.append(lambda a=ps: pins.test_paged_history_equals_contiguous_keys(a))
    for causal in (False, True):
        for nq, nk in ((4, 4), (4, 2), (6, 1)):
            checks.append(lambda c=causal, a=nq, b=nk: pins.test_equal_lengths_match_torch_matmul(c, a, b))
    for case in pins._cases():
        checks.append(lambda c=case: pins.test_mask_matrices_through_forward(c))
    return checks


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutant = src.replace(old, new)
    if name == "transposed_scores":
        mutant = mutant.replace("const double *qi = J->q", "const double *qi0 = J->q", 1)
        mutant = mutant.replace("const double *qi0 = J->q + ((t0 + i) * J->Nq + h) * D;",
                                "const double *qi0 = J->q + ((t0 + i) * J->Nq + h) * D;\n"
                                "  const double *qi = qi0;", 1)
    c = tmp_path / "mutant.c"
    c.write_text(mutant)
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(c),
                           "-lm", "-lpthread"])
    caught = 0
    with oracle.use_library(str(so)):
        for chk in _pin_checks():
            try:
                chk()
            except (AssertionError, ValueError):
                caught += 1
    assert caught > 0, f"no pin caught the planted mistake {name}"
