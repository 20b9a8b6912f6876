"""Planted mistakes in the oracle must be caught by its pins (no GPU).

Each mutant is a copy of oracle/bsattn_oracle.c with one plausible mistake (a
dropped term, a wrong sign, an off-by-one, a transposed operand, a wrong
index), compiled into a temporary library.  The pins of test_oracle.py are run
against it and at least one must fail.  The real oracle is restored afterwards.
"""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle as T

MUTANTS = {
    "causal_strict": ("case KIND_CAUSAL: return j <= i;", "case KIND_CAUSAL: return j < i;"),
    "window_off_by_one": ("i - j < p->window_left", "i - j <= p->window_left"),
    "sink_off_by_one": ("j < p->sink_tokens", "j <= p->sink_tokens"),
    "prefix_and": ("return j < p->prefix_len || j <= i;", "return j < p->prefix_len && j <= i;"),
    "ascending_lists": ("for (int64_t n = nn - 1; n >= 0; --n) {",
                        "for (int64_t n = 0; n < nn; ++n) {"),
    "zero_padding": ("mt->full_idx[idx_at + e] = -1;", "mt->full_idx[idx_at + e] = 0;"),
    "lse_drops_max": ("*lse = mx + log(sum);", "*lse = log(sum);"),
    "scale_dropped": ("sc->s[t] = c->scale * dot;", "sc->s[t] = dot;"),
    "scores_use_v": ("const uint16_t *kj = c->k +", "const uint16_t *kj = c->v +"),
    "valid_len_off_by_one": ("n * p->tile_n >= p->kv_valid_len", "n * p->tile_n > p->kv_valid_len"),
    "all_selected_full": ("if (some && all) mt->full_idx", "if (some) mt->full_idx"),
    "full_tile_ignores_seqlen": ("j < (n + 1) * p->tile_n && j < sk; ++j) sc->keys",
                                 "j < (n + 1) * p->tile_n; ++j) sc->keys"),
    "offsets_sum_num_n": ("cn += num_m_of(p, b) * num_n_of(p, b);", "cn += num_n_of(p, b);"),
    "varlen_row_stride": ("mt->cu_block_idx_offsets[b] + m * num_n_of(p, b);",
                          "mt->cu_block_idx_offsets[b] + m * p->num_n;"),
    "softmax_weight_sign": ("double w = exp(sc->s[t] - mx) / sum;",
                            "double w = exp(mx - sc->s[t]) / sum;"),
    "head_index": ("const uint16_t *qi = c->q + ((int64_t)tok * H + h) * D;",
                   "const uint16_t *qi = c->q + ((int64_t)tok * H) * D;"),
}

PINS = [
    (T.test_worked_example_reversed_list, {}),
    (T.test_tiny_walk_example, {}),
    (T.test_varlen_offsets_hand_worked, {}),
    (T.test_varlen_identities_random_lengths, {"seed": 0}),
    (T.test_config1_lists, {}),
    (T.test_all_ones_map_equals_library_attention, {"kind": 0, "causal": False}),
    (T.test_all_ones_map_equals_library_attention, {"kind": 1, "causal": True}),
    (T.test_sliding_window_of_one_is_identity, {}),
    (T.test_window_of_one_with_sinks_is_library_attention_on_gathered_keys, {"sinks": 5}),
    (T.test_prefix_extremes_equal_library, {"prefix": 0, "causal": True}),
    (T.test_valid_length_one_is_strided_library_attention, {}),
    (T.test_partial_tail_tile_never_full, {}),
    (T.test_empty_rows_give_zero_and_minus_inf, {}),
    (T.test_full_list_tile_past_seqlen_is_clipped, {}),
] + [(T.test_meta_classification_matches_dense_predicate, {"case": i})
     for i in range(len(T.META_CASES))] + [
    (T.test_fwd_matches_dense_bruteforce, {"case": i}) for i in (2, 3)]


@pytest.fixture(scope="module")
def restore_oracle():
    yield
    oracle._use_library(None)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path, restore_oracle):
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = str(tmp_path / f"libmutant_{name}.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-o", lib, str(path),
                    "-lm", "-lpthread"], check=True)
    oracle._use_library(lib)
    try:
        caught = []
        for fn, kw in PINS:
            try:
                fn(**kw)
            except (AssertionError, ValueError):
                caught.append(fn.__name__)
                break
        assert caught, f"no pin caught the planted mistake {name}"
    finally:
        oracle._use_library(None)
