"""The pins are strong enough: a copy of the oracle with one plausible mistake
planted in it (on the CPU, in a temporary build) must fail at least one pin.

Each mutant is a textual edit of the committed C source; the committed oracle is
never modified.
"""
import pytest

import oracle
from tests import test_oracle_golden as golden
from tests import test_oracle_pins as pins

MUTANTS = {
    # values taken from the rope end of the key instead of the latent prefix
    "values_from_wrong_dims": ("o[j] += w * bf16_to_double(v[j]);",
                               "o[j] += w * bf16_to_double(v[j + (d_qk - d_v)]);"),
    # softmax temperature dropped
    "scale_dropped": ("s[t - lo] = scale * acc;", "s[t - lo] = acc;"),
    # wrong sign inside the exponent
    "exponent_sign": ("double w = exp(s[t - lo] - M);", "double w = exp(M - s[t - lo]);"),
    # log-sum-exp without the max shift added back
    "lse_missing_max": ("lse[(int64_t)r * H + h] = M + log(Z);", "lse[(int64_t)r * H + h] = log(Z);"),
    # transposed head index (reads another head's query)
    "wrong_query_head": ("const uint16_t* qrow = q + ((int64_t)r * H + h) * d_qk;",
                         "const uint16_t* qrow = q + ((int64_t)r * H + (H - 1 - h)) * d_qk;"),
    # value gathered from the neighbouring slot of the page
    "value_slot_off_by_one": ("const uint16_t* v = pool + (((int64_t)page * Hkv + kvh) * P + t % P) * d_qk;",
                              "const uint16_t* v = pool + (((int64_t)page * Hkv + kvh) * P + (t + 1) % P) * d_qk;"),
    # query heads mapped to KV heads round-robin instead of in contiguous groups
    "wrong_kv_head": ("const int kvh = h / group;", "const int kvh = h % Hkv;"),
    # merge forgets to normalise by the summed weights
    "merge_unnormalised": ("for (int j = 0; j < d_v; ++j) o[j] /= W;", ""),
    # merge weights not taken relative to the max (exp(lse) directly, wrong when M != 0)
    "merge_lse_without_max": ("lse[row] = M + log(W);", "lse[row] = log(W);"),
    # first token of every range skipped
    "range_skips_first_token": ("for (int64_t t = lo; t < hi; ++t) {\n                int32_t page",
                                "for (int64_t t = lo + 1; t < hi; ++t) {\n                int32_t page"),
    # migration copies half a page
    "migrate_half_page": ("(size_t)page_bytes);", "(size_t)page_bytes / 2);"),
}


def _checks():
    return [
        pins.test_single_token_returns_its_value,
        pins.test_zero_query_gives_mean_of_values_and_log_count,
        pins.test_equal_scores_through_rope_dims_only,
        pins.test_two_tokens_sigmoid_weights,
        pins.test_dominant_token_wins,
        lambda: pins.test_matches_torch_sdpa_float64([1, 17, 40], 5, 16),
        lambda: pins.test_gqa_matches_torch_sdpa_float64([1, 17, 40], 8, 2, 16),
        lambda: pins.test_cp_token_ranges_merge_to_unsplit(2),
        pins.test_merge_weights_closed_form,
        pins.test_merge_equal_parts_adds_ln2,
        pins.test_migrate_copies_bytes_and_touches_nothing_else,
        pins.test_migrated_pages_decode_identically,
        golden.test_merge_fixture,
    ] + [(lambda p=p: golden.test_attention_fixture(p)) for p in golden.ATTN]


def test_unmutated_source_passes_every_check():
    for chk in _checks():
        chk()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    so = oracle.compile_variant(src.replace(old, new), str(tmp_path), name)
    mutant = oracle.OracleLib(so)
    monkeypatch.setattr(oracle, "_lib", mutant.lib)
    failures = 0
    for chk in _checks():
        try:
            chk()
        except (AssertionError, ValueError):
            failures += 1
    assert failures >= 1, f"no pin caught the planted mistake '{name}'"
