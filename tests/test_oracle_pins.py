"""The CPU oracle against what the pages and mathematics fix (no GPU needed)."""
import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def test_philox_matches_triton(orc):
    pytest.importorskip("triton")
    pins.pin_philox_vs_triton(orc)


def test_uniform_mapping(orc):
    pins.pin_uniform_mapping(orc)


def test_uniform_statistics(orc):
    pins.pin_uniform_statistics(orc)


def test_softmax(orc):
    pins.pin_softmax(orc)


def test_argmax(orc):
    pins.pin_argmax(orc)


def test_topk(orc):
    pins.pin_topk(orc)


def test_choice(orc):
    pins.pin_choice(orc)


def test_toy_closed_forms(orc):
    pins.pin_toy_closed_forms(orc)


def test_losslessness_toy_chain(orc):
    pins.pin_losslessness_toy_chain(orc)


def test_losslessness_random(orc):
    pins.pin_losslessness_random(orc)


def test_greedy(orc):
    pins.pin_greedy(orc)


def test_low_temperature_limit(orc):
    pins.pin_low_temperature_limit(orc)


def test_expected_tokens(orc):
    pins.pin_expected_tokens(orc)


def test_toy_kl(orc):
    pins.pin_toy_kl(orc)


def test_speedup_formula():
    pins.pin_speedup_formula()


def test_saguaro_toy_topk(orc):
    pins.pin_saguaro_toy_topk(orc)


def test_saguaro_bonus_position(orc):
    pins.pin_saguaro_bonus_position(orc)


def test_saguaro_disjoint_supports(orc):
    pins.pin_saguaro_disjoint_supports(orc)


def test_saguaro_equal_distributions(orc):
    pins.pin_saguaro_equal_distributions(orc)


def test_cache_hit_rate(orc):
    pins.pin_cache_hit_rate(orc)


def test_draft_topk(orc):
    pins.pin_draft_topk(orc)


def test_saguaro_draft_lossless(orc):
    pins.pin_saguaro_draft_lossless(orc)


def test_top_p(orc):
    pins.pin_top_p(orc)


def test_saguaro_clamp_order(orc):
    pins.pin_saguaro_clamp_order(orc)


def test_draw_row(orc):
    pins.pin_draw_row(orc)
