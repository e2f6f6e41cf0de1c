"""Each planted oracle mistake (ORC_MUTANT=n in oracle.c) must fail some pin.

This shows the pins are sharp enough: a dropped term, a flipped sign, a wrong
row index, an off-by-one in the inverse CDF, a wrong tie-break or a wrong
round count would not go unnoticed.  Mutants are built on the CPU into a
temporary directory; nothing here touches a GPU.
"""
import os
import shutil

import pytest

import oracle
import pins

# cheap pins first; the battery stops at the first failure
BATTERY = [
    pins.pin_softmax, pins.pin_argmax, pins.pin_topk, pins.pin_choice, pins.pin_uniform_mapping,
    pins.pin_greedy, pins.pin_toy_closed_forms, pins.pin_saguaro_bonus_position,
    pins.pin_saguaro_disjoint_supports, pins.pin_saguaro_equal_distributions, pins.pin_saguaro_clamp_order,
    pins.pin_low_temperature_limit, pins.pin_losslessness_random, pins.pin_losslessness_toy_chain,
    pins.pin_cache_hit_rate, pins.pin_draft_topk, pins.pin_saguaro_draft_lossless, pins.pin_top_p,
    pins.pin_philox_vs_triton,
]

MUTANTS = {
    1: "bonus drawn from target row gamma-1 (the toy driver's slip)",
    2: "residual sign flipped, (p - q)+",
    3: "accept ratio inverted, p(x)/q(x)",
    4: "inverse CDF off by one",
    5: "temperature ignored in the softmax",
    6: "Saguaro clamp applied to p_D instead of the residual",
    7: "top-k ties to the higher index",
    8: "Philox with 9 rounds",
    9: "Saguaro without the square root",
    10: "greedy argmax ties to the higher index",
    11: "cache check against the top-k of acceptance length n-1",
    12: "draft-logit top-k taken from the target row",
    13: "Saguaro-draft verification with the draft's p(x) in the accept test",
    14: "top-p truncating the target but not the draft",
    15: "Saguaro clamp applied to the residual before it is normalised",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_mutant_is_caught(mutant, tmp_path):
    if mutant == 8:
        pytest.importorskip("triton")
    if shutil.which("gcc") is None:
        pytest.skip("gcc missing")
    path = oracle.build(os.path.join(str(tmp_path), f"liboracle_m{mutant}.so"), mutant=mutant)
    o = oracle.load(path)
    assert o.mutant == mutant
    for pin in BATTERY:
        try:
            pin(o)
        except AssertionError:
            return
    pytest.fail(f"no pin caught mutant {mutant}: {MUTANTS[mutant]}")
