"""Pins of oracle/budget.py against the figures the pages print and against enumeration."""
import json
import math
import os
from fractions import Fraction

import pytest

from oracle import budget

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))
GIB = 1 << 30


def test_bytes_per_token_printed():
    g = GOLD["bytes_per_token"]
    assert budget.kv_bytes_per_token(g["layers"], g["kv_heads"], g["head_dim"], g["bytes_per_scalar"]) == g["value"]
    assert g["value"] == 128 * 1024


def test_request_4096_tokens():
    g = GOLD["request_4096_gib"]
    assert budget.kv_bytes([g["tokens"]], 32, 8, 128, 2) == g["value_gib"] * GIB
    assert budget.kv_bytes([g["tokens"]], 32, 32, 128, 2) == g["with_32_kv_heads_gib"] * GIB


def test_worked_example_40_layers():
    g = GOLD["worked_example_40_layers"]
    per = budget.kv_bytes_per_token(g["layers"], g["kv_heads"], g["head_dim"], g["bytes_per_scalar"])
    assert per == g["bytes_per_position"]
    assert budget.kv_bytes([g["positions"]], 40, 8, 128, 2) == g["bytes_per_sequence"] == g["gib_per_sequence"] * GIB
    six = budget.kv_bytes([g["positions"]] * g["sequences"], 40, 8, 128, 2)
    assert six == g["bytes_six"] == g["gib_six"] * GIB
    # doubling the retained length doubles the term; 8 -> 40 KV heads multiplies it by 5
    assert budget.kv_bytes([2 * g["positions"]], 40, 8, 128, 2) == 2 * g["bytes_per_sequence"]
    assert budget.kv_bytes_per_token(40, 40, 128, 2) == g["heads_8_to_40_factor"] * per


def test_ragged_batch_uses_sum_of_lengths():
    # P4: for unequal lengths without padding, B x T becomes the sum of stored positions
    ls = [3, 1000, 17, 4096]
    assert budget.kv_bytes(ls, 32, 8, 128, 2) == 131072 * sum(ls)
    assert budget.kv_bytes([], 32, 8, 128, 2) == 0


def test_pages_for_500_tokens():
    g = GOLD["pages_for_500"]
    assert budget.pages(g["tokens"], g["page_tokens"]) == g["pages"]
    assert budget.tail_slots(500, 16) == 12


@pytest.mark.parametrize("B", [1, 2, 3, 7, 16, 32, 100])
def test_tail_within_one_page(B):
    for T in range(1, 700):
        t = budget.tail_slots(T, B)
        assert 0 <= t <= B - 1
        assert (T + t) % B == 0
        assert budget.allocated_slots(T, B) >= T
    assert budget.pages(0, B) == 0 and budget.tail_slots(0, B) == 0


def test_mean_tail_closed_form():
    g = GOLD["tail_waste"]
    for k in range(10):
        B = 1 << k
        assert budget.mean_tail_uniform(g["n_max"], B) == Fraction(B - 1, 2)
    assert budget.mean_reservation_waste(g["n_max"], g["reservation"]) == Fraction(g["reservation_mean_waste"])
    # the "~8 tokens" of the 16-token example is the exact 7.5 rounded
    assert round(float(budget.mean_tail_uniform(512, 16))) == GOLD["pages_for_500"]["approx_mean_waste_tokens"]


def test_reservation_and_utilisation_figures():
    g = GOLD["reservation_2048"]
    unused = 1 - budget.utilisation_reserved([g["average"]], g["reserved"])
    assert unused > g["unused_more_than"]
    u = GOLD["utilisation"]
    naive = float(budget.utilisation_reserved([500], 2048))
    assert abs(naive - u["naive_about"]) < 0.005
    paged_single = float(budget.utilisation_paged([500], 16))
    paged_mean_tail = 500 / (500 + 7.5)
    assert paged_single == 500 / 512
    assert u["paged_band"][0] - 0.005 <= paged_mean_tail <= u["paged_band"][1]
    assert abs(100 * (paged_mean_tail - naive) - u["gap_points_about"]) < 1.0
