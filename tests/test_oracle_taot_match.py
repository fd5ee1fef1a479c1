"""Pins of the TAOT Phase 2 oracle ([P4] §2, §3): hand cases for the tokens a
match moves, the topology preference, the flow tie-break and the arbitration,
and invariants of the plan (the readings themselves stay unpinned)."""

import pins
from oracle import taot_match


def test_hand_single_cold_rank():
    pins.check_match_hand_single(taot_match)


def test_hand_arbitration_topology_and_flow():
    pins.check_match_hand_arbitration(taot_match)


def test_invariants():
    pins.check_match_invariants(taot_match)


def test_column_first_beats_row_first():
    from oracle import sinkhorn
    pins.check_match_column_first_claim(taot_match, sinkhorn)


def test_residual_imbalance_hand_cases():
    pins.check_residual_imbalance_hand(taot_match)
