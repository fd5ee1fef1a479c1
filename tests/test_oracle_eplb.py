"""Pins of the EPLB oracle ([P3] §4.1.2): the worked packing example, closed
forms, brute-force optimality of the replication and the plans' invariants."""

import pins
from oracle import eplb


def test_packing_worked_example():
    pins.check_packing_worked_example(eplb)


def test_packing_equal_weights():
    pins.check_packing_equal_weights_round_robin(eplb)


def test_packing_cardinality_and_mass():
    pins.check_packing_cardinality_and_mass(eplb)


def test_replication_bruteforce():
    pins.check_replication_bruteforce(eplb)


def test_replication_hand_case():
    pins.check_replication_hand_case(eplb)


def test_plan_invariants():
    pins.check_plan_invariants(eplb)


def test_plan_hand_cases():
    pins.check_plan_hand_cases(eplb)
