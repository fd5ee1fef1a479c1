"""Pins of the TAOT Phase 1 Sinkhorn oracle."""

import numpy as np

import oracle
import pins


def _loads(B=12, R=64, seed=3):
    rng = np.random.default_rng(seed)
    loads = rng.poisson(384, size=(B, R)).astype(np.float64)
    loads[0] = 384.0                                   # all equal: no transfer
    loads[1, :8] += 600.0                              # one hot node
    return loads


def test_two_rank_closed_form():
    pins.check_sinkhorn_two_rank(oracle.sinkhorn)


def test_matches_independent_dual_solve():
    pins.check_sinkhorn_dual(oracle.sinkhorn)


def test_marginals_and_form():
    pins.check_sinkhorn_marginals(oracle.sinkhorn, _loads())


def test_topology_kernel_ratio():
    pins.check_sinkhorn_topology_kernel(oracle.sinkhorn)


def test_fifty_iterations_reach_the_fixed_point():
    loads = _loads(B=4, seed=5)
    a50 = oracle.sinkhorn.taot_phase1(loads, 8, 10.0, iters=50)
    a10k = oracle.sinkhorn.taot_phase1(loads, 8, 10.0, iters=10000)
    np.testing.assert_allclose(a50["plan"], a10k["plan"], rtol=1e-9, atol=1e-15)


def test_zero_mass_status():
    out = oracle.sinkhorn.taot_phase1(np.full((2, 16), 7.0), 8, 10.0)
    assert list(out["status"]) == [1, 1] and not out["plan"].any() and not out["u"].any()


def test_supply_demand_hand_cases():
    pins.check_supply_demand_hand(oracle.sinkhorn)


def test_topology_cost_hand_case():
    pins.check_topology_cost_hand(oracle.sinkhorn)
