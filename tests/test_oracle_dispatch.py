"""Pins of the dispatch oracle (capacity, stable capacity-limited dispatch)."""

import oracle
import synth
import pins


def test_capacity_worked_example():
    pins.check_capacity_example(oracle.dispatch)


def test_capacity_of_the_workloads():
    # ceil(ceil(T*k/E) * factor) on the four router workloads
    want = {"switch-top1-T4096-E8": 640, "zipf-top2-T65536-E64": 2560,
            "zipf-hot-top8-T131072-E256": 4096, "zipf-ep64-top6-T262144-E384": 5120}
    for name, C in want.items():
        w = synth.ROUTER_WORKLOADS[name]
        assert oracle.dispatch.capacity(w.T, w.k, w.E, w.capacity_factor) == C


def test_dispatch_bruteforce():
    pins.check_dispatch_bruteforce(oracle.dispatch, oracle.router)


def test_dispatch_identities_with_drops():
    pins.check_dispatch_identities(oracle.dispatch, oracle.router, synth)
