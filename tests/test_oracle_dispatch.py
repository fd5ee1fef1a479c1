"""Pins of the dispatch oracle (capacity, stable capacity-limited dispatch)."""
import numpy as np

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


def test_sharded_dispatch_reading():
    """The capacity of [P1] §4.5 is per batch.  A batch split into ranks in row
    order is dispatched as one: an assignment's slot is its rank among its own
    rank's assignments to the expert, after the expert's assignments on all
    lower ranks, dropped at C.  Checked against the whole batch's dispatch for
    several splits, including drops that start inside a rank."""
    rng = np.random.default_rng(7)
    E, k = 9, 3
    idx = np.stack([rng.choice(E, size=k, replace=False, p=None) for _ in range(400)])
    idx[:150, 0] = 4                                   # one hot expert, so its buffer fills on the first rank
    for cf in (0.3, 1.0, 2.0):
        C = oracle.dispatch.capacity(idx.shape[0], k, E, cf)
        whole = oracle.dispatch.dispatch(idx, E, C)
        for cuts in ([0, 400], [0, 1, 400], [0, 133, 250, 399, 400], [0, 100, 200, 300, 400]):
            slots = []
            for a, b in zip(cuts, cuts[1:]):
                below = np.bincount(idx[:a].ravel(), minlength=E)
                local = oracle.dispatch.dispatch(idx[a:b], E, 10 ** 9)["slot"]     # ranks within this rank, nothing dropped
                g = below[idx[a:b].ravel()] + local
                slots.append(np.where(g < C, g, -1))
            assert np.array_equal(np.concatenate(slots), whole["slot"]), (cf, cuts)
