"""GPU parity of the EPLB planner ([P3] §4.1.2) through the C ABI against the
CPU oracle: the physical-slot map, the copy counts and the GPU loads must all
match bit for bit (the replication compares integers exactly, and the packing
takes its decisions and sums in the same fp32 arithmetic on both sides)."""

import numpy as np
import pytest
import torch

import synth
from oracle import eplb

pytestmark = pytest.mark.gpu

W = synth.EPLB_WORKLOADS["eplb-zipf-E384-B1024"]


@pytest.fixture(scope="module")
def mr(native_lib):
    import moe_expert_routing_router_gb300 as m
    return m


def run(mr, loads: np.ndarray, num_phys, num_gpus, num_nodes, num_groups):
    got = mr.moe_eplb_plan(torch.from_numpy(loads.astype(np.int32)).cuda(), num_phys, num_gpus, num_nodes, num_groups)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in got.items()}


def check(got: dict, loads: np.ndarray, num_phys, num_gpus, num_nodes, num_groups, rows=None) -> None:
    for b in (range(loads.shape[0]) if rows is None else rows):
        want = eplb.plan(loads[b], num_phys, num_gpus, num_nodes, num_groups)
        assert np.array_equal(got["phy2log"][b], want["phy2log"]), f"phy2log of problem {b}"
        assert np.array_equal(got["log_count"][b], want["log_count"]), f"log_count of problem {b}"
        g, w = got["gpu_load"][b], want["gpu_load"].astype(np.float32)
        assert np.array_equal(g.view(np.uint32), w.view(np.uint32)), f"gpu_load of problem {b}: {g} vs {w}"


@pytest.mark.parametrize("num_groups", [0, W.num_groups], ids=["global", "hierarchical"])
def test_full_workload(mr, num_groups):
    loads = synth.eplb_loads(W)
    got = run(mr, loads, W.num_phys, W.num_gpus, W.num_nodes, num_groups)
    check(got, loads, W.num_phys, W.num_gpus, W.num_nodes, num_groups)


@pytest.mark.parametrize("E,num_phys,num_gpus,num_nodes,num_groups", [
    (8, 8, 1, 1, 0),            # no replication, one GPU
    (1, 4, 4, 2, 1),            # one expert copied onto every slot; one group cannot split over 2 nodes: global
    (48, 64, 16, 4, 8),         # hierarchical
    (48, 96, 12, 3, 6),         # three nodes, hierarchical
    (40, 40, 8, 8, 5),          # groups not divisible by nodes: global
    (1024, 4096, 256, 32, 64),  # the largest sizes, hierarchical
    (1024, 4096, 256, 1, 0),    # the largest sizes, global
    (256, 320, 64, 8, 0),
])
def test_shapes(mr, E, num_phys, num_gpus, num_nodes, num_groups):
    rng = np.random.default_rng(E + num_phys)
    loads = rng.integers(0, 5000, size=(6, E))
    loads[1] = 0                                         # nothing routed: ties everywhere
    loads[2] = 7                                         # equal loads
    loads[3, :] = rng.integers(0, 3, size=E)            # heavy ties
    loads[4, 0] = 2 ** 30                                # one expert far above the rest (64-bit products)
    got = run(mr, loads, num_phys, num_gpus, num_nodes, num_groups)
    check(got, loads, num_phys, num_gpus, num_nodes, num_groups)


def test_worked_example_through_the_abi(mr):
    """Four groups of one expert each, loads [9, 7, 5, 3], onto 2 nodes of one GPU
    (2 slots each), no replication: the nodes get {9, 3} and {7, 5}, 12 / 12."""
    got = run(mr, np.array([[9, 7, 5, 3]]), 4, 2, 2, 4)
    assert got["phy2log"][0].tolist() == [0, 3, 1, 2]
    assert got["gpu_load"][0].tolist() == [12.0, 12.0]
    assert got["log_count"][0].tolist() == [1, 1, 1, 1]
