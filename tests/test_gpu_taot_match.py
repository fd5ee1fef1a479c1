"""GPU parity of TAOT Phase 2 matching ([P4] §2, §3) through the C ABI against
the CPU oracle: replica slots, tokens per slot and rank loads bit-exact (the
decisions are integer comparisons plus fp32 comparisons of the given plan).
The Phase 1 plans fed to both sides come from the oracle's Sinkhorn."""

import numpy as np
import pytest
import torch

import oracle_pool
import synth
from oracle import sinkhorn, taot_match

pytestmark = pytest.mark.gpu

W = synth.EPLB_WORKLOADS["eplb-zipf-E384-B1024"]
R, RPN, K = 64, 8, 4


@pytest.fixture(scope="module")
def mr(native_lib):
    import moe_expert_routing_router_gb300 as m
    return m


def oracle_plans(loads: np.ndarray, R: int, rpn: int) -> np.ndarray:
    rank = loads.reshape(loads.shape[0], R, -1).sum(axis=2).astype(np.float64)
    return np.asarray(sinkhorn.taot_phase1(rank, rpn, 10.0, None, 50)["plan"], dtype=np.float32)


def run(mr, loads, plans, rpn, k):
    got = mr.taot_match_batched(torch.from_numpy(loads.astype(np.int32)).cuda(),
                                torch.from_numpy(np.ascontiguousarray(plans)).cuda(), rpn, k)
    torch.cuda.synchronize()
    return {key: v.cpu().numpy() for key, v in got.items()}


def check(got, loads, plans, R, rpn, k, rows):
    for b in rows:
        want = taot_match.match(loads[b], plans[b], R, rpn, k)
        assert np.array_equal(got["slot_expert"][b], want["slot_expert"]), f"slot_expert of microbatch {b}"
        assert np.array_equal(got["slot_tokens"][b], want["slot_tokens"]), f"slot_tokens of microbatch {b}"
        assert np.array_equal(got["rank_load"][b], want["rank_load"]), f"rank_load of microbatch {b}"


def test_full_workload_every_microbatch(mr):
    """All 1024 microbatches on the GPU, as the benchmark runs them, each
    against the oracle (run in a process pool across the host's cores), and the
    plan's invariants on all of them."""
    loads = synth.eplb_loads(W)
    plans = oracle_plans(loads, R, RPN)
    got = run(mr, loads, plans, RPN, K)
    want = oracle_pool.match_all(loads, plans, R, RPN, K)
    for b, (se, st, rl) in enumerate(want):
        assert np.array_equal(got["slot_expert"][b], se), f"slot_expert of microbatch {b}"
        assert np.array_equal(got["slot_tokens"][b], st), f"slot_tokens of microbatch {b}"
        assert np.array_equal(got["rank_load"][b], rl), f"rank_load of microbatch {b}"
    before = loads.reshape(W.B, R, -1).sum(axis=2)
    total = before.sum(axis=1, keepdims=True)
    after = got["rank_load"]
    assert np.array_equal(after.sum(axis=1, keepdims=True), total)
    hot, cold = before * R > total, before * R < total
    assert np.all((after * R >= total) | ~hot) and np.all((after * R <= total) | ~cold)
    assert np.all((got["slot_expert"] >= 0) == (got["slot_tokens"] > 0))


@pytest.mark.parametrize("E,R_,rpn,k", [(384, 64, 8, 0), (8, 1, 1, 4), (64, 64, 8, 3), (96, 16, 4, 16),
                                        (1024, 64, 8, 16), (48, 8, 8, 2), (60, 12, 3, 5)])
def test_shapes(mr, E, R_, rpn, k):
    rng = np.random.default_rng(E + R_ + k)
    p = (np.arange(E) + 1.0) ** -1.3
    loads = np.stack([rng.multinomial(20 * E, p[rng.permutation(E)] / p.sum()) for _ in range(5)])
    loads[1] = 9                                        # balanced: nothing moves
    loads[2, :] = 0
    loads[2, 0] = 5000                                  # one expert holds everything
    plans = oracle_plans(loads, R_, rpn)
    plans[3] = 0.0                                      # every flow ties: the expert / rank order decides
    got = run(mr, loads, plans, rpn, k)
    check(got, loads, plans, R_, rpn, k, range(loads.shape[0]))


def test_hand_case_through_the_abi(mr):
    """Loads [10, 2, 2, 2] on four ranks of two nodes: the same-node rank wins
    round 1, the larger flow round 2, the last rank round 3; all end at 4."""
    plan = np.zeros((1, 4, 4), np.float32)
    plan[0, 0, 2], plan[0, 0, 3] = 0.25, 0.5
    got = run(mr, np.array([[10, 2, 2, 2]]), plan, 2, 3)
    assert got["slot_expert"][0, :, 0].tolist() == [-1, 0, 0, 0]
    assert got["rank_load"][0].tolist() == [4, 4, 4, 4]
