"""bench.py's host arithmetic: the algorithmic bytes each launch must move and
the committed DRAM-traffic table it reads."""

import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))

import bench  # noqa: E402
import synth  # noqa: E402


def test_algorithmic_bytes_per_launch():
    # logits read once + fp32 dlogits written + 16 bytes per assignment (idx, gate, perm, slot)
    want = {"switch-top1-T4096-E8": 327_680, "zipf-top2-T65536-E64": 27_262_976,
            "zipf-hot-top8-T131072-E256": 218_103_808, "zipf-ep64-top6-T262144-E384": 629_145_600}
    for name, b in want.items():
        assert bench.algorithmic_bytes(synth.ROUTER_WORKLOADS[name]) == b


def test_traffic_table_parses_and_matches_its_hash():
    lines = [ln.split() for ln in (ROOT / "profiles" / "router_step_dram_traffic.txt").read_text().splitlines()
             if ln.startswith("workload ")]
    assert {f[1] for f in lines} == {"zipf-top2-T65536-E64", "zipf-hot-top8-T131072-E256", "zipf-ep64-top6-T262144-E384"}
    for f in lines:
        assert f[2] == "read_bytes" and f[4] == "write_bytes" and f[6] == "source_hash"
        assert int(f[3]) > 0 and int(f[5]) >= 0 and len(f[7]) == 16
    # bench reports a row only while the kernel sources hash to the row's value
    cur = bench.kernel_source_hash()
    for f in lines:
        got = bench.measured_traffic(f[1])
        assert (got is not None) == (f[7] == cur)


def test_replay_plan_times_exactly_k_steps():
    # (steps per graph, replays, buffer sets): replays * steps per graph == K, >= 10 replays where K allows,
    # and the buffer sets divide the steps per graph
    assert bench.replay_plan(200, 2) == (20, 10, 2)
    assert bench.replay_plan(200, 15) == (20, 10, 20)
    assert bench.replay_plan(20, 2) == (2, 10, 2)
    assert bench.replay_plan(200, 1184) == (200, 1, 1184)
    assert bench.replay_plan(7, 2) == (7, 1, 2)
    for K in (10, 12, 50, 97, 200, 256):
        for n_min in (1, 2, 3, 15):
            S, R, n = bench.replay_plan(K, n_min)
            assert S * R == K and n >= n_min
            assert R == 1 or S % n == 0


def test_percentile_interpolates():
    xs = [5.0, 1.0, 3.0, 2.0, 4.0]
    assert bench.percentile(xs, 0.5) == 3.0
    assert bench.percentile(xs, 0.0) == 1.0 and bench.percentile(xs, 1.0) == 5.0
    assert abs(bench.percentile(xs, 0.1) - 1.4) < 1e-12
    assert bench.percentile([2.5], 0.9) == 2.5
