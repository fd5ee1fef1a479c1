"""Host check of the extended forward's selection scheme (bias routing, [P1]
§4.3), restated in numpy for the 32-lane row layout of E = 384 (lane l holds
columns v*128 + 4*l + i, v < 3, i < 4): 32-bit keys of the biased scores (the
order-preserving image with its low 10 bits replaced by 1023 - column), each
lane's two largest keys, k rounds of the warp maximum, then the check the
kernel applies before it keeps the picks:

  * with bf16 logits and no bias the keys hold the whole scores, and the picks
    stand iff exactly k keys are at or above the k-th pick (no lane that ran
    out of cached keys hid one);
  * otherwise they stand iff exactly k keys have a value image at or above the
    k-th pick's (the count half) and no two picks share a value image (the
    duplicate half).

Wherever the check accepts a row, its picks must be the oracle's top-k of the
scores (ties to the lower expert), in order.  Rows are planted so that each
half of the check is the only thing standing between the rounds and a wrong
pick, and the same rows run with that half taken out must go wrong.
"""

import numpy as np
import pytest

import oracle
import synth

E, LPR, VW, NV = 384, 32, 4, 3
MASK = np.uint32(0xFFFFFC00)


def lane_columns() -> np.ndarray:
    """[32, 12] column of each lane's elements."""
    cols = np.empty((LPR, VW * NV), np.int64)
    for l in range(LPR):
        for v in range(NV):
            for i in range(VW):
                cols[l, v * VW + i] = v * LPR * VW + l * VW + i
    return cols


COLS = lane_columns()
LANE_OF = np.empty(E, np.int64)
LANE_OF[COLS.ravel()] = np.repeat(np.arange(LPR), VW * NV)


def images(s: np.ndarray) -> np.ndarray:
    """Order-preserving uint32 image of fp32 values, -0.0 folded into +0.0."""
    u = (np.asarray(s, np.float32) + np.float32(0.0)).astype(np.float32).view(np.uint32)
    return u ^ np.where(u >> np.uint32(31), np.uint32(0xFFFFFFFF), np.uint32(0x80000000))


def sel_keys(scores: np.ndarray) -> np.ndarray:
    """[rows, E] fp32 scores -> [rows, E] uint32 selection keys."""
    col = np.arange(E, dtype=np.uint32)
    return ((images(scores) | np.uint32(0x3FF)) - col[None, :]).astype(np.uint32)


def emulate(scores: np.ndarray, k: int, whole: bool, count_half: bool = True,
            dup_half: bool = True) -> tuple[np.ndarray, np.ndarray]:
    """The kernel's rounds and check: (picked columns [rows, k], accepted [rows]).
    `count_half` / `dup_half` False take that half of the check out."""
    keys = sel_keys(scores)
    srt = np.sort(keys[:, COLS], axis=2)
    m1, m2 = srt[:, :, -1].copy(), srt[:, :, -2].copy()
    picks = np.empty((scores.shape[0], k), np.uint32)
    for j in range(k):
        w = m1.max(axis=1)                                    # the warp maximum
        picks[:, j] = w
        won = m1 == w[:, None]
        m1 = np.where(won, m2, m1)
        m2 = np.where(won, np.uint32(0), m2)
    wk = picks[:, k - 1]
    thr = wk if whole else (wk & MASK)
    ok = np.ones(scores.shape[0], bool)
    if count_half:
        ok &= (keys >= thr[:, None]).sum(axis=1) == k
    if dup_half and not whole and k > 1:
        ok &= ~((picks[:, :-1] & MASK) == (picks[:, 1:] & MASK)).any(axis=1)
    cols = (np.uint32(1023) - (picks & np.uint32(0x3FF))).astype(np.int64)
    return cols, ok


def exact_picks(scores: np.ndarray, k: int) -> np.ndarray:
    """The oracle's top-k of the scores (descending, ties to the lower index)."""
    return oracle.router.top_k(scores.astype(np.float64), k)


def outcome(scores, k, whole, **halves):
    """(accepted, wrong) masks of the emulated rows against the oracle."""
    cols, ok = emulate(scores, k, whole, **halves)
    return ok, (cols != exact_picks(scores, k)).any(axis=1)


def check(scores: np.ndarray, k: int, whole: bool, min_accept: float) -> None:
    ok, wrong = outcome(scores, k, whole)
    bad = ok & wrong
    assert not bad.any(), f"{int(bad.sum())} accepted rows with wrong picks, first {np.flatnonzero(bad)[:5]}"
    assert ok.mean() >= min_accept, f"only {ok.mean():.3f} of the rows accepted"


def background(rng, rows: int) -> np.ndarray:
    """Scores in [-3, 3): below every planted pick."""
    return rng.uniform(-3.0, 3.0, size=(rows, E)).astype(np.float32)


def with_image_low_bits(x: float, low: int) -> np.float32:
    """A positive fp32 value whose bits agree with x's above bit 10, `low` below."""
    u = np.float32(x).view(np.uint32) & MASK
    return (u | np.uint32(low)).view(np.float32)


def plant_top(rng, rows: int, k: int, spread_lanes: bool):
    """Rows of background() with k + 1 values in [4, 8) planted, descending, at
    random columns (in distinct lanes if `spread_lanes`).  The values sit at
    least 0.04 apart, far more than 1024 ulps, so no two share a value image."""
    s = background(rng, rows)
    tops = np.empty((rows, k + 1), np.int64)
    for r in range(rows):
        if spread_lanes:
            lanes = rng.choice(LPR, size=k + 1, replace=False)
            tops[r] = [rng.choice(COLS[l]) for l in lanes]
        else:
            tops[r] = rng.choice(E, size=k + 1, replace=False)
        grid = np.sort(rng.choice(80, size=k + 1, replace=False))[::-1]
        vals = (4.0 + 0.05 * grid + rng.uniform(0.0, 0.01, size=k + 1)).astype(np.float32)
        s[r, tops[r]] = vals
    return s, tops


def test_bf16_images_keep_order_under_the_key():
    """Whole mode rests on this: every bf16 value's image has its low 10 bits all
    zero (positive) or all one (negative), so replacing them loses no order.
    Checked over all finite bf16 patterns, in value order."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    f = (bits << np.uint32(16)).view(np.float32)
    f = np.unique(f[np.isfinite(f)])                          # ascending, -0.0 == +0.0
    img = images(f)
    low = img & np.uint32(0x3FF)
    assert np.isin(low, [0, 0x3FF]).all()
    assert (np.diff((img | np.uint32(0x3FF)).astype(np.int64)) > 0).all()


@pytest.mark.parametrize("k", [1, 2, 6, 8])
def test_biased_workload_rows(k):
    """bf16 logits of the E = 384 workload plus a seeded fp32 bias: almost every
    row is accepted, and every accepted row is exact."""
    w = synth.ROUTER_WORKLOADS["zipf-ep64-top6-T262144-E384"].with_tokens(4000)
    z = oracle.router.widen(synth.router_logits(w), w.dtype).astype(np.float32)
    b = (np.random.default_rng(k).standard_normal(E) * 0.5).astype(np.float32)
    check((z + b[None, :]).astype(np.float32), k, whole=False, min_accept=0.9)


@pytest.mark.parametrize("k", [2, 6, 8])
def test_bf16_without_bias_is_whole(k):
    """bf16 logits and no bias: the keys hold the whole scores; ties between equal
    bf16 values are frequent and decided by the lower column, exactly."""
    w = synth.ROUTER_WORKLOADS["zipf-ep64-top6-T262144-E384"].with_tokens(4000)
    z = oracle.router.widen(synth.router_logits(w), w.dtype).astype(np.float32)
    check(z, k, whole=True, min_accept=0.97)


@pytest.mark.parametrize("k", [2, 8])
def test_integer_ties_whole(k):
    """Integer scores (exact in bf16): ties everywhere, including at the k-th
    pick, all decided by the lower column; rows whose lane ran out of cached
    keys are refused."""
    rng = np.random.default_rng(20 + k)
    s = rng.integers(-3, 4, size=(3000, E)).astype(np.float32)
    ok, wrong = outcome(s, k, whole=True)
    assert not (ok & wrong).any()
    assert 0.5 < ok.mean() <= 1.0


@pytest.mark.parametrize("k", [2, 6, 8])
def test_shared_image_inside_the_picks(k):
    """Two of the top k share a value image, the larger at the higher column: the
    count holds, the rounds put the pair in column order (wrong), and only the
    duplicate half refuses the row."""
    rng = np.random.default_rng(30 + k)
    s, tops = plant_top(rng, 400, k, spread_lanes=True)
    for r in range(s.shape[0]):
        j = rng.integers(0, k - 1)
        a, b = sorted(tops[r, j:j + 2])
        s[r, b] = with_image_low_bits(s[r, tops[r, j]], 0x200)
        s[r, a] = with_image_low_bits(s[r, tops[r, j]], 0x100)
    ok, wrong = outcome(s, k, whole=False)
    assert wrong.all() and not ok.any()
    ok_nodup, _ = outcome(s, k, whole=False, dup_half=False)
    assert ok_nodup.all()                                     # without that half, every wrong row stands


@pytest.mark.parametrize("k", [1, 2, 6, 8])
def test_shared_image_at_the_kth_pick(k):
    """The k-th and (k+1)-th scores share a value image, the larger at the higher
    column: the rounds pick the wrong one, and the count half refuses the row."""
    rng = np.random.default_rng(40 + k)
    s, tops = plant_top(rng, 400, k, spread_lanes=True)
    for r in range(s.shape[0]):
        a, b = sorted(tops[r, k - 1:k + 1])
        s[r, b] = with_image_low_bits(s[r, tops[r, k - 1]], 0x300)
        s[r, a] = with_image_low_bits(s[r, tops[r, k - 1]], 0x001)
    ok, wrong = outcome(s, k, whole=False)
    assert wrong.all() and not ok.any()
    ok_nocount, _ = outcome(s, k, whole=False, count_half=False)
    assert ok_nocount.all()


@pytest.mark.parametrize("whole", [False, True])
@pytest.mark.parametrize("k", [3, 6, 8])
def test_lane_out_of_cached_keys(k, whole):
    """Three of the top k in one lane (its two-deep cache runs out): the rounds
    pick wrongly, the count half refuses the row, and without it the row stands."""
    rng = np.random.default_rng(50 + k)
    s, tops = plant_top(rng, 400, k, spread_lanes=True)
    if whole:
        s = np.round(s * 32.0).astype(np.float32) / np.float32(32.0)  # exact in bf16, picks still distinct
    for r in range(s.shape[0]):
        lane = LANE_OF[tops[r, 0]]
        others = [c for c in COLS[lane] if c != tops[r, 0]]
        third = rng.choice(others, size=2, replace=False)
        vals = s[r, tops[r, 1:3]].copy()
        s[r, tops[r, 1:3]] = s[r, third]
        s[r, third] = vals                                    # picks 0..2 now in one lane
    ok, wrong = outcome(s, k, whole)
    assert wrong.all() and not ok.any()
    ok_nocount, _ = outcome(s, k, whole, count_half=False)
    assert ok_nocount.all()


@pytest.mark.parametrize("k", [2, 6, 8])
def test_mixed_rows_accept_only_exact(k):
    """Planted tops at random columns (lanes may hold several picks) plus
    near-equal pairs in a third of the rows: accepted and refused rows both
    occur, and every accepted row is exact."""
    rng = np.random.default_rng(60 + k)
    s, tops = plant_top(rng, 3000, k, spread_lanes=False)
    for r in range(0, s.shape[0], 3):
        j = rng.integers(0, k)
        c = rng.choice(np.setdiff1d(np.arange(E), tops[r]))
        s[r, c] = with_image_low_bits(s[r, tops[r, j]], int(rng.integers(0, 1024)))
    ok, wrong = outcome(s, k, whole=False)
    assert not (ok & wrong).any()
    assert 0.2 < ok.mean() < 1.0
