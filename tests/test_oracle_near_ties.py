"""Pins of the oracle's near-tie flags.

A float32 implementation may decide differently from the double-precision
oracle only where a decision margin is below its rounding, so the oracle flags
a request when (1) an accept test at a tested position (0..n, every position
when all drafts pass) has |r - min(1, p/q)| <= 1e-5 * max(r, min(1, p/q)), or
(2) the race that draws the extra token has its two best keys within 1e-5
relative.  (The vllbc page's Appendix A.1 remarks that floating-point
implementations are equivalent in distribution, not bit for bit; the 1e-5
margin is the benchmark's tolerance for such rows.)

Every case below is built around the 1e-5 boundary, with a margin of 0.6e-5 on
the flagged side and 1.5e-5 on the other, so that a wrong threshold, a flag
taken at an untested position, or a second-best key not updated when the best
changes fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle

NEAR = 0.6e-5       # relative margin that must be flagged
FAR = 1.5e-5        # relative margin that must not be flagged


def _run(tgt, q, ids, gammas, seed, T=1.0):
    tgt = np.asarray(tgt, np.float32)
    q = None if q is None else np.asarray(q, np.float32)
    cu = np.concatenate([[0], np.cumsum(gammas)]).astype(np.int32)
    return oracle.rejection_sample(tgt, q, np.asarray(ids, np.int32), cu, T, seed)


def _two_way_row(a):
    """Logits (0, L) whose softmax gives p(1) = a / 2 (q = (1/2, 1/2) then makes
    p(1)/q(1) = a), and the ratio the stored float32 logits actually give."""
    L = np.float32(math.log(a / (2.0 - a)))
    p1 = math.exp(float(L)) / (1.0 + math.exp(float(L)))
    return [0.0, float(L)], 2.0 * p1


def _seed_with_r(lo, hi, pos=0, b=0):
    """A seed whose accept uniform at (b, pos) lies in (lo, hi)."""
    for seed in range(10000):
        r = oracle.uniform(seed, b, pos, 0, 0, 1)[0]
        if lo < r < hi:
            return seed, r
    raise AssertionError("no seed found")


@pytest.mark.parametrize("side", [+1, -1])
@pytest.mark.parametrize("margin,flag", [(NEAR, 1), (FAR, 0)])
def test_accept_margin_at_the_first_position(side, margin, flag):
    # ratio a = r (1 + side * margin): side +1 accepts (r < a), side -1 rejects
    # and position 0 is then the first rejection, still a tested position
    seed, r = _seed_with_r(0.2, 0.8)
    row, a = _two_way_row(r * (1.0 + side * margin))
    rel = abs(r - a) / max(r, a)
    assert abs(rel - margin) < 0.1e-5          # the stored logits keep the margin
    res = _run([row, [0.0, 0.0]], [[0.5, 0.5]], [1], [1], seed)
    assert res.accept[0] == (1 if side > 0 else 0)
    assert res.pos_near_tie[0] == flag
    assert res.near_tie[0] == flag


@pytest.mark.parametrize("margin,flag", [(NEAR, 1), (FAR, 0)])
def test_accept_margin_after_accepted_positions_is_tested(margin, flag):
    # position 0 surely accepted (q(x) <= p(x)), position 1 near its margin:
    # position 1 is tested, so the request is flagged exactly when it is near
    seed, r = _seed_with_r(0.2, 0.8, pos=1)
    assert oracle.uniform(seed, 0, 0, 0, 0, 1)[0] < 0.999
    row1, _ = _two_way_row(r * (1.0 + margin))
    tgt = [[0.0, 1.0], row1, [0.0, 0.0]]
    res = _run(tgt, [[0.5, 0.5], [0.5, 0.5]], [1, 1], [2], seed)
    assert res.accept[0] == 1 and res.accept[1] == 1
    assert res.num_accepted[0] == 2
    assert list(res.pos_near_tie) == [0, flag]
    assert res.near_tie[0] == flag


def test_accept_margin_after_the_first_rejection_is_not_tested():
    # position 0 surely rejected (p(x) = 0); a near margin at position 1 is
    # recorded for that position but does not flag the request
    seed, r = _seed_with_r(0.2, 0.8, pos=1)
    row1, _ = _two_way_row(r * (1.0 + NEAR))
    tgt = [[0.0, -np.inf], row1, [0.0, 0.0]]
    res = _run(tgt, [[0.5, 0.5], [0.5, 0.5]], [1, 1], [2], seed)
    assert res.num_accepted[0] == 0
    assert list(res.pos_near_tie) == [0, 1]
    assert res.near_tie[0] == 0


def _race_row(ratios, E, base=0.0):
    """Logits whose race keys p(v)/E_v stand in the given ratios to key 0
    (ratio None: the entry is masked out, w = 0)."""
    row = []
    for v, k in enumerate(ratios):
        row.append(-np.inf if k is None else base + math.log(k * E[v] / E[0]))
    return np.asarray(row, np.float32)


def _realized_keys(row, E, T=1.0):
    l = row.astype(np.float64)
    w = np.exp((l - l.max()) / T)
    with np.errstate(invalid="ignore", divide="ignore"):
        return np.where(w > 0, w / E, -np.inf)


def _race_seed(pos, n):
    """A seed whose race exponentials at output position pos are all in
    [0.3, 3], so the key ratios above need only moderate logits."""
    for seed in range(10000):
        E = -np.log(oracle.uniform(seed, 0, pos, 1, 0, n))
        if E.min() > 0.3 and E.max() < 3.0:
            return seed, E
    raise AssertionError("no seed found")


# keys relative to key 0: the best changes at v = 1 (k2 is the old best);
# a later entry becomes second (k2 updated without a new best); the best
# changes at v = 2 while the old best, not entry 1, becomes second
RACE_CASES = [
    ("best changes", lambda d: [1.0, 1.0 + d, 0.5]),
    ("second arrives later", lambda d: [1.0 + d, 0.5, 1.0]),
    ("old best becomes second", lambda d: [1.0, 0.5, 1.0 + d]),
    ("masked entries do not compete", lambda d: [1.0, None, 1.0 + d, None]),
]


@pytest.mark.parametrize("name,keys", RACE_CASES, ids=[c[0] for c in RACE_CASES])
@pytest.mark.parametrize("margin,flag", [(NEAR, 1), (FAR, 0)])
def test_bonus_race_top_two(name, keys, margin, flag):
    ratios = keys(margin)
    seed, E = _race_seed(0, len(ratios))
    row = _race_row(ratios, E)
    k = np.sort(_realized_keys(row, E))[::-1]
    assert abs((k[0] - k[1]) / k[0] - margin / (1 + margin)) < 0.1e-5
    res = _run([row], np.zeros((0, len(ratios))), [], [0], seed)   # gamma = 0: bonus only
    best = int(np.argmax(_realized_keys(row, E)))
    assert res.tokens[0] == best
    assert res.near_tie[0] == flag


@pytest.mark.parametrize("margin,flag", [(NEAR, 1), (FAR, 0)])
def test_correction_race_over_the_residual(margin, flag):
    # position 0 is surely rejected (p(x) = 0 at x = 3); the residual
    # max(0, p - q) with q = onehot(3) is p on entries 0..2; its race keys are
    # built around the boundary.  The bonus row's race is never run.
    seed, E = _race_seed(0, 4)
    row0 = _race_row([1.0, 0.5, 1.0 + margin, None], E)
    q = [[0.0, 0.0, 0.0, 1.0]]
    res = _run([row0, [0.0, 0.0, 0.0, 0.0]], q, [3], [1], seed)
    assert res.num_accepted[0] == 0
    assert res.tokens[0] == 2 and res.tokens[1] == -1
    assert res.near_tie[0] == flag


def test_race_tie_in_a_row_that_is_not_drawn_does_not_flag():
    # position 0 surely rejected with well separated residual keys; the bonus
    # row would be a near tie but its race is not run
    seed, E0 = _race_seed(0, 4)
    E1 = -np.log(oracle.uniform(seed, 0, 1, 1, 0, 4))
    row0 = _race_row([1.0, 0.5, 2.0, None], E0)
    row1 = _race_row([1.0, 1.0 + NEAR, 0.5, 0.25], E1)
    res = _run([row0, row1], [[0.0, 0.0, 0.0, 1.0]], [3], [1], seed)
    assert res.num_accepted[0] == 0 and res.tokens[0] == 2
    assert res.near_tie[0] == 0
    # the same bonus row drawn (gamma = 0) is flagged
    seed1 = seed
    E = -np.log(oracle.uniform(seed1, 0, 0, 1, 0, 4))
    row = _race_row([1.0, 1.0 + NEAR, 0.5, 0.25], E)
    res = _run([row], np.zeros((0, 4)), [], [0], seed1)
    assert res.near_tie[0] == 1


def test_flags_are_per_request_in_a_batch():
    # two requests; only the second one's race is near a tie
    seed, E = _race_seed(0, 3)
    far = _race_row([1.0, 0.5, 0.25], E)
    E_b1 = -np.log(oracle.uniform(seed, 1, 0, 1, 0, 3))
    near = _race_row([1.0, 1.0 + NEAR, 0.5], E_b1)
    res = _run([far, near], np.zeros((0, 3)), [], [0, 0], seed)
    assert list(res.near_tie) == [0, 1]
