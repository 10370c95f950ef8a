"""Pins of the oracle's top-k / top-p adjusted target distribution (the vllbc
page's Section 2.2 note folds top-k and top-p into the adjusted p before the
same rejection test).  The kept set and its renormalisation are checked against
hand values, against a token-by-token evaluation of the definition on tiny rows
with planted ties, against the properties that make it the nucleus, and through
the output distribution of the whole verify step.  The band of reachable cuts
around the top-p edge (the group boundaries a float32 evaluation may decide the
other way) is checked on rows built around its 1e-5 boundary."""
import numpy as np
import pytest

import oracle
import stat_checks as sc


def _f32(x):
    return np.asarray(x, np.float32)


def _near_edge(l, T, k, P, rel=1e-12):
    """True when some group's larger-logit mass lies within `rel` of the top-p
    bound: there a different order of the double sums may decide the edge
    the other way, so the token-by-token evaluation is not a pin."""
    if P >= 1.0:
        return False
    l = np.asarray(l, np.float64)
    e = np.exp((l - l.max()) / T)
    V = len(l)
    in_k = np.ones(V, bool) if not (1 <= k < V) else np.array([(l > x).sum() < k for x in l])
    bound = max(P, 0.0) * e[in_k].sum()
    for x in np.unique(l[in_k]):
        a = e[l > x].sum()
        if a > 0 and abs(a - bound) <= rel * e[in_k].sum():
            return True
    return False


def test_closed_forms():
    # p = (1/2, 1/4, 1/8, 1/8) at T = 1
    l = _f32(np.log([4.0, 2.0, 1.0, 1.0]))
    cases = {
        (1, 1.0): [1, 0, 0, 0],
        (2, 1.0): [2 / 3, 1 / 3, 0, 0],
        (3, 1.0): [1 / 2, 1 / 4, 1 / 8, 1 / 8],    # the 3rd and 4th logits tie: both kept
        (0, 0.6): [2 / 3, 1 / 3, 0, 0],            # 1/2 < 0.6 <= 3/4
        (0, 0.4): [1, 0, 0, 0],                    # the top token alone reaches 0.4
        (0, 0.8): [1 / 2, 1 / 4, 1 / 8, 1 / 8],    # 3/4 < 0.8: the tied pair is kept whole
        (0, 0.0): [1, 0, 0, 0],                    # P <= 0 keeps the most probable tokens
        (2, 0.5): [1, 0, 0, 0],                    # top-2 gives (2/3, 1/3); 2/3 >= 0.5
        (2, 0.7): [2 / 3, 1 / 3, 0, 0],            # 2/3 < 0.7
        (4, 1.0): [1 / 2, 1 / 4, 1 / 8, 1 / 8],    # k >= V: off
        (-3, 1.5): [1 / 2, 1 / 4, 1 / 8, 1 / 8],   # k <= 0 and P >= 1: off
    }
    for (k, p), want in cases.items():
        got = oracle.adjusted_probs(l, 1.0, k, p)
        assert np.allclose(got, want, atol=1e-7, rtol=0), (k, p, got)


def test_temperature_applies_before_the_cut():
    # logits (0, ln 3): p = (1/4, 3/4) at T = 1 and (1/(1+sqrt 3), sqrt3/(1+sqrt 3)) at T = 2
    l = _f32([0.0, np.log(3.0)])
    got = oracle.adjusted_probs(l, 1.0, 0, 0.7)
    assert np.allclose(got, [0, 1])          # 3/4 >= 0.7 keeps the top token alone
    got = oracle.adjusted_probs(l, 2.0, 0, 0.7)
    assert np.allclose(got, [1 / (1 + np.sqrt(3)), np.sqrt(3) / (1 + np.sqrt(3))])  # 0.634 < 0.7


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    for _ in range(60):
        V = int(rng.integers(1, 10))
        l = rng.integers(-3, 4, size=V).astype(np.float32)   # many ties
        if V > 2 and rng.random() < 0.3:
            l[rng.integers(V)] = -np.inf
        if rng.random() < 0.3:
            l[l == 0] = -0.0                                   # -0 and +0 are one value
            l[: V // 2][l[: V // 2] == 0] = 0.0
        T = float(rng.choice([0.5, 1.0, 2.0]))
        k = int(rng.integers(-1, V + 2))
        p = float(rng.choice([0.0, 0.1, 0.33, 0.5, 0.77, 0.9, 0.999, 1.0, 1.2]))
        if _near_edge(l, T, k, p):
            continue
        got = oracle.adjusted_probs(l, T, k, p)
        want = sc.adjusted64(l, T, k, p)
        assert np.allclose(got, want, atol=1e-12, rtol=0), (l, T, k, p, got, want)


def test_bf16_rows_match_f32_rows_of_the_same_values():
    rng = np.random.default_rng(3)
    l = rng.normal(0, 2, size=64).astype(np.float32)
    bits = (l.view(np.uint32) >> 16).astype(np.uint16)           # truncation: exact bf16 values
    l16 = (bits.astype(np.uint32) << 16).view(np.float32)
    for k, p in [(5, 1.0), (0, 0.8), (10, 0.5)]:
        a = oracle.adjusted_probs(bits, 1.0, k, p, dtype="bf16")
        b = oracle.adjusted_probs(l16, 1.0, k, p)
        assert np.array_equal(a, b)


def test_nucleus_properties_on_large_rows():
    rng = np.random.default_rng(9)
    for trial in range(20):
        V = 5000
        l = (rng.normal(0, 3, size=V)).astype(np.float32)
        T = float(rng.choice([0.7, 1.0, 1.5]))
        k = int(rng.choice([0, 1, 7, 50, 1000, 4999]))
        P = float(rng.choice([0.3, 0.9, 0.99, 1.0]))
        if _near_edge(l, T, k, P):
            continue
        got = oracle.adjusted_probs(l, T, k, P)
        kept = got > 0
        assert abs(got.sum() - 1.0) < 1e-12
        # a top set: every kept logit is >= every dropped logit
        if (~kept).any():
            assert l[kept].min() >= l[~kept].max()
        e = np.exp((l.astype(np.float64) - l.max()) / T)
        p0 = e / e.sum()
        assert np.allclose(got[kept], p0[kept] / p0[kept].sum(), rtol=1e-12, atol=0)
        # top-k: fewer than k tokens above the smallest kept logit
        if 1 <= k < V:
            assert (l > l[kept].min()).sum() < k
        # top-p: the kept mass reaches P of the top-k mass; without the lowest kept
        # group it does not
        in_k = np.array([True] * V) if not (1 <= k < V) else (
            np.array([(l > x).sum() for x in l]) < k)
        s_k = e[in_k].sum()
        if P < 1:
            lo = l[kept].min()
            above = e[l > lo].sum()
            assert above == 0 or above < P * s_k
            if (in_k & ~kept).any():
                assert e[kept].sum() >= P * s_k


def test_switched_off_equals_the_plain_verifier():
    w_rng = np.random.default_rng(4)
    V, B, g = 50, 12, 3
    tgt = w_rng.normal(0, 2, size=(B * (g + 1), V)).astype(np.float32)
    q = w_rng.dirichlet(np.ones(V), size=B * g).astype(np.float32)
    ids = np.array([w_rng.choice(V, p=r / r.sum()) for r in q.astype(np.float64)], np.int32)
    cu = (np.arange(B + 1) * g).astype(np.int32)
    a = oracle.rejection_sample(tgt, q, ids, cu, 0.9, 7)
    b = oracle.rejection_sample(tgt, q, ids, cu, 0.9, 7, top_k=np.full(B, V), top_p=np.full(B, 1.0))
    for f in ("tokens", "num_accepted", "beta", "p_x", "accept"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f


def test_top_k_one_reproduces_greedy_tokens():
    # p' is one-hot at the argmax: a draft equal to it is accepted (ratio 1/q >= 1),
    # any other is rejected (p'(x) = 0) and the residual is the argmax alone.
    rng = np.random.default_rng(5)
    V, B, g = 40, 64, 4
    tgt = rng.normal(0, 2, size=(B * (g + 1), V)).astype(np.float32)
    q = rng.dirichlet(np.ones(V), size=B * g).astype(np.float32)
    am = tgt.reshape(B, g + 1, V)[:, :g].argmax(-1).reshape(-1)
    rnd = rng.integers(0, V, size=B * g)
    ids = np.where(rng.random(B * g) < 0.7, am, rnd).astype(np.int32)
    cu = (np.arange(B + 1) * g).astype(np.int32)
    greedy = oracle.rejection_sample(tgt, None, ids, cu, 0.0, 0)
    for T in (0.5, 1.0, 3.0):
        a = oracle.rejection_sample(tgt, q, ids, cu, T, 11, top_k=1)
        assert np.array_equal(a.tokens, greedy.tokens)
        assert np.array_equal(a.num_accepted, greedy.num_accepted)
        assert np.allclose(a.p_x, greedy.p_x)
        # a vanishing nucleus is the same cut
        b = oracle.rejection_sample(tgt, q, ids, cu, T, 11, top_p=1e-9)
        assert np.array_equal(b.tokens, greedy.tokens)


@pytest.mark.parametrize("top_k,top_p", [(3, 1.0), (0, 0.7), (5, 0.8)])
def test_output_distribution_follows_the_adjusted_target(top_k, top_p):
    def run(tgt, q, ids, cu, T, seed, k, p):
        r = oracle.rejection_sample(tgt, q, ids, cu, T, seed, top_k=k, top_p=p)
        assert r.status == 0
        return r.tokens, r.num_accepted, r.accept, r.beta
    out = sc.check_adjusted_distribution(run, top_k, top_p, n=300_000)
    assert out["slot0"] > sc.P_MIN
    assert out["residual"] > sc.P_MIN
    assert out["bonus"] > sc.P_MIN
    assert out["accept_z"] < 3.0
    assert out["beta_err"] < 1e-12


def test_a_planted_tie_exclusive_cut_is_caught():
    # cutting ties at the k-th logit by index (keeping exactly k tokens) is a
    # plausible mistake; the token-by-token definition keeps the whole group
    l = _f32([1.0, 2.0, 2.0, 0.0])
    got = oracle.adjusted_probs(l, 1.0, 1, 1.0)
    want = sc.adjusted64(l, 1.0, 1, 1.0)
    assert np.allclose(got, want) and np.allclose(got, [0, 0.5, 0.5, 0])
    exclusive = np.array([0, 1.0, 0, 0])
    assert not np.allclose(exclusive, want)


# ----------------------------------------------------------------------------
# The band of reachable top-p cuts
# ----------------------------------------------------------------------------

NEAR = 0.6e-5
FAR = 1.5e-5


def _masses(l, T=1.0):
    l = np.asarray(l, np.float64)
    return np.exp((l - l.max()) / T)


def _bound_at(l, g, rel, T=1.0):
    """A top-p value that puts P * S at A_g (1 + rel): A_g the mass of the
    first g groups of a row of distinct logits (largest first)."""
    e = np.sort(_masses(l, T))[::-1]
    a = e[:g].sum()
    return a * (1.0 + rel) / e.sum()


ROW = _f32(np.log([0.4, 0.3, 0.2, 0.1]))          # distinct logits, in order


@pytest.mark.parametrize("rel,expect", [(+NEAR, (-1, 0)), (-NEAR, (0, 1)), (+FAR, (0, 0)),
                                        (-FAR, (0, 0))])
def test_band_around_one_boundary(rel, expect):
    # P * S just above A_2 (the mass of groups 0 and 1): the exact cut keeps
    # group 2 (A_2 < P S) and, within the band, dropping it is reachable.  Just
    # below: the exact cut drops group 2 (A_2 >= P S) and keeping it is
    # reachable.
    P = _bound_at(ROW, 2, rel)
    p, rng = oracle.adjusted_probs(ROW, 1.0, 0, P, with_range=True)
    assert rng == expect
    kept = (p > 0).sum()
    assert kept == (3 if rel > 0 else 2)
    for s in range(expect[0], expect[1] + 1):
        ps = oracle.adjusted_probs(ROW, 1.0, 0, P, shift=s)
        assert (ps > 0).sum() == kept + s
        e = _masses(ROW)
        keep = ps > 0
        assert np.allclose(ps[keep], e[keep] / e[keep].sum(), rtol=1e-12, atol=0)
    for s in (expect[0] - 1, expect[1] + 1):
        with pytest.raises(ValueError):
            oracle.adjusted_probs(ROW, 1.0, 0, P, shift=s)


def test_band_spans_several_small_groups():
    # many light groups right at the bound: every cut among them is reachable
    light = [1e-6 * (1.06 - 0.01 * j) for j in range(6)]       # six distinct light logits
    l = _f32(np.log([0.5, 0.5 - 6.3e-6] + light))
    e = np.sort(_masses(l))[::-1]
    P = (e[:2].sum() + 3 * e[2]) / e.sum()        # the bound in the middle of the light groups
    p, (lo, hi) = oracle.adjusted_probs(l, 1.0, 0, P, with_range=True)
    assert lo <= -2 and hi >= 2
    base = (p > 0).sum()
    for s in range(lo, hi + 1):
        assert (oracle.adjusted_probs(l, 1.0, 0, P, shift=s) > 0).sum() == base + s


def test_no_band_without_a_positive_top_p():
    # top-k alone, P <= 0 and P >= 1 decide exactly: no shift is reachable
    for k, P in [(2, 1.0), (0, 0.0), (0, -0.5), (3, 0.0), (0, 1.0), (0, float("nan"))]:
        _, rng = oracle.adjusted_probs(ROW, 1.0, k, P, with_range=True)
        assert rng == (0, 0), (k, P)
        with pytest.raises(ValueError):
            oracle.adjusted_probs(ROW, 1.0, k, P, shift=1)


def test_band_is_relative_to_the_top_k_mass():
    # with top-k = 3 the bound is P times the mass of the first three groups;
    # a boundary within 1e-5 of it is in the band, one 1.5e-5 away is not
    e = np.sort(_masses(ROW))[::-1]
    for rel, expect in [(NEAR, (-1, 0)), (FAR, (0, 0))]:
        P = e[:2].sum() * (1 + rel) / e[:3].sum()
        _, rng = oracle.adjusted_probs(ROW, 1.0, 3, P, with_range=True)
        assert rng == expect


def test_request_under_a_shifted_cut():
    # the accept test at position 0 depends on whether the draft token's group
    # is kept: with the exact cut it is dropped (p'(x) = 0, rejected); with the
    # reachable shift +1 it is kept and accepted (q(x) = p'(x) / 2 < p'(x))
    P = _bound_at(ROW, 2, -NEAR)                  # group 2 (token 2) just dropped
    tgt = np.stack([ROW, ROW]).astype(np.float32)
    x = 2
    p_kept = _masses(ROW)[:3] / _masses(ROW)[:3].sum()
    q = np.full((1, 4), 0.0, np.float32)
    q[0, x] = p_kept[x] / 2
    q[0, 3] = 1 - q[0, x]
    r0 = oracle.verify_request(0, tgt, q, [x], 1.0, 5, top_p=P)
    assert r0.status == 0 and r0.accept[0] == 0 and r0.p_x[0] == 0
    # row 0 is tested and drawn from; the bonus row is never adjusted (n = 0)
    assert list(r0.edge_lo) == [0, 0] and list(r0.edge_hi) == [1, 0]
    r1 = oracle.verify_request(0, tgt, q, [x], 1.0, 5, top_p=P, edge_shift=[1, 0])
    assert r1.status == 0 and r1.accept[0] == 1
    assert r1.p_x[0] == pytest.approx(p_kept[x], rel=1e-12)
    assert r1.beta[0] == pytest.approx(np.minimum(np.r_[p_kept, 0], q[0]).sum(), rel=1e-12)
    bad = oracle.verify_request(0, tgt, q, [x], 1.0, 5, top_p=P, edge_shift=[2, 0])
    assert bad.status == oracle.INVALID_ARG


def test_batch_reports_edge_ranges_per_target_row():
    P = _bound_at(ROW, 2, NEAR)
    tgt = np.stack([ROW] * 5).astype(np.float32)            # two requests: gamma 1 and 2
    q = np.full((3, 4), 0.25, np.float32)
    cu = np.array([0, 1, 3], np.int32)
    r = oracle.rejection_sample(tgt, q, np.zeros(3, np.int32), cu, 1.0, 3, top_p=P)
    assert r.status == 0
    # every row the requests adjusted reports the same band; rows they never
    # adjusted (a bonus row after a rejection) report none
    for b in range(2):
        t0, t1 = cu[b] + b, cu[b + 1] + b
        n = r.num_accepted[b]
        for t in range(t0, t1 + 1):
            used = (t - t0) < (cu[b + 1] - cu[b]) or n == cu[b + 1] - cu[b]
            assert (r.edge_lo[t], r.edge_hi[t]) == ((-1, 0) if used else (0, 0))
