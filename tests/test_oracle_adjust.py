"""Pins of the oracle's top-k / top-p adjusted target distribution (the vllbc
page's Section 2.2 note folds top-k and top-p into the adjusted p before the
same rejection test).  The kept set and its renormalisation are checked against
hand values, against a token-by-token evaluation of the definition on tiny rows
with planted ties, against the properties that make it the nucleus, and through
the output distribution of the whole verify step."""
import numpy as np
import pytest

import oracle
import stat_checks as sc


def _f32(x):
    return np.asarray(x, np.float32)


def _near_edge(l, T, k, P, rel=1e-5):
    """True when some group's larger-logit mass lies within `rel` of the top-p
    bound in exact arithmetic: there the float32 decision of the edge may go
    either way, so the exact definition is not a pin."""
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


def test_pow2_neg_definition():
    # 2^-z on the float32 definition: 0 from z = 64 on, exact powers of two at
    # integer z, within 4e-7 of 2^-z elsewhere
    assert oracle.pow2_neg(0.0) == 1.0
    for k in range(64):
        assert oracle.pow2_neg(float(k)) == 2.0 ** -k
    assert oracle.pow2_neg(64.0) == 0.0 and oracle.pow2_neg(1e30) == 0.0
    assert oracle.pow2_neg(float("nan")) == 0.0
    rng = np.random.default_rng(0)
    z = np.concatenate([rng.uniform(0, 64, 20000), rng.uniform(0, 1, 20000)]).astype(np.float32)
    got = np.array([oracle.pow2_neg(float(x)) for x in z])
    rel = np.abs(got - np.exp2(-z.astype(np.float64))) / np.exp2(-z.astype(np.float64))
    assert rel.max() < 4e-7, rel.max()
    # monotone non-increasing in z on a fine grid of one unit
    g = np.array([oracle.pow2_neg(float(x)) for x in np.linspace(3, 4, 5001, dtype=np.float32)])
    assert np.all(np.diff(g) <= 0)


def test_selection_mass_definition():
    # the integer mass 2^-z * 2^F rounded to the nearest integer, ties to even,
    # with F = 62 - ceil(log2 V): F from V's powers of two, exact powers of two
    # at integer z, 1/2 rounds to 0 and 2^-1/2 to 1, nothing past z = 64, a row
    # of V entries at the maximum sums to at most 2^62, and 2^-z as above
    for V, F in [(1, 62), (2, 61), (3, 60), (4, 60), (5, 59), (32000, 47), (151936, 44),
                 (256000, 44), (262144, 44), (262145, 43), (1 << 30, 32)]:
        z = np.array([0.0, 1.0, 5.0, F - 1.0, float(F), F + 0.5, F + 1.0, F + 2.0, 64.0],
                     np.float32)
        mass, p2 = oracle.selection_mass(z, V)
        assert mass.dtype == np.uint64
        assert [int(m) for m in mass] == [2 ** F, 2 ** (F - 1), 2 ** (F - 5), 2, 1, 1, 0, 0, 0], V
        assert V * int(mass[0]) <= 2 ** 62
        assert np.array_equal(p2, np.array([oracle.pow2_neg(float(x)) for x in z], np.float32))
    mass, _ = oracle.selection_mass(np.array([np.nan, np.inf, 1e30], np.float32), 1000)
    assert mass.tolist() == [0, 0, 0]
    # non-increasing in z
    m, _ = oracle.selection_mass(np.linspace(0, 50, 20001, dtype=np.float32), 256000)
    assert np.all(np.diff(m.astype(np.float64)) <= 0)


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
