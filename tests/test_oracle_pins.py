"""Deterministic pins of the CPU oracle: closed forms, hand-computed values,
identities, special cases and brute force on tiny inputs.  Each would catch a
plausible slip in the oracle (a transposed operand, a wrong sign or index, a
missing temperature, a <= for a <)."""
import math

import numpy as np
import pytest

import oracle


def _run(tgt, q, ids, T=1.0, seed=0, gammas=None):
    tgt = np.asarray(tgt, np.float32)
    q = None if q is None else np.asarray(q, np.float32)
    ids = np.asarray(ids, np.int32)
    if gammas is None:
        gammas = [len(ids)]
    cu = np.concatenate([[0], np.cumsum(gammas)]).astype(np.int32)
    return oracle.rejection_sample(tgt, q, ids, cu, T, seed)


def test_softmax_closed_form_and_temperature():
    # logits (0, ln 3) at T=1 give p = (1/4, 3/4); (0, 2 ln 3) at T=2 as well.
    for logits, T in (([0.0, math.log(3.0)], 1.0), ([0.0, 2 * math.log(3.0)], 2.0),
                      ([5.0, 5.0 + math.log(3.0)], 1.0)):
        tgt = np.array([logits, [0.0, 0.0]], np.float32)
        r = _run(tgt, [[0.5, 0.5]], [1], T=T)
        assert r.p_x[0] == pytest.approx(0.75, abs=2e-7)     # float32 storage of ln 3
        assert r.q_x[0] == 0.5
        r0 = _run(tgt, [[0.5, 0.5]], [0], T=T)
        assert r0.p_x[0] == pytest.approx(0.25, abs=2e-7)


def test_beta_by_hand():
    # p = (1/4, 3/4), q = (1/2, 1/2): beta = 1/4 + 1/2 = 3/4 (Theorem 3.5).
    tgt = np.array([[0.0, math.log(3.0)], [0.0, 0.0]], np.float32)
    r = _run(tgt, [[0.5, 0.5]], [0])
    assert r.beta[0] == pytest.approx(0.75, abs=2e-7)
    # p = softmax(0, ln 2, ln 5) = (1/8, 2/8, 5/8); q = (1/2, 1/4, 1/4): beta = 1/8+1/4+1/4.
    tgt = np.array([[0.0, math.log(2.0), math.log(5.0)], [0, 0, 0]], np.float32)
    r = _run(tgt, [[0.5, 0.25, 0.25]], [2])
    assert r.beta[0] == pytest.approx(0.625, abs=2e-7)
    assert r.p_x[0] == pytest.approx(0.625, abs=2e-7)


def test_beta_brute_force_random_rows():
    rng = np.random.default_rng(5)
    for V in (3, 5, 8):
        logits = rng.normal(0, 2, size=(4, V)).astype(np.float32)
        qraw = rng.random((3, V))
        q = (qraw / qraw.sum(1, keepdims=True)).astype(np.float32)
        ids = rng.integers(0, V, size=3)
        T = 0.8
        r = _run(logits, q, ids, T=T)
        for i in range(3):
            l = logits[i].astype(np.float64) / T
            p = np.exp(l - l.max())
            p /= p.sum()
            assert r.beta[i] == pytest.approx(np.minimum(p, q[i].astype(np.float64)).sum(), abs=1e-12)
            assert r.p_x[i] == pytest.approx(p[ids[i]], abs=1e-12)
            # identity used in the correctness argument (App. A.1 on the vllbc page)
            assert np.maximum(p - q[i], 0).sum() == pytest.approx(1 - r.beta[i], abs=1e-7)


def test_ratio_conventions():
    # q(x) <= p(x) always accepts; p(x) = 0 always rejects; q(x) = 0 < p(x) accepts.
    tgt = np.array([[0.0, 0.0], [0.0, 0.0]], np.float32)     # p = (1/2, 1/2)
    for seed in range(50):
        assert _run(tgt, [[0.6, 0.4]], [1], seed=seed).accept[0] == 1
        assert _run(tgt, [[1.0, 0.0]], [1], seed=seed).accept[0] == 1
    tgt = np.array([[0.0, -np.inf], [0.0, 0.0]], np.float32)  # p = (1, 0)
    for seed in range(50):
        r = _run(tgt, [[0.5, 0.5]], [1], seed=seed)
        assert r.accept[0] == 0 and r.num_accepted[0] == 0
        assert r.tokens[0] == 0                       # residual max(0, p - q) = (1/2, 0)


def test_accept_threshold_uses_generator_stream_zero():
    # With p(x)/q(x) = a, position i is accepted iff U(seed, b, i, 0, 0) < a.
    tgt = np.array([[0.0, math.log(3.0)]] * 4, np.float32)      # p = (1/4, 3/4)
    q = np.array([[0.5, 0.5]] * 3, np.float32)
    for seed in range(40):
        r = _run(tgt, q, [0, 0, 0], seed=seed)
        for i in range(3):
            u = oracle.uniform(seed, 0, i, 0, 0, 1)[0]
            if abs(u - 0.5) > 1e-6:
                assert r.accept[i] == int(u < 0.5)


def test_worked_example_layout():
    # The reading-notes example (bloss0m, "Walk one example through the method"):
    # gamma = 3, the first two drafts pass, the third is rejected, and the step
    # emits 2 drafts + 1 correction.  Rows built so that the outcome is forced.
    V = 4
    tgt = np.array([[0.0, 3.0, 0.0, 0.0],          # p0(1) large
                    [0.0, 0.0, 3.0, 0.0],          # p1(2) large
                    [0.0, 0.0, 0.0, -np.inf],      # p2(3) = 0 -> reject draft 3
                    [0.0, 0.0, 0.0, 0.0]], np.float32)
    q = np.array([[0.1, 0.1, 0.1, 0.7], [0.7, 0.1, 0.1, 0.1], [0.0, 0.0, 0.0, 1.0]], np.float32)
    ids = [1, 2, 3]
    r = _run(tgt, q, ids, seed=3)
    assert r.num_accepted[0] == 2
    assert list(r.tokens[:2]) == [1, 2]
    assert 0 <= r.tokens[2] < 3                    # correction comes from the residual support
    assert r.tokens[3] == -1


def test_gamma_zero_request_only_bonus():
    tgt = np.array([[0.0, 1.0, 2.0]], np.float32)
    r = _run(tgt, np.zeros((0, 3), np.float32), [], gammas=[0])
    assert r.num_accepted[0] == 0 and 0 <= r.tokens[0] < 3


def test_bad_draft_id_is_rejected_and_reported():
    tgt = np.zeros((3, 4), np.float32)
    q = np.full((2, 4), 0.25, np.float32)
    r = _run(tgt, q, [7, 1])
    assert r.status == oracle.BAD_DRAFT_ID
    assert r.num_accepted[0] == 0 and r.accept[0] == 0
    assert r.p_x[0] == 0 and r.q_x[0] == 0


def test_invalid_arguments():
    tgt = np.zeros((2, 4), np.float32)
    q = np.full((1, 4), 0.25, np.float32)
    assert _run(tgt, q, [0], T=-1.0).status == oracle.INVALID_ARG
    assert _run(tgt, q, [0], T=float("nan")).status == oracle.INVALID_ARG
    r = oracle.rejection_sample(np.zeros((4, 4), np.float32), np.full((2, 4), .25, np.float32),
                                np.zeros(2, np.int32), np.array([0, 1, 2], np.int32), 1.0, 0)
    assert r.status == oracle.OK
    # cu must start at 0 and never decrease
    r = oracle.rejection_sample(np.zeros((3, 4), np.float32), np.full((1, 4), .25, np.float32),
                                np.zeros(1, np.int32), np.array([0, 2, 1], np.int32), 1.0, 0)
    assert r.status == oracle.INVALID_ARG
    r = oracle.rejection_sample(np.zeros((4, 4), np.float32), np.full((2, 4), .25, np.float32),
                                np.zeros(2, np.int32), np.array([1, 1, 2], np.int32), 1.0, 0)
    assert r.status == oracle.INVALID_ARG


# ----------------------------------------------------------------------------
# Greedy (T = 0): argmax with the lowest index on ties, against brute force.
# ----------------------------------------------------------------------------

def _bf16_bits(x):
    """Round-to-nearest-even float32 -> bf16 bit patterns (numpy, test-side)."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def _bf16_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_greedy_brute_force_with_ties(dtype):
    rng = np.random.default_rng(11)
    B, gamma, V = 40, 5, 37
    x = rng.normal(0, 3, size=(B * (gamma + 1), V)).astype(np.float32)
    # plant exact ties of the row maximum, including -0.0 vs +0.0 rows
    for r in range(0, x.shape[0], 3):
        j, k = sorted(rng.choice(V, 2, replace=False))
        x[r, k] = x[r, j] = np.abs(x[r]).max() + 1.0
    x[1] = -1.0
    x[1, 2] = -0.0          # -0.0 == +0.0: the lower index (2) must win
    x[1, 5] = 0.0
    stored = _bf16_bits(x) if dtype == "bf16" else x
    vals = _bf16_to_f64(stored) if dtype == "bf16" else x.astype(np.float64)
    g = vals.argmax(1)                    # numpy returns the first maximal index
    cu = (np.arange(B + 1) * gamma).astype(np.int32)
    ids = np.empty(B * gamma, np.int32)
    for b in range(B):
        for i in range(gamma):
            row = b * (gamma + 1) + i
            ids[b * gamma + i] = g[row] if rng.random() < 0.7 else rng.integers(0, V)
    r = oracle.rejection_sample(stored, None, ids, cu, 0.0, 0)
    assert r.status == 0
    for b in range(B):
        acc = [ids[b * gamma + i] == g[b * (gamma + 1) + i] for i in range(gamma)]
        n = acc.index(False) if False in acc else gamma
        assert r.num_accepted[b] == n
        toks = r.tokens[b * (gamma + 1):(b + 1) * (gamma + 1)]
        assert list(toks[:n]) == list(ids[b * gamma:b * gamma + n])
        assert toks[n] == g[b * (gamma + 1) + n]
        assert all(t == -1 for t in toks[n + 1:])
        assert list(r.beta[b * gamma:(b + 1) * gamma]) == [float(a) for a in acc]
    assert r.near_tie.sum() == 0


# ----------------------------------------------------------------------------
# One-hot drafter (no draft probabilities at T > 0): q_i = [v == x_i].
# ----------------------------------------------------------------------------

def test_onehot_draft_closed_forms():
    # beta = sum min(p, onehot(x)) = p(x); q(x) = 1; the accept test is r < p(x).
    rng = np.random.default_rng(8)
    V, gamma, T = 9, 4, 0.7
    logits = rng.normal(0, 2, size=(gamma + 1, V)).astype(np.float32)
    ids = rng.integers(0, V, size=gamma)
    for seed in range(20):
        r = _run(logits, None, ids, T=T, seed=seed)
        assert r.status == 0
        for i in range(gamma):
            l = logits[i].astype(np.float64) / T
            p = np.exp(l - l.max())
            p /= p.sum()
            assert r.beta[i] == pytest.approx(p[ids[i]], abs=1e-12)
            assert r.q_x[i] == 1.0 and r.p_x[i] == pytest.approx(p[ids[i]], abs=1e-12)
            u = oracle.uniform(seed, 0, i, 0, 0, 1)[0]
            if abs(u - p[ids[i]]) > 1e-9:
                assert r.accept[i] == int(u < p[ids[i]])
        n = r.num_accepted[0]
        if n < gamma:
            assert r.tokens[n] != ids[n]          # the residual excludes the draft token
