"""Pins of the oracle's token-tree verifier (several candidates per position).

The pages give no multi-candidate rule; the oracle applies their
single-candidate step again after each rejection (accept x with probability
min(1, t(x)/q(x)), else continue with t = norm(max(0, t - q))).  What fixes it
without reference to itself:
  - the emitted token at every node follows the target distribution p of that
    node (the theorem of the vllbc page's Appendix A.1 / the bloss0m page's
    Section 2.3, applied at every round), checked by chi-square over many
    independent trees, and likewise the second token given the first;
  - the first candidate is accepted with probability beta = sum min(p, q)
    (Theorem 3.5), the second, after a rejection, with sum min(p1, q) for the
    normalised residual p1;
  - a chain is the chain verifier (which has its own pins), bit for bit;
  - special cases: p = q accepts the first candidate; disjoint supports reject
    every candidate and draw from p; a rejected candidate's duplicate is always
    rejected; the r-th candidate uses the uniform U(seed, b, u, 0, r);
  - greedy trees against brute force; malformed trees are refused.
"""
import numpy as np
import pytest

import oracle
import stat_checks as sc


def _tree_batch(roots, child_tokens, child_rows, q_root, n):
    """n copies of a depth-1 tree: node 0 (target row `roots`, draft row
    q_root), children with the given tokens and target rows."""
    K = len(child_tokens)
    V = roots.shape[0]
    rows = np.concatenate([roots[None], np.asarray(child_rows, np.float32).reshape(K, V)])
    tgt = np.tile(rows, (n, 1)).astype(np.float32)
    q = np.tile(np.concatenate([q_root[None], np.full((K, V), 1.0 / V)]), (n, 1)).astype(np.float32)
    tok = np.tile(np.r_[0, child_tokens], n).astype(np.int32)
    par = np.tile(np.r_[-1, np.zeros(K, int)], n).astype(np.int32)
    cu = (np.arange(n + 1) * (K + 1)).astype(np.int32)
    return tgt, q, tok, par, cu


def test_chain_is_the_chain_verifier():
    rng = np.random.default_rng(3)
    for trial in range(30):
        V = int(rng.integers(2, 40))
        gamma = int(rng.integers(0, 7))
        T = float(rng.choice([0.0, 0.5, 1.0, 2.0]))
        tgt = rng.normal(0, 2, size=(gamma + 1, V)).astype(np.float32)
        q = rng.dirichlet(np.ones(V) * 0.5, size=max(gamma, 1)).astype(np.float32)[:gamma]
        ids = rng.integers(0, V, size=gamma).astype(np.int32)
        seed = int(rng.integers(0, 1 << 30))
        lin = oracle.verify_request(5, tgt, None if T == 0 else q, ids, T, seed)
        # tree: node i + 1 is the only child of node i and carries draft i
        dr = None if T == 0 else np.concatenate([q, np.full((1, V), 1.0 / V, np.float32)])
        tok = np.r_[0, ids].astype(np.int32)
        par = np.arange(-1, gamma).astype(np.int32)
        tr = oracle.tree_verify_request(5, tgt, dr, tok, par, T, seed)
        assert tr.status == 0
        assert tr.num_accepted[0] == lin.num_accepted[0]
        assert np.array_equal(tr.tokens, lin.tokens)
        assert tr.near_tie[0] == lin.near_tie[0]
        n = lin.num_accepted[0]
        assert list(tr.path[:n]) == list(range(1, n + 1))


@pytest.mark.parametrize("K", [2, 3, 5])
def test_first_token_follows_p(K):
    # K candidates drawn independently from q at the root; every child is a
    # leaf.  Whatever happens, the first emitted token must follow p.
    rng = np.random.default_rng(K)
    V, n = 6, 300_000
    lr = np.array([0.4, -1.0, 1.1, 0.0, 0.7, -0.3], np.float32)
    p = sc.softmax64(lr, 1.0)
    q_root = np.array([0.05, 0.3, 0.1, 0.35, 0.15, 0.05], np.float32)
    cand = rng.choice(V, size=(n, K), p=q_root.astype(np.float64) / q_root.astype(np.float64).sum())
    tgt, q, tok, par, cu = _tree_batch(lr, np.zeros(K, int), np.zeros((K, V)), q_root, n)
    tok.reshape(n, K + 1)[:, 1:] = cand
    r = oracle.tree_verify(tgt, q, tok, par, cu, 1.0, 11)
    assert r.status == 0
    first = r.tokens.reshape(n, K + 1)[:, 0]
    assert sc.chi2_ok(np.bincount(first, minlength=V), p) > sc.P_MIN
    # acceptance: the first candidate with probability beta = sum min(p, q),
    # the second (after a rejection) with sum min(p1, q), p1 the residual
    path = r.path.reshape(n, K + 1)
    beta = np.minimum(p, q_root).sum()
    acc0 = (path[:, 0] == 1).mean()
    assert abs(acc0 - beta) < 3 * np.sqrt(beta * (1 - beta) / n)
    p1 = np.maximum(p - q_root, 0)
    p1 /= p1.sum()
    beta1 = np.minimum(p1, q_root).sum()
    rej0 = path[:, 0] != 1
    acc1 = (path[rej0, 0] == 2).mean()
    m = rej0.sum()
    assert abs(acc1 - beta1) < 3 * np.sqrt(beta1 * (1 - beta1) / m)


def test_second_token_follows_its_context():
    # two levels with two candidates each; the target row of a child depends
    # on its token (a context-dependent table); given the first token y1, the
    # second token must follow p(. | y1)
    rng = np.random.default_rng(7)
    V, n = 5, 200_000
    l0 = np.array([0.2, 1.0, -0.5, 0.6, 0.0], np.float32)
    table = rng.normal(0, 1, size=(V, V)).astype(np.float32)      # row y1: logits after y1
    q0 = np.array([0.3, 0.2, 0.1, 0.2, 0.2], np.float32)
    q1 = rng.dirichlet(np.ones(V), size=V).astype(np.float32)     # drafter after y1
    # nodes: 0 root; 1, 2 children of 0; 3, 4 children of 1; 5, 6 children of 2
    c1 = rng.choice(V, size=(n, 2), p=q0.astype(np.float64) / q0.astype(np.float64).sum())
    c2 = np.empty((n, 4), np.int64)
    for k, parent in enumerate((0, 0, 1, 1)):
        y1 = c1[:, parent]
        cum = np.cumsum(q1[y1].astype(np.float64), axis=1)
        c2[:, k] = (rng.random(n)[:, None] * cum[:, -1:] > cum).sum(axis=1)
    tok = np.zeros((n, 7), np.int32)
    tok[:, 1:3] = c1
    tok[:, 3:7] = c2
    par = np.tile(np.array([-1, 0, 0, 1, 1, 2, 2], np.int32), n)
    tgt = np.empty((n, 7, V), np.float32)
    tgt[:, 0] = l0
    tgt[:, 1] = table[c1[:, 0]]
    tgt[:, 2] = table[c1[:, 1]]
    tgt[:, 3:7] = 0.0
    q = np.empty((n, 7, V), np.float32)
    q[:, 0] = q0
    q[:, 1] = q1[c1[:, 0]]
    q[:, 2] = q1[c1[:, 1]]
    q[:, 3:7] = 1.0 / V
    cu = (np.arange(n + 1) * 7).astype(np.int32)
    r = oracle.tree_verify(tgt.reshape(-1, V), q.reshape(-1, V), tok.reshape(-1), par, cu, 1.0, 5)
    assert r.status == 0
    toks = r.tokens.reshape(n, 7)
    nacc = r.num_accepted
    assert sc.chi2_ok(np.bincount(toks[:, 0], minlength=V), sc.softmax64(l0, 1.0)) > sc.P_MIN
    deep = nacc >= 1
    for y1 in range(V):
        sel = deep & (toks[:, 0] == y1)
        if sel.sum() < 2000:
            continue
        want = sc.softmax64(table[y1], 1.0)
        assert sc.chi2_ok(np.bincount(toks[sel, 1], minlength=V), want) > sc.P_MIN, y1


def test_p_equals_q_accepts_the_first_candidate_and_disjoint_rejects_all():
    V, n = 6, 20_000
    rng = np.random.default_rng(2)
    l = rng.normal(0, 1, size=V).astype(np.float32)
    p = sc.softmax64(l, 1.0).astype(np.float32)
    cand = rng.choice(V, size=(n, 3), p=p.astype(np.float64) / p.astype(np.float64).sum())
    tgt, q, tok, par, cu = _tree_batch(l, np.zeros(3, int), np.zeros((3, V)), p, n)
    tok.reshape(n, 4)[:, 1:] = cand
    r = oracle.tree_verify(tgt, q, tok, par, cu, 1.0, 3)
    assert np.all(r.path.reshape(n, 4)[:, 0] == 1)
    # disjoint: p lives on {0, 1, 2}, q on {3, 4, 5}
    l2 = np.array([0.5, 0.0, -0.5, -np.inf, -np.inf, -np.inf], np.float32)
    q2 = np.array([0, 0, 0, 0.2, 0.3, 0.5], np.float32)
    cand = rng.choice([3, 4, 5], size=(n, 3), p=[0.2, 0.3, 0.5])
    tgt, q, tok, par, cu = _tree_batch(l2, np.zeros(3, int), np.zeros((3, V)), q2, n)
    tok.reshape(n, 4)[:, 1:] = cand
    r = oracle.tree_verify(tgt, q, tok, par, cu, 1.0, 3)
    assert np.all(r.num_accepted == 0)
    first = r.tokens.reshape(n, 4)[:, 0]
    assert sc.chi2_ok(np.bincount(first, minlength=V)[:3], sc.softmax64(l2[:3], 1.0)) > sc.P_MIN


def test_duplicate_of_a_rejected_candidate_is_rejected():
    # once x is rejected (t(x) < q(x)), the residual has t1(x) = 0
    V, n = 4, 5000
    l = np.log(np.array([0.1, 0.4, 0.3, 0.2])).astype(np.float32)
    q_root = np.array([0.7, 0.1, 0.1, 0.1], np.float32)      # p(0) < q(0)
    tgt, q, tok, par, cu = _tree_batch(l, [0, 0, 2], np.zeros((3, V)), q_root, n)
    r = oracle.tree_verify(tgt, q, tok, par, cu, 1.0, 9)
    path = r.path.reshape(n, 4)[:, 0]
    assert np.all(path != 2)                 # the duplicate (node 2) is never accepted
    assert (path == 1).any() and (path == 3).any()


def test_candidate_r_uses_uniform_r():
    # candidate 0 surely rejected (t(x) = 0); candidate 1 has ratio a in the
    # residual, which here equals p: accepted iff U(seed, b, 0, 0, 1) < a
    V = 3
    l = np.array([0.0, np.log(3.0), -np.inf], np.float32)      # p = (1/4, 3/4, 0)
    q_root = np.array([0.5, 0.0, 0.5], np.float32)
    # residual after rejecting token 2: max(0, p - q) = (0, 3/4, 0) -> (0, 1, 0)
    tgt, q, tok, par, cu = _tree_batch(l, [2, 0], np.zeros((2, V)), q_root, 1)
    for seed in range(40):
        r = oracle.tree_verify(tgt, q, tok, par, cu, 1.0, seed)
        # t1(0) = 0 so candidate 1 (token 0) is rejected too; the extra token is 1
        assert r.num_accepted[0] == 0 and r.tokens[0] == 1
    q_root = np.array([0.0, 0.4, 0.6], np.float32)
    # p(2) = 0: candidate 0 (token 2) rejected; residual (1/4, 3/4 - 0.4, 0) / 0.6
    tgt, q, tok, par, cu = _tree_batch(l, [2, 1], np.zeros((2, V)), q_root, 1)
    p1_1 = (0.75 - 0.4) / 0.6
    a = min(1.0, p1_1 / 0.4)
    for seed in range(60):
        r = oracle.tree_verify(tgt, q, tok, par, cu, 1.0, seed)
        u1 = oracle.uniform(seed, 0, 0, 0, 1, 1)[0]
        if abs(u1 - a) > 1e-6:
            assert (r.path[0] == 2) == (u1 < a), seed


def test_greedy_tree_brute_force():
    rng = np.random.default_rng(4)
    for trial in range(40):
        V = int(rng.integers(2, 9))
        nn = int(rng.integers(1, 12))
        par = np.r_[-1, [rng.integers(0, j) for j in range(1, nn)]].astype(np.int32)
        tgt = rng.integers(-2, 3, size=(nn, V)).astype(np.float32)    # ties
        am = tgt.argmax(1)
        tok = np.r_[0, [am[par[j]] if rng.random() < 0.6 else rng.integers(0, V)
                        for j in range(1, nn)]].astype(np.int32)
        r = oracle.tree_verify_request(0, tgt, None, tok, par, 0.0, 0)
        u, path = 0, []
        while True:
            nxt = [c for c in range(u + 1, nn) if par[c] == u and tok[c] == am[u]]
            if not nxt:
                break
            path.append(nxt[0])
            u = nxt[0]
        assert r.num_accepted[0] == len(path)
        assert list(r.tokens[:len(path)]) == [tok[c] for c in path]
        assert r.tokens[len(path)] == am[u]
        assert list(r.path[:len(path)]) == path


def test_malformed_trees_are_refused():
    tgt = np.zeros((3, 4), np.float32)
    q = np.full((3, 4), 0.25, np.float32)
    for par in ([0, 0, 1], [-1, 1, 0], [-1, 0, 3], [-1, -1, 0]):
        r = oracle.tree_verify_request(0, tgt, q, [0, 1, 2], par, 1.0, 0)
        assert r.status == oracle.INVALID_ARG, par
    r = oracle.tree_verify_request(0, tgt, q, [0, 9, 2], [-1, 0, 0], 1.0, 0)
    assert r.status == oracle.BAD_DRAFT_ID
