"""Statistical checks (a)-(e) of the verifier's guarantees, shared by the
oracle tests (CPU) and the CUDA tests (GPU).  Each check takes a callable
``run(target, draft, ids, cu, T, seed) -> (tokens, num_accepted, accept, beta)``
with numpy inputs and outputs, so that the same statistics judge both sides.

What the pages fix:
  (a) the emitted token is distributed as p (Section 2.3 and Appendix A.1 on the
      bloss0m and vllbc pages: "output distribution identical to M_p");
  (b) a draft is accepted with probability beta = sum min(p, q) (Theorem 3.5,
      Corollary 3.6);
  (c) with i.i.d. positions, E[#tokens per step] = sum_{k=0}^{gamma} alpha^k and
      P(n >= k) = alpha^k (Eq. (1));
  (d) p = q accepts everything, disjoint supports accept nothing (vllbc page,
      after Theorem 3.5);
  (e) every step emits at least one token (tarrragon page, key property 3;
      Algorithm 1 output line on the bloss0m page).
"""
from __future__ import annotations

import numpy as np
from scipy import stats

P_MIN = 0.01          # chi-square p-value floor


def softmax64(logits, T):
    l = np.asarray(logits, np.float64) / T
    l = l - l.max(axis=-1, keepdims=True)
    e = np.exp(l)
    return e / e.sum(axis=-1, keepdims=True)


def adjusted64(logits, T, top_k=0, top_p=1.0):
    """Top-k / top-p restricted softmax of one row, token by token from the
    definition (O(V^2), tiny rows only): v is kept when fewer than k tokens
    have a larger logit and the mass of the larger-logit tokens is 0 or below
    top_p times the top-k mass."""
    l = np.asarray(logits, np.float64)
    V = l.shape[0]
    e = np.exp((l - l.max()) / T)
    use_k = 1 <= top_k < V
    use_p = not (top_p >= 1.0)
    in_k = np.array([(not use_k) or int((l > l[v]).sum()) < top_k for v in range(V)])
    s_k = e[in_k].sum()
    keep = in_k.copy()
    if use_p:
        for v in range(V):
            a = e[l > l[v]].sum()
            keep[v] = in_k[v] and (a == 0.0 or a < top_p * s_k)
    w = np.where(keep, e, 0.0)
    return w / w.sum()


def expected_tokens(alpha: float, gamma: int) -> float:
    """Eq. (1): (1 - alpha^(gamma+1)) / (1 - alpha), limit gamma+1 at alpha = 1."""
    if alpha == 1.0:
        return gamma + 1.0
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def tile_batch(tgt_rows, draft_rows, n, rng):
    """n identical requests (same target / draft rows), drafts x_i ~ q_i drawn
    independently per request."""
    tgt_rows = np.asarray(tgt_rows, np.float32)
    draft_rows = np.asarray(draft_rows, np.float32)
    gamma, V = draft_rows.shape
    tgt = np.tile(tgt_rows, (n, 1))
    q = np.tile(draft_rows, (n, 1))
    ids = np.empty((n, gamma), np.int32)
    for i in range(gamma):
        w = draft_rows[i].astype(np.float64)
        ids[:, i] = rng.choice(V, size=n, p=w / w.sum())
    cu = (np.arange(n + 1) * gamma).astype(np.int32)
    return tgt, q, ids.reshape(-1), cu


def chi2_ok(counts, probs, min_expected=5.0):
    counts = np.asarray(counts, np.float64)
    probs = np.asarray(probs, np.float64)
    n = counts.sum()
    keep = probs * n >= min_expected
    if (~keep).any():       # pool thin cells
        c = np.append(counts[keep], counts[~keep].sum())
        p = np.append(probs[keep], probs[~keep].sum())
    else:
        c, p = counts, probs
    nz = p > 0
    assert np.all(c[~nz] == 0), "token emitted outside the support"
    res = stats.chisquare(c[nz], p[nz] / p[nz].sum() * c[nz].sum())
    return res.pvalue


def check_a_output_distribution(run, n=1_000_000, seed=12, T=1.0):
    """(a) slot-0 token ~ p_0; within n = 0, token ~ norm(max(0, p_0 - q_0));
    within n = gamma, bonus ~ p_gamma."""
    rng = np.random.default_rng(seed)
    V, gamma = 8, 2
    tgt_rows = np.array([[0.3, -1.0, 1.2, 0.0, 0.7, -0.4, 0.5, -2.0],
                         [1.0, 0.2, -0.5, 0.9, 0.0, -1.5, 0.4, 0.1],
                         [-0.2, 0.8, 0.1, -1.0, 1.4, 0.3, -0.6, 0.9]], np.float32)
    draft_rows = np.array([[0.05, 0.25, 0.10, 0.20, 0.10, 0.15, 0.05, 0.10],
                           [0.20, 0.15, 0.15, 0.05, 0.20, 0.10, 0.10, 0.05]], np.float32)
    tgt, q, ids, cu = tile_batch(tgt_rows, draft_rows, n, rng)
    tokens, nacc, accept, beta = run(tgt, q, ids, cu, T, seed)
    tok = tokens.reshape(n, gamma + 1)
    p = softmax64(tgt_rows, T)
    out = {}
    out["slot0"] = chi2_ok(np.bincount(tok[:, 0], minlength=V), p[0])
    rej0 = nacc == 0
    resid = np.maximum(p[0] - draft_rows[0].astype(np.float64), 0.0)
    out["residual"] = chi2_ok(np.bincount(tok[rej0, 0], minlength=V), resid / resid.sum())
    full = nacc == gamma
    out["bonus"] = chi2_ok(np.bincount(tok[full, gamma], minlength=V), p[gamma])
    # (b) on the same run: accept rate at position 0 vs beta_0.
    beta0 = np.minimum(p[0], draft_rows[0].astype(np.float64)).sum()
    acc0 = accept.reshape(n, gamma)[:, 0].mean()
    sigma = np.sqrt(beta0 * (1 - beta0) / n)
    out["accept_z"] = abs(acc0 - beta0) / sigma
    out["beta_err"] = float(np.abs(beta.reshape(n, gamma)[:, 0] - beta0).max())
    # (e) at least one token; accepted prefix equals the drafts; tail is -1.
    check_e_layout(tokens, nacc, ids, cu, V)
    return out


def check_joint_two_tokens(run, n=400_000, seed=1):
    """(a), joint form: with a context-dependent target P(.|prefix) and drafter
    Q(.|prefix) on V=4, the first two emitted tokens (a second step when the
    first emitted only one) are distributed as P(y1) P(y2|y1)."""
    rng = np.random.default_rng(seed)
    V = 4
    P0 = np.array([0.1, 0.4, 0.3, 0.2])
    P1 = np.array([[0.7, 0.1, 0.1, 0.1], [0.1, 0.2, 0.3, 0.4], [0.25, 0.25, 0.25, 0.25],
                   [0.05, 0.05, 0.6, 0.3]])
    Q0 = np.array([0.25, 0.25, 0.25, 0.25])
    Q1 = np.array([[0.4, 0.2, 0.2, 0.2], [0.1, 0.6, 0.2, 0.1], [0.1, 0.1, 0.1, 0.7],
                   [0.3, 0.3, 0.2, 0.2]])
    # P(.|y1, y2) for the bonus row: any fixed table works; use P1[y2].
    L0, L1 = np.log(P0), np.log(P1)
    # step 1: gamma = 2; drafts x1 ~ Q0, x2 ~ Q1[x1]
    x1 = rng.choice(V, size=n, p=Q0)
    u = rng.random(n)
    x2 = (u[:, None] > np.cumsum(Q1[x1], axis=1)).sum(1).clip(0, V - 1)
    tgt = np.empty((n, 3, V), np.float32)
    tgt[:, 0] = L0
    tgt[:, 1] = L1[x1]
    tgt[:, 2] = L1[x2]
    q = np.empty((n, 2, V), np.float32)
    q[:, 0] = Q0
    q[:, 1] = Q1[x1]
    ids = np.stack([x1, x2], 1).astype(np.int32).reshape(-1)
    cu = (np.arange(n + 1) * 2).astype(np.int32)
    tokens, nacc, _, _ = run(tgt.reshape(-1, V), q.reshape(-1, V), ids, cu, 1.0, seed)
    tok = tokens.reshape(n, 3)
    y1 = tok[:, 0].copy()
    y2 = np.where(nacc >= 1, tok[:, 1], -1)
    # step 2 for requests that emitted a single token: gamma = 1 from prefix y1.
    need = np.nonzero(y2 < 0)[0]
    m = len(need)
    if m:
        z1 = np.array([rng.choice(V, p=Q1[a]) for a in y1[need]])
        tgt2 = np.empty((m, 2, V), np.float32)
        tgt2[:, 0] = L1[y1[need]]
        tgt2[:, 1] = L1[z1]
        q2 = Q1[y1[need]][:, None, :].astype(np.float32)
        cu2 = np.arange(m + 1).astype(np.int32)
        tok2, _, _, _ = run(tgt2.reshape(-1, V), q2.reshape(-1, V), z1.astype(np.int32), cu2,
                            1.0, seed + 1)
        y2[need] = tok2.reshape(m, 2)[:, 0]
    joint = np.bincount(y1 * V + y2, minlength=V * V)
    expected = (P0[:, None] * P1).reshape(-1)
    return chi2_ok(joint, expected)


def check_c_eq1(run, n=400_000, gamma=5, seed=303):
    """(c) i.i.d. positions (the same p and q at every position): the number of
    accepted drafts n satisfies P(n = k) = alpha^k (1 - alpha) for k < gamma,
    P(n = gamma) = alpha^gamma, and E[n + 1] = Eq. (1)."""
    rng = np.random.default_rng(seed)
    V = 8
    lt = np.array([0.5, -0.3, 1.1, 0.0, -1.2, 0.8, 0.2, -0.6], np.float32)
    qd = np.array([0.20, 0.05, 0.10, 0.15, 0.20, 0.10, 0.10, 0.10], np.float32)
    p = softmax64(lt, 1.0)
    alpha = float(np.minimum(p, qd.astype(np.float64)).sum())
    tgt, q, ids, cu = tile_batch(np.tile(lt, (gamma + 1, 1)), np.tile(qd, (gamma, 1)), n, rng)
    tokens, nacc, _, _ = run(tgt, q, ids, cu, 1.0, seed)
    check_e_layout(tokens, nacc, ids, cu, V)
    hist = np.bincount(nacc, minlength=gamma + 1)
    probs = np.array([alpha ** k * (1 - alpha) for k in range(gamma)] + [alpha ** gamma])
    pval = chi2_ok(hist, probs)
    N = nacc + 1.0
    mean_exp = expected_tokens(alpha, gamma)
    var = (probs * (np.arange(gamma + 1) + 1.0) ** 2).sum() - mean_exp ** 2
    z = abs(N.mean() - mean_exp) / np.sqrt(var / n)
    return dict(alpha=alpha, pvalue=pval, mean=N.mean(), expected=mean_exp, z=z)


def check_d_special(run, n=100_000, seed=404):
    """(d) p = q: every draft accepted (alpha = 1) and the bonus ~ p_gamma;
    disjoint supports: nothing accepted (alpha = 0) and the correction ~ p_0."""
    rng = np.random.default_rng(seed)
    gamma, V = 3, 8
    # p exactly dyadic: exp of logits (0, 0, ln2, ln4, -inf ...) / 8
    lt = np.array([0.0, 0.0, np.log(2.0), np.log(4.0), -np.inf, -np.inf, -np.inf, -np.inf],
                  np.float32)
    pd = np.array([1, 1, 2, 4, 0, 0, 0, 0], np.float32) / 8
    tgt, q, ids, cu = tile_batch(np.tile(lt, (gamma + 1, 1)), np.tile(pd, (gamma, 1)), n, rng)
    tokens, nacc, accept, beta = run(tgt, q, ids, cu, 1.0, seed)
    same = dict(all_accepted=bool((nacc == gamma).all()),
                beta_min=float(beta.min()),
                bonus_p=chi2_ok(np.bincount(tokens.reshape(n, gamma + 1)[:, gamma], minlength=V),
                                pd.astype(np.float64)))
    # disjoint: q lives on {4..7} where p = 0
    qd = np.array([0, 0, 0, 0, 0.25, 0.25, 0.25, 0.25], np.float32)
    tgt, q, ids, cu = tile_batch(np.tile(lt, (gamma + 1, 1)), np.tile(qd, (gamma, 1)), n, rng)
    tokens, nacc, accept, beta = run(tgt, q, ids, cu, 1.0, seed + 1)
    disjoint = dict(none_accepted=bool((nacc == 0).all()), beta_max=float(beta.max()),
                    correction_p=chi2_ok(np.bincount(tokens.reshape(n, gamma + 1)[:, 0],
                                                     minlength=V), pd.astype(np.float64)))
    return same, disjoint


def check_e_layout(tokens, nacc, ids, cu, V):
    """(e) n_b <= gamma_b; slots 0..n-1 hold the drafts, slot n a token in
    [0, V), the rest -1."""
    B = len(cu) - 1
    gam = np.diff(cu)
    assert np.all((nacc >= 0) & (nacc <= gam))
    start = cu[:-1] + np.arange(B)
    emitted = tokens[start + nacc]
    assert np.all((emitted >= 0) & (emitted < V))
    # vectorised prefix / tail checks
    slot = np.arange(len(tokens))
    req = np.repeat(np.arange(B), gam + 1)
    off = slot - start[req]
    draft_index = cu[:-1][req] + off
    pre = off < nacc[req]
    assert np.array_equal(tokens[pre], ids[draft_index[pre]])
    tail = off > nacc[req]
    assert np.all(tokens[tail] == -1)


def check_adjusted_distribution(run_adj, top_k, top_p, n=400_000, seed=31, T=1.0):
    """(a) with the adjusted target of the vllbc page's Section 2.2 note: the
    emitted slot-0 token follows the top-k / top-p restricted p_0, a correction
    at position 0 follows norm(max(0, p'_0 - q_0)), and a bonus p'_gamma.
    ``run_adj(tgt, q, ids, cu, T, seed, top_k, top_p)`` returns
    (tokens, num_accepted, accept, beta)."""
    rng = np.random.default_rng(seed)
    V, gamma = 8, 2
    tgt_rows = np.array([[0.3, -1.0, 1.2, 0.0, 0.7, -0.4, 0.5, -2.0],
                         [1.0, 0.2, -0.5, 0.9, 0.0, -1.5, 0.4, 0.1],
                         [-0.2, 0.8, 0.1, -1.0, 1.4, 0.3, -0.6, 0.9]], np.float32)
    draft_rows = np.array([[0.05, 0.25, 0.10, 0.20, 0.10, 0.15, 0.05, 0.10],
                           [0.20, 0.15, 0.15, 0.05, 0.20, 0.10, 0.10, 0.05]], np.float32)
    tgt, q, ids, cu = tile_batch(tgt_rows, draft_rows, n, rng)
    tokens, nacc, accept, beta = run_adj(tgt, q, ids, cu, T, seed, top_k, top_p)
    check_e_layout(tokens, nacc, ids, cu, V)
    tok = tokens.reshape(n, gamma + 1)
    pa = np.stack([adjusted64(r, T, top_k, top_p) for r in tgt_rows])
    out = {}
    out["slot0"] = chi2_ok(np.bincount(tok[:, 0], minlength=V), pa[0])
    rej0 = nacc == 0
    resid = np.maximum(pa[0] - draft_rows[0].astype(np.float64), 0.0)
    out["residual"] = chi2_ok(np.bincount(tok[rej0, 0], minlength=V), resid / resid.sum())
    full = nacc == gamma
    out["bonus"] = chi2_ok(np.bincount(tok[full, gamma], minlength=V), pa[gamma])
    beta0 = np.minimum(pa[0], draft_rows[0].astype(np.float64)).sum()
    out["beta_err"] = float(np.abs(beta.reshape(n, gamma)[:, 0] - beta0).max())
    acc0 = accept.reshape(n, gamma)[:, 0].mean()
    out["accept_z"] = abs(acc0 - beta0) / np.sqrt(beta0 * (1 - beta0) / n)
    return out
