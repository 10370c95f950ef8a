"""Statistical pins (a)-(e) run on the CPU oracle alone: the oracle must
reproduce what the pages prove before it is allowed to judge the CUDA path."""
import numpy as np
import pytest

import oracle
import stat_checks as sc


def run_oracle(tgt, q, ids, cu, T, seed):
    r = oracle.rejection_sample(tgt, q, ids, cu, T, seed)
    assert r.status == 0
    return r.tokens, r.num_accepted, r.accept, r.beta


def test_eq1_against_printed_values():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "leviathan_eq1_values.txt")
    seen = 0
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        a, g, what, val, tol = line.split()
        a, g, val, tol = float(a), int(g), float(val), float(tol)
        e = sc.expected_tokens(a, g)
        got = e if what == "speed" else (g + 1) / e        # ops factor with c_hat = 0
        assert abs(got - val) <= tol, (line, got)
        seen += 1
    assert seen == 3
    assert sc.expected_tokens(1.0, 7) == 8.0


def test_a_output_distribution_matches_p():
    out = sc.check_a_output_distribution(run_oracle)
    assert out["slot0"] > sc.P_MIN
    assert out["residual"] > sc.P_MIN
    assert out["bonus"] > sc.P_MIN
    # (b) acceptance rate vs beta within 3 sigma
    assert out["accept_z"] < 3.0
    assert out["beta_err"] < 1e-12


def test_a_output_distribution_at_temperature():
    out = sc.check_a_output_distribution(run_oracle, n=400_000, seed=7, T=0.6)
    assert out["slot0"] > sc.P_MIN and out["bonus"] > sc.P_MIN and out["accept_z"] < 3.0


def test_a_joint_two_token_string():
    assert sc.check_joint_two_tokens(run_oracle) > sc.P_MIN


def test_c_eq1_iid_positions():
    out = sc.check_c_eq1(run_oracle)
    assert out["pvalue"] > sc.P_MIN
    assert out["z"] < 3.0
    assert 0.3 < out["alpha"] < 0.95


def test_d_special_cases():
    same, disjoint = sc.check_d_special(run_oracle)
    assert same["all_accepted"] and same["beta_min"] > 1 - 1e-7   # float32 ln 2, ln 4
    assert same["bonus_p"] > sc.P_MIN
    assert disjoint["none_accepted"] and disjoint["beta_max"] == 0.0
    assert disjoint["correction_p"] > sc.P_MIN


def test_e_generated_workloads_emit_a_token():
    from speculative_decoding_rejection_decode_gb300.inputs import make_config, to_numpy_logits
    for k, kw in ((0, {}), (1, dict(V=512)), (2, dict(B=16, V=300)), (3, dict(B=24, V=400))):
        w = make_config(k, **kw)
        q = None if w.draft_probs is None else w.draft_probs.numpy()
        r = oracle.rejection_sample(to_numpy_logits(w.target_logits), q, w.draft_ids.numpy(),
                                    w.cu.numpy(), w.T, w.seed)
        assert r.status == 0
        sc.check_e_layout(r.tokens, r.num_accepted, w.draft_ids.numpy(), w.cu.numpy(), w.V)


def _mutant_run(tgt, q, ids, cu, T, seed):
    """The oracle with a planted mistake: the correction distribution uses
    max(0, q - p) instead of max(0, p - q).  Emulated on the oracle's outputs by
    redrawing the token of rejected requests (CPU only)."""
    tokens, nacc, acc, beta = run_oracle(tgt, q, ids, cu, T, seed)
    V = tgt.shape[1]
    B = len(cu) - 1
    rng = np.random.default_rng(seed)
    tokens = tokens.copy()
    for b in range(B):
        n = nacc[b]
        g = cu[b + 1] - cu[b]
        if n < g:
            p = sc.softmax64(tgt[cu[b] + b + n], T)
            w = np.maximum(q[cu[b] + n].astype(np.float64) - p, 0)
            tokens[cu[b] + b + n] = rng.choice(V, p=w / w.sum())
    return tokens, nacc, acc, beta


def test_pins_detect_a_planted_mistake():
    # Check (a) must reject the mutant: either its chi-square collapses or it
    # emits a token outside the residual's support.
    try:
        out = sc.check_a_output_distribution(_mutant_run, n=60_000)
        detected = out["slot0"] < 1e-6 or out["residual"] < 1e-6
    except AssertionError:
        detected = True
    assert detected


def test_a_onehot_drafter_output_distribution():
    # A deterministic (greedy) drafter is q = onehot(x): the emitted token still
    # follows p, and the acceptance rate is p(x).
    from scipy import stats  # noqa: F401
    rng = np.random.default_rng(21)
    n, V = 400_000, 8
    lt = np.array([[0.3, -1.0, 1.2, 0.0, 0.7, -0.4, 0.5, -2.0],
                   [1.0, 0.2, -0.5, 0.9, 0.0, -1.5, 0.4, 0.1]], np.float32)
    x = 2
    tgt = np.tile(lt, (n, 1))
    ids = np.full(n, x, np.int32)
    cu = np.arange(n + 1).astype(np.int32)
    r = oracle.rejection_sample(tgt, None, ids, cu, 1.0, 5)
    assert r.status == 0
    p = sc.softmax64(lt, 1.0)
    tok0 = r.tokens.reshape(n, 2)[:, 0]
    assert sc.chi2_ok(np.bincount(tok0, minlength=V), p[0]) > sc.P_MIN
    acc = r.accept.mean()
    assert abs(acc - p[0, x]) < 3 * np.sqrt(p[0, x] * (1 - p[0, x]) / n)
