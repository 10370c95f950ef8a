"""Host logic of the parity comparison (CPU): results decided on a reachable
top-p cut other than the exact one are accepted, results no reachable cut
explains are not, and the near-tie budget counts rows.  The "library results"
here are oracle results under a chosen cut, with mistakes planted in them."""

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import compare, flag_budget_ok, run_oracle
from speculative_decoding_rejection_decode_gb300.inputs import from_rows

ROW = np.log(np.array([0.4, 0.3, 0.2, 0.1])).astype(np.float32)


def _workload(rel, x=2, gamma=1):
    """One request whose rows all hold ROW, and a top-p value (float32) that
    puts P * S at A_2 (1 + rel): within the band for |rel| < 1e-5."""
    e = np.sort(np.exp(ROW.astype(np.float64) - ROW.max()))[::-1]
    P = np.float32(e[:2].sum() * (1.0 + rel) / e.sum())
    tgt = torch.from_numpy(np.tile(ROW, (gamma + 1, 1)))
    q = torch.full((gamma, 4), 0.25)
    ids = torch.full((gamma,), x, dtype=torch.int32)
    w = from_rows(tgt, q, ids, [gamma], T=1.0, seed=7)
    return w, torch.tensor([0], dtype=torch.int32), torch.tensor([P])


def _as_library(one):
    return dict(tokens=one.tokens.copy(), num_accepted=one.num_accepted.copy(),
                beta=one.beta.astype(np.float32), p_x=one.p_x.astype(np.float32),
                q_x=one.q_x.astype(np.float32), accept=one.accept.copy())


def _shifted(w, tk, tp, shift):
    return oracle.verify_request(0, w.target_logits.numpy(), w.draft_probs.numpy(),
                                 w.draft_ids.numpy(), w.T, w.seed, top_k=int(tk[0]),
                                 top_p=float(tp[0]), edge_shift=shift)


@pytest.mark.parametrize("rel", [-0.6e-5, 0.6e-5])
def test_a_result_on_another_reachable_cut_is_accepted(rel):
    w, tk, tp = _workload(rel)
    r = run_oracle(w, tk, tp)
    lo, hi = r.edge_lo[0], r.edge_hi[0]
    assert (lo, hi) != (0, 0)
    s = lo if lo else hi
    other = _shifted(w, tk, tp, [s, 0])
    assert other.status == 0
    assert abs(other.beta[0] - r.beta[0]) > 1e-5 or other.accept[0] != r.accept[0]
    st = compare(w, _as_library(other), r, top_k=tk, top_p=tp, label="")
    assert st["edge_requests"] == 1 and st["edge_shifted"] == 1
    st = compare(w, _as_library(r), r, top_k=tk, top_p=tp, label="")
    assert st["edge_requests"] == 1 and st["edge_shifted"] == 0


def test_a_result_no_reachable_cut_explains_fails():
    w, tk, tp = _workload(0.6e-5)
    r = run_oracle(w, tk, tp)
    bad = _as_library(r)
    bad["beta"][0] += 0.01
    with pytest.raises(AssertionError):
        compare(w, bad, r, top_k=tk, top_p=tp, label="")
    bad = _as_library(r)
    n = int(bad["num_accepted"][0])
    bad["tokens"][n] = (bad["tokens"][n] + 1) % 4
    with pytest.raises(AssertionError):
        compare(w, bad, r, top_k=tk, top_p=tp, label="")


def test_outside_the_band_only_the_exact_cut_passes():
    w, tk, tp = _workload(1.5e-5)
    r = run_oracle(w, tk, tp)
    assert r.edge_lo[0] == 0 and r.edge_hi[0] == 0
    st = compare(w, _as_library(r), r, top_k=tk, top_p=tp, label="")
    assert st["edge_requests"] == 0
    # what the shifted cut would have given is now a mistake
    e = np.exp(ROW.astype(np.float64) - ROW.max())
    keep = e[:2] / e[:2].sum()          # the cut one group earlier
    bad = _as_library(r)
    bad["beta"][0] = np.minimum(np.r_[keep, 0, 0], 0.25).sum()
    with pytest.raises(AssertionError):
        compare(w, bad, r, top_k=tk, top_p=tp, label="")


def test_flag_budget_counts_rows():
    assert flag_budget_ok(dict(flagged_rows=0, rows=10))
    assert not flag_budget_ok(dict(flagged_rows=8, rows=8192))           # 0.098 %
    assert flag_budget_ok(dict(flagged_rows=8, rows=100000))             # 0.008 %
    assert not flag_budget_ok(dict(flagged_rows=1, rows=9999))
