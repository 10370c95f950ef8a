"""Helpers for the GPU parity tests: run the CUDA library through its C ABI
(via the package's ctypes binding) and compare with the CPU oracle."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from speculative_decoding_rejection_decode_gb300.inputs import Workload, to_numpy_logits

BETA_TOL = 1e-5      # absolute, beta and probabilities (sampling mode)
PROB_TOL = 1e-5


def run_gpu(verifier, w: Workload, extended: bool = True):
    dev = verifier.device
    wd = w.to(dev)
    out = verifier(wd.target_logits, wd.draft_probs, wd.draft_ids, wd.cu, w.T, w.seed,
                   extended=extended, n_draft=w.n_draft)
    torch.cuda.synchronize(dev)
    res = dict(tokens=out.tokens.cpu().numpy(), num_accepted=out.num_accepted.cpu().numpy(),
               beta=out.beta.cpu().numpy())
    if extended:
        res.update(p_x=out.target_prob.cpu().numpy(), q_x=out.draft_prob.cpu().numpy(),
                   accept=out.accept.cpu().numpy())
    return res


def run_oracle(w: Workload, top_k=None, top_p=None):
    q = None if w.draft_probs is None else w.draft_probs.cpu().numpy()
    tk = None if top_k is None else np.asarray(top_k.cpu() if hasattr(top_k, "cpu") else top_k)
    tp = None if top_p is None else np.asarray(top_p.cpu() if hasattr(top_p, "cpu") else top_p)
    return oracle.rejection_sample(to_numpy_logits(w.target_logits), q, w.draft_ids.cpu().numpy(),
                                   w.cu.cpu().numpy(), w.T, w.seed, top_k=tk, top_p=tp)


def run_gpu_adj(verifier, w: Workload, top_k, top_p, extended: bool = True):
    """The top-k / top-p entry point (top_k / top_p: torch tensors or None)."""
    dev = verifier.device
    wd = w.to(dev)
    tk = None if top_k is None else top_k.to(dev)
    tp = None if top_p is None else top_p.to(dev)
    out = verifier(wd.target_logits, wd.draft_probs, wd.draft_ids, wd.cu, w.T, w.seed,
                   extended=extended, n_draft=w.n_draft, top_k=tk, top_p=tp)
    torch.cuda.synchronize(dev)
    res = dict(tokens=out.tokens.cpu().numpy(), num_accepted=out.num_accepted.cpu().numpy(),
               beta=out.beta.cpu().numpy())
    if extended:
        res.update(p_x=out.target_prob.cpu().numpy(), q_x=out.draft_prob.cpu().numpy(),
                   accept=out.accept.cpu().numpy())
    return res


def compare(w: Workload, g: dict, r: oracle.OracleResult, exact: bool = False,
            requests=None) -> dict:
    """Element-by-element comparison.  Greedy (exact=True): everything
    bit-exact.  Sampling: tokens / counts identical on requests the oracle does
    not flag as near ties, probabilities and beta within 1e-5."""
    cu = w.cu.cpu().numpy().astype(np.int64)
    B = len(cu) - 1
    reqs = range(B) if requests is None else requests
    flagged = 0
    for b in reqs:
        d0, d1 = cu[b], cu[b + 1]
        t0, t1 = d0 + b, d1 + b + 1
        if not exact and r.near_tie[b]:
            flagged += 1
            continue
        assert g["num_accepted"][b] == r.num_accepted[b], f"request {b}: n"
        assert np.array_equal(g["tokens"][t0:t1], r.tokens[t0:t1]), f"request {b}: tokens"
    d_all = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in reqs]) if len(cu) > 1 else []
    d_all = np.asarray(d_all, np.int64)
    if d_all.size:
        if exact:
            assert np.array_equal(g["beta"][d_all], r.beta[d_all].astype(np.float32))
            if "accept" in g:
                assert np.array_equal(g["accept"][d_all], r.accept[d_all])
                assert np.array_equal(g["p_x"][d_all], r.p_x[d_all].astype(np.float32))
        else:
            db = np.abs(g["beta"][d_all] - r.beta[d_all])
            assert db.max() <= BETA_TOL, f"beta max err {db.max()}"
            if "p_x" in g:
                assert np.abs(g["p_x"][d_all] - r.p_x[d_all]).max() <= PROB_TOL
                assert np.abs(g["q_x"][d_all] - r.q_x[d_all]).max() <= PROB_TOL
                ok = r.pos_near_tie[d_all] == 0
                assert np.array_equal(g["accept"][d_all][ok], r.accept[d_all][ok])
    n_req = len(list(reqs))
    return dict(flagged=flagged, requests=n_req)


def flag_budget_ok(flagged: int, n_requests: int) -> bool:
    """Near-tie exemptions must stay under 0.01 % of rows (at least one allowed
    on small batches)."""
    return flagged <= max(1, math.ceil(1e-4 * n_requests))


def sampled_oracle(w: Workload, requests, top_k=None, top_p=None):
    """Oracle results for a few requests of a large workload, one at a time,
    scattered into full-size arrays (entries of other requests are unset)."""
    cu = w.cu.cpu().numpy().astype(np.int64)
    n_t, n_d, B = w.n_target, w.n_draft, w.B
    res = oracle.OracleResult(tokens=np.full(n_t, -2, np.int32), num_accepted=np.zeros(B, np.int32),
                              beta=np.zeros(n_d), p_x=np.zeros(n_d), q_x=np.zeros(n_d),
                              accept=np.zeros(n_d, np.int32), pos_near_tie=np.zeros(n_d, np.int32),
                              near_tie=np.zeros(B, np.int32), status=0)
    tk = None if top_k is None else top_k.cpu().numpy()
    tp = None if top_p is None else top_p.cpu().numpy()
    for b in requests:
        d0, d1 = cu[b], cu[b + 1]
        t0, t1 = d0 + b, d1 + b + 1
        tgt = to_numpy_logits(w.target_logits[t0:t1])
        q = None if w.draft_probs is None else w.draft_probs[d0:d1].cpu().numpy()
        one = oracle.verify_request(int(b), tgt, q, w.draft_ids[d0:d1].cpu().numpy(), w.T, w.seed,
                                    top_k=0 if tk is None else int(tk[b]),
                                    top_p=1.0 if tp is None else float(tp[b]))
        res.tokens[t0:t1] = one.tokens
        res.num_accepted[b] = one.num_accepted[0]
        res.beta[d0:d1] = one.beta
        res.p_x[d0:d1] = one.p_x
        res.q_x[d0:d1] = one.q_x
        res.accept[d0:d1] = one.accept
        res.pos_near_tie[d0:d1] = one.pos_near_tie
        res.near_tie[b] = one.near_tie[0]
    return res


def numpy_runner(verifier, path=None):
    """A run(tgt, q, ids, cu, T, seed) callable over numpy inputs for the shared
    statistical checks."""
    def run(tgt, q, ids, cu, T, seed):
        if path is not None:
            verifier.set_path(path)
        dev = verifier.device
        tt = torch.from_numpy(np.ascontiguousarray(tgt)).to(dev)
        qq = None if q is None else torch.from_numpy(np.ascontiguousarray(q, np.float32)).to(dev)
        ii = torch.from_numpy(np.ascontiguousarray(ids, np.int32)).to(dev)
        cc = torch.from_numpy(np.ascontiguousarray(cu, np.int32)).to(dev)
        out = verifier(tt, qq, ii, cc, T, seed, extended=True, n_draft=int(cu[-1]))
        torch.cuda.synchronize(dev)
        assert verifier.get_error() == 0
        return (out.tokens.cpu().numpy(), out.num_accepted.cpu().numpy(),
                out.accept.cpu().numpy(), out.beta.cpu().numpy().astype(np.float64))
    return run
