"""Token trees (several candidates per position): the CUDA library through
specdec_tree_verify against the CPU oracle, on seeded synthetic trees."""
import numpy as np
import pytest
import torch

import oracle
import stat_checks as sc
from gpu_helpers import FLAG_LOG, run_gpu
from speculative_decoding_rejection_decode_gb300.inputs import (from_rows, make_tree_workload,
                                                                to_numpy_logits)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def V():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_rejection_decode_gb300 import Verifier
    v = Verifier(0)
    yield v
    v.close()


def _run(v, w, request_offset=0):
    wd = w.to(v.device)
    out = v.tree(wd.target_logits, wd.draft_probs, wd.node_tokens, wd.node_parent, wd.cu, w.T,
                 w.seed, request_offset=request_offset)
    torch.cuda.synchronize()
    return (out.tokens.cpu().numpy(), out.num_accepted.cpu().numpy(), out.path.cpu().numpy())


def _oracle(w):
    return oracle.tree_verify(to_numpy_logits(w.target_logits),
                              None if w.draft_probs is None else w.draft_probs.cpu().numpy(),
                              w.node_tokens.cpu().numpy(), w.node_parent.cpu().numpy(),
                              w.cu.cpu().numpy(), w.T, w.seed)


def _compare(w, g, r, exact=False):
    tok, nacc, path = g
    cu = w.cu.cpu().numpy()
    flagged = rows = 0
    for b in range(w.B):
        s0, s1 = cu[b], cu[b + 1]
        rows += int(s1 - s0)
        if not exact and r.near_tie[b]:
            flagged += int(s1 - s0)
            continue
        assert nacc[b] == r.num_accepted[b], f"request {b}: depth"
        assert np.array_equal(tok[s0:s1], r.tokens[s0:s1]), f"request {b}: tokens"
        assert np.array_equal(path[s0:s1], r.path[s0:s1]), f"request {b}: path"
    import os
    label = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    acc = FLAG_LOG.setdefault(label, [0, 0, 0, 0, 0])
    acc[0] += int(sum(r.near_tie))
    acc[1] += flagged
    acc[2] += rows
    assert flagged == 0 or flagged < 1e-4 * rows, (flagged, rows)


@pytest.mark.parametrize("Vsz,dtype,T", [(1000, "f32", 1.0), (4099, "f32", 0.8), (32000, "bf16", 1.0),
                                         (8, "bf16", 1.3), (151936, "f32", 0.7)])
def test_random_trees_match_the_oracle(V, Vsz, dtype, T):
    w = make_tree_workload(name="random trees", B=64, V=Vsz, dtype=dtype, T=T, seed=Vsz % 97,
                           max_nodes=20, device="cuda")
    g = _run(V, w)
    assert V.get_error() == 0
    r = _oracle(w)
    assert r.status == 0
    _compare(w, g, r)
    assert r.num_accepted.max() >= 2          # the workload reaches below the first level


@pytest.mark.parametrize("shape", [[4, 2, 2], [2, 2, 2, 2], [8], [1, 1, 1, 1, 1, 1, 1]])
def test_full_trees_match_the_oracle(V, shape):
    w = make_tree_workload(name="full trees", B=48, V=20000, dtype="bf16", T=1.0, seed=len(shape),
                           shape=shape, device="cuda")
    g = _run(V, w)
    assert V.get_error() == 0
    _compare(w, g, _oracle(w))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_greedy_trees_bit_exact(V, dtype):
    w = make_tree_workload(name="greedy trees", B=64, V=3001, dtype=dtype, T=0.0, seed=5,
                           max_nodes=24, device="cuda")
    # a quarter of the candidates are the target argmax, so paths get deep
    tgt = w.target_logits.float()
    par = w.node_parent.long()
    cu = w.cu.long()
    base = torch.repeat_interleave(cu[:-1], torch.diff(cu))
    am = tgt.argmax(-1).to(torch.int32)
    gpar = base + par.clamp(min=0)
    pick = torch.rand(w.n_nodes, generator=torch.Generator().manual_seed(1)).to(w.node_tokens.device) < 0.5
    w.node_tokens = torch.where(pick & (par >= 0), am[gpar], w.node_tokens)
    g = _run(V, w)
    assert V.get_error() == 0
    r = _oracle(w)
    _compare(w, g, r, exact=True)
    assert r.num_accepted.max() >= 2


def test_chain_equals_the_chain_verifier(V):
    # the ragged standard shape as chains: node i + 1 the only child of node i
    from speculative_decoding_rejection_decode_gb300 import SPECDEC_PATH_SWEEP
    from speculative_decoding_rejection_decode_gb300.inputs import make_config
    w = make_config(3, device="cuda", B=48, V=20000)
    V.set_path(SPECDEC_PATH_SWEEP)      # the row kernel whose (max, sum) the tree walk shares
    lin = run_gpu(V, w, extended=False)
    V.set_path(0)
    cu = w.cu.cpu().numpy()
    B = w.B
    rows, par, tok, qrows = [], [], [], []
    ncu = [0]
    for b in range(B):
        g = cu[b + 1] - cu[b]
        t0 = cu[b] + b
        rows.append(w.target_logits[t0:t0 + g + 1])
        qrows.append(torch.cat([w.draft_probs[cu[b]:cu[b + 1]],
                                torch.full((1, w.V), 1.0 / w.V, device="cuda")]))
        par += [-1] + list(range(g))
        tok += [0] + w.draft_ids[cu[b]:cu[b + 1]].cpu().tolist()
        ncu.append(ncu[-1] + g + 1)
    tgt = torch.cat(rows).contiguous()
    q = torch.cat(qrows).contiguous()
    out = V.tree(tgt, q, torch.tensor(tok, dtype=torch.int32, device="cuda"),
                 torch.tensor(par, dtype=torch.int32, device="cuda"),
                 torch.tensor(ncu, dtype=torch.int32, device="cuda"), w.T, w.seed)
    torch.cuda.synchronize()
    assert V.get_error() == 0
    # same slots: request b's chain occupies cu[b] + b .. cu[b+1] + b in both
    assert np.array_equal(out.tokens.cpu().numpy(), lin["tokens"])
    assert np.array_equal(out.num_accepted.cpu().numpy(), lin["num_accepted"])


def test_first_token_follows_p(V):
    # three candidates drawn from q at the root, every child a leaf: the first
    # emitted token follows p whatever is accepted (chi-square, 300k trees)
    rng = np.random.default_rng(3)
    Vs, n, K = 6, 300_000, 3
    lr = np.array([0.4, -1.0, 1.1, 0.0, 0.7, -0.3], np.float32)
    qr = np.array([0.05, 0.3, 0.1, 0.35, 0.15, 0.05], np.float32)
    cand = rng.choice(Vs, size=(n, K), p=qr.astype(np.float64) / qr.astype(np.float64).sum())
    tgt = np.tile(np.concatenate([lr[None], np.zeros((K, Vs), np.float32)]), (n, 1))
    q = np.tile(np.concatenate([qr[None], np.full((K, Vs), 1.0 / Vs, np.float32)]), (n, 1))
    tok = np.zeros((n, K + 1), np.int32)
    tok[:, 1:] = cand
    par = np.tile(np.r_[-1, np.zeros(K, int)], n).astype(np.int32)
    cu = (np.arange(n + 1) * (K + 1)).astype(np.int32)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = V.tree(d(tgt.astype(np.float32)), d(q.astype(np.float32)), d(tok.reshape(-1)), d(par),
                 d(cu), 1.0, 11)
    torch.cuda.synchronize()
    first = out.tokens.cpu().numpy().reshape(n, K + 1)[:, 0]
    assert sc.chi2_ok(np.bincount(first, minlength=Vs), sc.softmax64(lr, 1.0)) > sc.P_MIN
    beta = np.minimum(sc.softmax64(lr, 1.0), qr).sum()
    acc0 = (out.path.cpu().numpy().reshape(n, K + 1)[:, 0] == 1).mean()
    assert abs(acc0 - beta) < 3 * np.sqrt(beta * (1 - beta) / n)


def test_malformed_trees_and_bad_tokens(V):
    from speculative_decoding_rejection_decode_gb300._lib import (SPECDEC_DEVERR_BAD_DRAFT_ID,
                                                                  SPECDEC_DEVERR_BAD_TREE)
    w = make_tree_workload(name="bad", B=6, V=512, dtype="f32", T=1.0, seed=9, max_nodes=8,
                           device="cuda")
    cu = w.cu.cpu().numpy()
    # request 2: a parent that is not an earlier node; request 4: a token past V
    par = w.node_parent.clone()
    if cu[3] - cu[2] > 1:
        par[cu[2] + 1] = 5
    else:
        par[cu[2]] = 0
    w.node_parent = par
    if cu[5] - cu[4] > 1:
        w.node_tokens[cu[4] + 1] = 10 ** 6
    g = _run(V, w)
    err = V.get_error()
    assert err & SPECDEC_DEVERR_BAD_TREE
    r = _oracle(w)
    assert r.status == oracle.INVALID_ARG       # the oracle refuses the whole batch
    ok = [b for b in range(w.B) if b != 2]
    for b in ok:
        s0, s1 = cu[b], cu[b + 1]
        one = oracle.tree_verify_request(b, to_numpy_logits(w.target_logits[s0:s1]),
                                         w.draft_probs[s0:s1].cpu().numpy(),
                                         w.node_tokens[s0:s1].cpu().numpy(),
                                         w.node_parent[s0:s1].cpu().numpy(), w.T, w.seed)
        if b == 4 and cu[5] - cu[4] > 1:
            assert one.status == oracle.BAD_DRAFT_ID
        if one.near_tie[0]:
            continue
        assert g[1][b] == one.num_accepted[0]
        assert np.array_equal(g[0][s0:s1], one.tokens)
    if cu[5] - cu[4] > 1:
        assert err & SPECDEC_DEVERR_BAD_DRAFT_ID


def test_request_offset_shards(V):
    w = make_tree_workload(name="shards", B=20, V=3000, dtype="f32", T=1.0, seed=13, device="cuda")
    whole = _run(V, w)
    cu = w.cu.cpu().numpy()
    b0 = 8
    s0 = cu[b0]
    out = V.tree(w.target_logits[s0:], w.draft_probs[s0:], w.node_tokens[s0:], w.node_parent[s0:],
                 (w.cu[b0:] - s0).contiguous(), w.T, w.seed, request_offset=b0)
    torch.cuda.synchronize()
    assert np.array_equal(out.tokens.cpu().numpy(), whole[0][s0:])
    assert np.array_equal(out.num_accepted.cpu().numpy(), whole[1][b0:])


def test_host_argument_errors(V):
    from speculative_decoding_rejection_decode_gb300 import specdec_tree_verify
    from speculative_decoding_rejection_decode_gb300._lib import (SPECDEC_ERR_INVALID_ARG,
                                                                  SPECDEC_ERR_UNSUPPORTED_DTYPE)
    w = make_tree_workload(name="args", B=2, V=64, dtype="f32", T=1.0, seed=1,
                           device="cuda")
    out = torch.empty(w.n_nodes, dtype=torch.int32, device="cuda")
    base = dict(h=V.handle, target_logits=w.target_logits.data_ptr(), dtype=0,
                draft_probs=w.draft_probs.data_ptr(), node_tokens=w.node_tokens.data_ptr(),
                node_parent=w.node_parent.data_ptr(), cu_num_nodes=w.cu.data_ptr(), B=2, V=64,
                T=1.0, seed=0, request_offset=0, out_tokens=out.data_ptr(),
                out_num_accepted=out.data_ptr(), out_path=None,
                stream=torch.cuda.current_stream().cuda_stream)
    for k, v, want in (("B", 0, SPECDEC_ERR_INVALID_ARG), ("V", 0, SPECDEC_ERR_INVALID_ARG),
                       ("T", -1.0, SPECDEC_ERR_INVALID_ARG), ("T", float("nan"), SPECDEC_ERR_INVALID_ARG),
                       ("dtype", 5, SPECDEC_ERR_UNSUPPORTED_DTYPE),
                       ("draft_probs", None, SPECDEC_ERR_INVALID_ARG),
                       ("node_parent", None, SPECDEC_ERR_INVALID_ARG),
                       ("h", None, SPECDEC_ERR_INVALID_ARG)):
        args = dict(base)
        args[k] = v
        assert specdec_tree_verify(*args.values()) == want, k
