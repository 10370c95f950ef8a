"""Multi-process path on CPU (gloo, world size 2): request sharding with
re-based cu and request offsets reproduces the unsharded batch exactly, and the
bench's timing reduction takes the max over ranks.  The per-shard verifier is
the CPU oracle called with global request indices (the same contract the CUDA
library's request_offset implements)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _verify_shard(w, offset):
    import oracle
    from speculative_decoding_rejection_decode_gb300.inputs import to_numpy_logits
    cu = w.cu.numpy().astype(np.int64)
    toks, nacc, beta = [], [], []
    for b in range(w.B):
        d0, d1 = cu[b], cu[b + 1]
        r = oracle.verify_request(offset + b, to_numpy_logits(w.target_logits[d0 + b:d1 + b + 1]),
                                  w.draft_probs[d0:d1].numpy(), w.draft_ids[d0:d1].numpy(), w.T,
                                  w.seed)
        toks.append(r.tokens)
        nacc.append(r.num_accepted)
        beta.append(r.beta)
    return (torch.from_numpy(np.concatenate(toks)), torch.from_numpy(np.concatenate(nacc)),
            torch.from_numpy(np.concatenate(beta)))


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    try:
        import bench
        from speculative_decoding_rejection_decode_gb300.inputs import make_config
        from speculative_decoding_rejection_decode_gb300.sharding import shard_workload, unshard
        d = bench.Dist()
        w = make_config(3, B=9, V=300)
        sub, off = shard_workload(w, world, rank)
        mine = _verify_shard(sub, off)
        parts = [None] * world
        dist.all_gather_object(parts, mine)
        tmax = d.max(float(rank + 1) * 0.5)
        d.barrier()
        if rank == 0:
            toks, nacc, beta = unshard(parts, w.cu)
            full = _verify_shard(w, 0)
            ok = (torch.equal(toks, full[0]) and torch.equal(nacc, full[1])
                  and torch.equal(beta, full[2]) and tmax == world * 0.5)
            q.put(("ok" if ok else "mismatch", sub.B))
        d.close()
    except Exception as e:  # pragma: no cover - reported to the parent
        q.put(("error", repr(e)))
        raise


def test_two_rank_request_sharding_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs)
    status, detail = q.get(timeout=5)
    assert status == "ok", detail


def test_shard_bounds_cover_batch():
    from speculative_decoding_rejection_decode_gb300.sharding import shard_bounds
    for B in (1, 7, 1024):
        for world in (1, 2, 3, 8):
            spans = [shard_bounds(B, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == B
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            assert max(s[1] - s[0] for s in spans) - min(s[1] - s[0] for s in spans) <= 1
