"""Request sharding across GPUs.

Requests are independent in the verify step (Algorithm 1 runs per request;
the vllbc notes describe vLLM's sampler scanning request by request over
cu_num_draft_tokens), so a batch splits across GPUs by contiguous request
ranges with no collective on the data path.  Each shard keeps its rows
contiguous, re-bases cu_num_draft_tokens to start at 0, and passes the index of
its first request as ``request_offset`` so that its random draws equal those of
one call over the whole batch.
"""
from __future__ import annotations

import torch

from .inputs import Workload


def shard_bounds(B: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous request range [b0, b1) of ``rank`` (sizes differ by at most 1)."""
    if not (0 <= rank < world):
        raise ValueError("rank out of range")
    return rank * B // world, (rank + 1) * B // world


def shard_workload(w: Workload, world: int, rank: int) -> tuple[Workload, int]:
    """The rows of requests [b0, b1) as a Workload of their own, and b0 (the
    request_offset to pass to the verifier)."""
    b0, b1 = shard_bounds(w.B, world, rank)
    cu = w.cu.to(torch.int64)
    d0, d1 = int(cu[b0]), int(cu[b1])
    t0, t1 = d0 + b0, d1 + b1
    sub_cu = (cu[b0:b1 + 1] - d0).to(torch.int32)
    sub = Workload(name=f"{w.name} [shard {rank}/{world}]", B=b1 - b0, V=w.V, dtype=w.dtype,
                   T=w.T, seed=w.seed, target_logits=w.target_logits[t0:t1],
                   draft_probs=None if w.draft_probs is None else w.draft_probs[d0:d1],
                   draft_ids=w.draft_ids[d0:d1], cu=sub_cu, meta=dict(w.meta))
    return sub, b0


def unshard(parts, cu: torch.Tensor):
    """Concatenates per-shard (tokens, num_accepted, beta) in rank order; the
    flattened layout of the whole batch is the concatenation of the shards'."""
    toks = torch.cat([p[0] for p in parts])
    nacc = torch.cat([p[1] for p in parts])
    beta = torch.cat([p[2] for p in parts])
    assert toks.numel() == int(cu[-1]) + cu.numel() - 1
    return toks, nacc, beta
