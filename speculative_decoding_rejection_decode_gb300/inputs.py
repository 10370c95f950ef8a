"""Seeded synthetic inputs for the speculative-sampling verifier.

This module holds none of the verifier's arithmetic: it plays the part of the
two models that are out of scope.  The target model becomes Gaussian logits,
the drafter becomes a softmax of those logits plus Gaussian noise (a stand-in
for a smaller model whose distribution overlaps the target's), and the draft
ids are drawn from the drafter's rows, exactly as Algorithm 1 draws
x_i ~ q_i.  Tests and the benchmark build their inputs here; the CPU oracle and
the CUDA library both receive the same tensors.

Layout (the flattened ragged batch of the vLLM verification path described on
the vllbc reading-notes page): request b has gamma_b drafts;
cu[b+1] = cu[b] + gamma_b; draft row / id of (b, i) is cu[b] + i; target row of
(b, i), i in [0, gamma_b], is cu[b] + b + i (the last one is the bonus row).

The five standard workloads:
  0 tiny     B=1,    gamma=4,        V=32,     f32 N(0,2^2),  q=softmax(L+N(0,0.5^2)),      T=1
  1 small    B=8,    gamma=5,        V=32000,  f32 N(0,3^2),  q=softmax((L+N(0,1))/T),      T=1
  2 greedy   B=64,   gamma=7,        V=128256, bf16 N(0,3^2), ids=argmax w.p. 0.75 else uniform, T=0
  3 ragged   B=256,  gamma~U{1..8},  V=151936, f32 N(0,3^2),  q=softmax((L+N(0,1.5^2))/0.7), T=0.7
  4 large    B=1024, gamma=7,        V=256000, bf16 N(0,3^2), q=softmax(L+N(0,1)),          T=1
Workload k uses generator seed k and verifier seed k.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass
class Workload:
    name: str
    B: int
    V: int
    dtype: str                      # "f32" or "bf16" (target logits)
    T: float
    seed: int                       # the verifier's generator seed
    target_logits: torch.Tensor     # [N_t, V] float32 or bfloat16
    draft_probs: torch.Tensor | None  # [N_d, V] float32, or None (greedy)
    draft_ids: torch.Tensor         # [N_d] int32
    cu: torch.Tensor                # [B+1] int32
    meta: dict = field(default_factory=dict)

    @property
    def n_draft(self) -> int:
        return int(self.cu[-1])

    @property
    def n_target(self) -> int:
        return self.n_draft + self.B

    def algorithmic_bytes(self) -> int:
        """One read of every target and draft row plus one extra target row per
        request (the correction / bonus row)."""
        esize = 2 if self.dtype == "bf16" else 4
        tb = self.n_target * self.V * esize
        db = 0 if self.draft_probs is None else self.n_draft * self.V * 4
        extra = 0 if self.T == 0 else self.B * self.V * esize
        return tb + db + extra

    def to(self, device) -> "Workload":
        mv = lambda t: None if t is None else t.to(device)
        return Workload(self.name, self.B, self.V, self.dtype, self.T, self.seed,
                        mv(self.target_logits), mv(self.draft_probs), mv(self.draft_ids),
                        mv(self.cu), dict(self.meta))


STANDARD_WORKLOADS = {
    0: dict(name="tiny B=1 gamma=4 V=32 f32 T=1", B=1, gamma=4, V=32, dtype="f32", T=1.0,
            target_std=2.0, noise_std=0.5, draft_T=1.0, ids="sample"),
    1: dict(name="B=8 gamma=5 V=32000 f32 T=1", B=8, gamma=5, V=32000, dtype="f32", T=1.0,
            target_std=3.0, noise_std=1.0, draft_T=1.0, ids="sample"),
    2: dict(name="greedy B=64 gamma=7 V=128256 bf16 T=0", B=64, gamma=7, V=128256, dtype="bf16",
            T=0.0, target_std=3.0, noise_std=None, draft_T=None, ids="argmax0.75"),
    3: dict(name="ragged B=256 gamma~U{1..8} V=151936 f32 T=0.7", B=256, gamma=(1, 8), V=151936,
            dtype="f32", T=0.7, target_std=3.0, noise_std=1.5, draft_T=0.7, ids="sample"),
    4: dict(name="large B=1024 gamma=7 V=256000 bf16 T=1", B=1024, gamma=7, V=256000, dtype="bf16",
            T=1.0, target_std=3.0, noise_std=1.0, draft_T=1.0, ids="sample"),
}


def make_config(idx: int, device="cpu", B: int | None = None, V: int | None = None,
                chunk_rows: int = 512) -> Workload:
    """Standard workload ``idx`` (0..4), optionally with a smaller batch or vocabulary."""
    c = dict(STANDARD_WORKLOADS[idx])
    if B is not None:
        c["B"] = B
    if V is not None:
        c["V"] = V
    name = c["name"] if (B is None and V is None) else f"{c['name']} (B={c['B']}, V={c['V']})"
    return make_workload(name=name, B=c["B"], gamma=c["gamma"], V=c["V"], dtype=c["dtype"],
                         T=c["T"], seed=idx, target_std=c["target_std"], noise_std=c["noise_std"],
                         draft_T=c["draft_T"], ids=c["ids"], device=device, chunk_rows=chunk_rows)


def make_workload(*, name: str, B: int, gamma, V: int, dtype: str, T: float, seed: int,
                  target_std: float = 3.0, noise_std: float | None = 1.0,
                  draft_T: float | None = None, ids: str = "sample", device="cpu",
                  chunk_rows: int = 512) -> Workload:
    """Generic generator.  ``gamma`` is an int or an inclusive range (lo, hi)
    drawn per request; ``ids`` is "sample" (x ~ q) or "argmax0.75" (greedy
    drafts that match the target argmax with probability 0.75)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    if isinstance(gamma, tuple):
        gam = torch.randint(gamma[0], gamma[1] + 1, (B,), generator=g, device=dev)
    else:
        gam = torch.full((B,), int(gamma), dtype=torch.int64, device=dev)
    cu = torch.zeros(B + 1, dtype=torch.int64, device=dev)
    cu[1:] = torch.cumsum(gam, 0)
    n_d = int(cu[-1])
    n_t = n_d + B
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    logits = torch.empty(n_t, V, dtype=tdt, device=dev)
    for r0 in range(0, n_t, chunk_rows):
        r1 = min(n_t, r0 + chunk_rows)
        blk = torch.randn(r1 - r0, V, generator=g, device=dev) * target_std
        logits[r0:r1] = blk.to(tdt)

    # Target row of draft position d: d + (request index of d).
    req_of_draft = torch.repeat_interleave(torch.arange(B, device=dev), gam, output_size=n_d)
    tgt_row_of_draft = torch.arange(n_d, device=dev) + req_of_draft

    draft_probs = None
    draft_ids = torch.empty(n_d, dtype=torch.int32, device=dev)
    if ids == "sample":
        draft_probs = torch.empty(n_d, V, dtype=torch.float32, device=dev)
        dT = 1.0 if draft_T is None else float(draft_T)
        for d0 in range(0, n_d, chunk_rows):
            d1 = min(n_d, d0 + chunk_rows)
            base = logits[tgt_row_of_draft[d0:d1]].float()
            noisy = base + torch.randn(d1 - d0, V, generator=g, device=dev) * noise_std
            q = torch.softmax(noisy / dT, dim=-1)
            draft_probs[d0:d1] = q
            draft_ids[d0:d1] = torch.multinomial(q, 1, generator=g).squeeze(1).to(torch.int32)
    elif ids == "argmax0.75":
        for d0 in range(0, n_d, chunk_rows):
            d1 = min(n_d, d0 + chunk_rows)
            rows = logits[tgt_row_of_draft[d0:d1]].float()
            am = torch.argmax(rows, dim=-1)      # first maximal index
            hit = torch.rand(d1 - d0, generator=g, device=dev) < 0.75
            rnd = torch.randint(0, V, (d1 - d0,), generator=g, device=dev)
            draft_ids[d0:d1] = torch.where(hit, am, rnd).to(torch.int32)
    else:
        raise ValueError(ids)
    return Workload(name=name, B=B, V=V, dtype=dtype, T=float(T), seed=seed,
                    target_logits=logits, draft_probs=draft_probs, draft_ids=draft_ids,
                    cu=cu.to(torch.int32), meta=dict(gamma=gamma, target_std=target_std,
                                                     noise_std=noise_std, draft_T=draft_T, ids=ids))


def to_numpy_logits(t: torch.Tensor):
    """Target logits as numpy: float32, or the uint16 bit patterns of bf16."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()


def from_rows(target_logits: torch.Tensor, draft_probs: torch.Tensor | None,
              draft_ids: torch.Tensor, gammas, T: float, seed: int, name: str = "custom") -> Workload:
    """Wraps hand-built tensors in a Workload (edge-case tests)."""
    gam = torch.as_tensor(list(gammas), dtype=torch.int64)
    cu = torch.zeros(len(gam) + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(gam, 0)
    dtype = "bf16" if target_logits.dtype == torch.bfloat16 else "f32"
    return Workload(name=name, B=len(gam), V=target_logits.shape[-1], dtype=dtype, T=float(T),
                    seed=seed, target_logits=target_logits, draft_probs=draft_probs,
                    draft_ids=draft_ids.to(torch.int32), cu=cu.to(torch.int32))


TOP_K_CHOICES = (1, 2, 5, 20, 50, 200, 1000)
TOP_P_CHOICES = (0.99, 0.95, 0.9, 0.8, 0.5, 0.2)


def make_top_k_top_p(B: int, V: int, seed: int, top_k: int | None = None,
                     top_p: float | None = None, device="cpu"):
    """Per-request top-k (int32 [B]) and top-p (float32 [B]) settings.

    With ``top_k`` / ``top_p`` given, every request gets that value.  Otherwise
    a seeded mix: a fifth of the requests use top-k only, a fifth top-p only,
    two fifths both, the rest neither, with values drawn from common settings
    plus the edge values the interface defines (k = V - 1, V, V + 7, 0 and -1;
    p = 0, 1e-6, 1 and 1.5)."""
    if top_k is not None or top_p is not None:
        k = torch.full((B,), 0 if top_k is None else int(top_k), dtype=torch.int32)
        p = torch.full((B,), 1.0 if top_p is None else float(top_p), dtype=torch.float32)
        return k.to(device), p.to(device)
    g = torch.Generator()
    g.manual_seed(seed)
    ks = list(TOP_K_CHOICES) + [V - 1, V, V + 7, 0, -1]
    ps = list(TOP_P_CHOICES) + [0.0, 1e-6, 1.0, 1.5]
    kind = torch.randint(0, 5, (B,), generator=g)
    ki = torch.randint(0, len(ks), (B,), generator=g)
    pi = torch.randint(0, len(ps), (B,), generator=g)
    k = torch.tensor([ks[i] for i in ki.tolist()], dtype=torch.int32)
    p = torch.tensor([ps[i] for i in pi.tolist()], dtype=torch.float32)
    k = torch.where((kind == 0) | (kind == 2) | (kind == 3), k, torch.zeros_like(k))
    p = torch.where((kind == 1) | (kind == 2) | (kind == 3), p, torch.ones_like(p))
    return k.to(device), p.to(device)


# ----------------------------------------------------------------------------
# Token trees (several candidates per position)
# ----------------------------------------------------------------------------

@dataclass
class TreeWorkload:
    name: str
    B: int
    V: int
    dtype: str
    T: float
    seed: int
    target_logits: torch.Tensor     # [N, V]: the target's row after every node
    draft_probs: torch.Tensor | None  # [N, V] float32: the drafter's row at every node
    node_tokens: torch.Tensor       # [N] int32 (node 0 of a request: 0)
    node_parent: torch.Tensor       # [N] int32, within the request (node 0: -1)
    cu: torch.Tensor                # [B+1] int32 node offsets

    @property
    def n_nodes(self) -> int:
        return int(self.cu[-1])

    def to(self, device) -> "TreeWorkload":
        mv = lambda t: None if t is None else t.to(device)
        return TreeWorkload(self.name, self.B, self.V, self.dtype, self.T, self.seed,
                            mv(self.target_logits), mv(self.draft_probs), mv(self.node_tokens),
                            mv(self.node_parent), mv(self.cu))


def tree_shape(branching) -> list[int]:
    """Parents of a full tree whose level d nodes have branching[d] children
    each, in breadth-first order (node 0 the root)."""
    par = [-1]
    level = [0]
    for k in branching:
        nxt = []
        for u in level:
            for _ in range(k):
                par.append(u)
                nxt.append(len(par) - 1)
        level = nxt
    return par


def make_tree_workload(*, name: str, B: int, V: int, dtype: str, T: float, seed: int,
                       shape="random", max_nodes: int = 16, target_std: float = 3.0,
                       noise_std: float = 1.0, device="cpu", chunk_rows: int = 512) -> TreeWorkload:
    """Synthetic token trees.  ``shape`` is "random" (each request gets 1 ..
    max_nodes nodes, every node's parent drawn uniformly from the earlier
    nodes) or a list of per-level branching factors (the same full tree for
    every request).  Target rows ~ N(0, target_std^2) (bf16 or f32); the
    drafter's row at node u is softmax((L_u + N(0, noise_std^2)) / T) of that
    node's own target row (T = 1 for greedy); the token of node j is drawn
    from the drafter's row at its parent, independently for every child, as the
    candidates of a tree drafter are."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    pars = []
    for b in range(B):
        if shape == "random":
            n = int(torch.randint(1, max_nodes + 1, (1,), generator=g))
            par = [-1] + [int(torch.randint(0, j, (1,), generator=g)) for j in range(1, n)]
        else:
            par = tree_shape(shape)
        pars.append(par)
    sizes = torch.tensor([len(p) for p in pars], dtype=torch.int64)
    cu = torch.zeros(B + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(sizes, 0)
    N = int(cu[-1])
    dev = torch.device(device)
    gd = torch.Generator(device=dev)
    gd.manual_seed(seed + 1)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    logits = torch.empty(N, V, dtype=tdt, device=dev)
    q = torch.empty(N, V, dtype=torch.float32, device=dev)
    dT = float(T) if T > 0 else 1.0
    for r0 in range(0, N, chunk_rows):          # in row blocks: no full-size temporaries
        r1 = min(N, r0 + chunk_rows)
        logits[r0:r1] = (torch.randn(r1 - r0, V, generator=gd, device=dev) * target_std).to(tdt)
        noisy = logits[r0:r1].float() + torch.randn(r1 - r0, V, generator=gd, device=dev) * noise_std
        q[r0:r1] = torch.softmax(noisy / dT, dim=-1)
    parent = torch.tensor([p for par in pars for p in par], dtype=torch.int32)
    base = torch.repeat_interleave(cu[:-1], sizes)
    gpar = (base + parent.to(torch.int64).clamp(min=0)).to(dev)
    tokens = torch.multinomial(q[gpar], 1, generator=gd).squeeze(1).to(torch.int32)
    root = (parent == -1).to(dev)
    tokens = torch.where(root, torch.zeros_like(tokens), tokens)
    return TreeWorkload(name=name, B=B, V=V, dtype=dtype, T=float(T), seed=seed,
                        target_logits=logits, draft_probs=q if T > 0 else None,
                        node_tokens=tokens, node_parent=parent.to(dev), cu=cu.to(torch.int32).to(dev))
