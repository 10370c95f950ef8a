"""Torch-facing wrapper of libspecdec.so: argument marshalling only (every
step of the verifier runs in the library's CUDA kernels)."""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import _lib
from ._lib import (SPECDEC_BF16, SPECDEC_F32, SPECDEC_PATH_AUTO, SPECDEC_PATH_DUAL,  # noqa: F401
                   SPECDEC_PATH_FUSED, SPECDEC_PATH_GREEDY, SPECDEC_PATH_PAIR, SPECDEC_PATH_STREAM, SPECDEC_PATH_SWEEP,
                   SPECDEC_PATH_TWO_PASS, specdec_create, specdec_destroy,
                   specdec_get_error, specdec_last_path, specdec_neg_log_uniform,
                   specdec_selection_mass,
                   specdec_rejection_sample, specdec_rejection_sample_ex,
                   specdec_rejection_sample_noalloc, specdec_rejection_sample_topk_topp,
                   specdec_reserve, specdec_set_adjust_counters,
                   specdec_set_path, specdec_set_timing_events, specdec_status_string,
                   specdec_tree_verify, specdec_uniform)


class SpecdecError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        super().__init__(f"{what}: {specdec_status_string(status)} ({status})")
        self.status = status


def _check(rc: int, what: str):
    if rc != 0:
        raise SpecdecError(rc, what)


@dataclass
class VerifyOutput:
    tokens: torch.Tensor         # int32 [N_t]
    num_accepted: torch.Tensor   # int32 [B]
    beta: torch.Tensor | None    # float32 [N_d]
    target_prob: torch.Tensor | None = None   # float32 [N_d] p_i(x_i)
    draft_prob: torch.Tensor | None = None    # float32 [N_d] q_i(x_i)
    accept: torch.Tensor | None = None        # int32 [N_d]


def _ptr(t):
    return 0 if t is None else t.data_ptr()


def _stream_handle(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


class Verifier:
    """One library handle on one CUDA device."""

    def __init__(self, device: int | torch.device = 0):
        dev = torch.device("cuda", device) if isinstance(device, int) else torch.device(device)
        if dev.type != "cuda":
            raise ValueError("the verifier runs on a CUDA device")
        self.device = dev
        idx = dev.index if dev.index is not None else torch.cuda.current_device()
        rc, self._h = specdec_create(idx)
        _check(rc, "specdec_create")
        # a valid device address for required arrays that are empty (draft_ids
        # when every request has gamma = 0): the C ABI wants a pointer even then
        self._empty = torch.zeros(4, dtype=torch.int32, device=dev)

    def _ids_ptr(self, draft_ids) -> int:
        if draft_ids is not None and draft_ids.numel() == 0:
            return self._empty.data_ptr()
        return _ptr(draft_ids)

    def close(self):
        if getattr(self, "_h", 0):
            specdec_destroy(self._h)
            self._h = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self) -> int:
        return self._h

    def reserve(self, max_draft_positions: int, max_batch: int):
        _check(specdec_reserve(self._h, max_draft_positions, max_batch), "specdec_reserve")

    def set_timing_events(self, before_rows, after_rows):
        """torch.cuda.Event pair (already recorded once, so that the CUDA event
        exists) recorded around the row kernel of every later call; None, None
        to stop."""
        a = None if before_rows is None else before_rows.cuda_event
        b = None if after_rows is None else after_rows.cuda_event
        _check(specdec_set_timing_events(self._h, a, b), "specdec_set_timing_events")

    def set_adjust_counters(self, counters: torch.Tensor | None):
        """int64 [8] device tensor that later calls add their top-k / top-p
        selection statistics to (see specdec_set_adjust_counters); None stops."""
        if counters is not None and (counters.device != self.device or counters.dtype != torch.int64
                                     or counters.numel() < 8):
            raise ValueError("counters must be an int64 tensor of 8 entries on the device")
        _check(specdec_set_adjust_counters(self._h, _ptr(counters)), "specdec_set_adjust_counters")

    def set_path(self, path: int):
        _check(specdec_set_path(self._h, path), "specdec_set_path")

    def last_path(self) -> tuple[int, int]:
        rc, p, c = specdec_last_path(self._h)
        _check(rc, "specdec_last_path")
        return p, c

    def get_error(self) -> int:
        rc, e = specdec_get_error(self._h, _stream_handle(self.device))
        _check(rc, "specdec_get_error")
        return e

    def tree(self, target_logits: torch.Tensor, draft_probs: torch.Tensor | None,
             node_tokens: torch.Tensor, node_parent: torch.Tensor, cu_num_nodes: torch.Tensor,
             T: float, seed: int, *, request_offset: int = 0, with_path: bool = True,
             out: "TreeOutput | None" = None) -> "TreeOutput":
        """Verifies token trees (several candidates per position) on the current
        torch stream: specdec_tree_verify.  One target and one draft row per
        node; node_parent holds indices within each request (node 0: -1)."""
        return _tree_call(self, target_logits, draft_probs, node_tokens, node_parent,
                          cu_num_nodes, T, seed, request_offset, with_path, out)

    def __call__(self, target_logits: torch.Tensor, draft_probs: torch.Tensor | None,
                 draft_ids: torch.Tensor, cu_num_draft_tokens: torch.Tensor, T: float, seed: int,
                 *, with_beta: bool = True, extended: bool = False,
                 out: VerifyOutput | None = None, n_draft: int | None = None,
                 request_offset: int = 0, top_k: torch.Tensor | None = None,
                 top_p: torch.Tensor | None = None) -> VerifyOutput:
        """Runs one verify step on the current torch stream.  ``n_draft`` (= cu[B])
        avoids a host read of cu when output tensors must be allocated.
        ``top_k`` (int32 [B]) / ``top_p`` (float32 [B]) restrict the target
        distribution per request (specdec_rejection_sample_topk_topp)."""
        for t in (target_logits, draft_ids, cu_num_draft_tokens):
            if t.device != self.device or not t.is_contiguous():
                raise ValueError("inputs must be contiguous tensors on the verifier's device")
        if draft_probs is not None and (draft_probs.device != self.device
                                        or draft_probs.dtype != torch.float32
                                        or not draft_probs.is_contiguous()):
            raise ValueError("draft_probs must be a contiguous float32 tensor on the device")
        if target_logits.dtype == torch.float32:
            dtype = SPECDEC_F32
        elif target_logits.dtype == torch.bfloat16:
            dtype = SPECDEC_BF16
        else:
            raise TypeError("target_logits must be float32 or bfloat16")
        if draft_ids.dtype != torch.int32 or cu_num_draft_tokens.dtype != torch.int32:
            raise TypeError("draft_ids and cu_num_draft_tokens must be int32")
        B = cu_num_draft_tokens.numel() - 1
        for t, dt, name in ((top_k, torch.int32, "top_k"), (top_p, torch.float32, "top_p")):
            if t is not None and (t.device != self.device or t.dtype != dt or t.numel() != B
                                  or not t.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous {dt} tensor of B entries on the device")
        V = target_logits.shape[-1]
        if out is None:
            nd = int(cu_num_draft_tokens[-1]) if n_draft is None else int(n_draft)
            kw = dict(device=self.device)
            out = VerifyOutput(
                tokens=torch.empty(nd + B, dtype=torch.int32, **kw),
                num_accepted=torch.empty(B, dtype=torch.int32, **kw),
                beta=torch.empty(nd, dtype=torch.float32, **kw) if with_beta else None)
            if extended:
                out.target_prob = torch.empty(nd, dtype=torch.float32, **kw)
                out.draft_prob = torch.empty(nd, dtype=torch.float32, **kw)
                out.accept = torch.empty(nd, dtype=torch.int32, **kw)
        stream = _stream_handle(self.device)
        if top_k is not None or top_p is not None:
            rc = specdec_rejection_sample_topk_topp(
                self._h, _ptr(target_logits), dtype, _ptr(draft_probs), self._ids_ptr(draft_ids),
                _ptr(cu_num_draft_tokens), B, V, float(T), _ptr(top_k), _ptr(top_p), int(seed),
                int(request_offset), _ptr(out.tokens), _ptr(out.num_accepted), _ptr(out.beta),
                _ptr(out.target_prob), _ptr(out.draft_prob), _ptr(out.accept), stream)
        elif (out.target_prob is not None or out.draft_prob is not None or out.accept is not None
                or request_offset):
            rc = specdec_rejection_sample_ex(
                self._h, _ptr(target_logits), dtype, _ptr(draft_probs), self._ids_ptr(draft_ids),
                _ptr(cu_num_draft_tokens), B, V, float(T), int(seed), int(request_offset),
                _ptr(out.tokens),
                _ptr(out.num_accepted), _ptr(out.beta), _ptr(out.target_prob),
                _ptr(out.draft_prob), _ptr(out.accept), stream)
        else:
            rc = specdec_rejection_sample(
                self._h, _ptr(target_logits), dtype, _ptr(draft_probs), self._ids_ptr(draft_ids),
                _ptr(cu_num_draft_tokens), B, V, float(T), int(seed), _ptr(out.tokens),
                _ptr(out.num_accepted), _ptr(out.beta), stream)
        _check(rc, "specdec_rejection_sample")
        return out


@dataclass
class TreeOutput:
    tokens: torch.Tensor         # int32 [N] request b: slots cu[b] .. cu[b+1]-1
    num_accepted: torch.Tensor   # int32 [B]
    path: torch.Tensor | None    # int32 [N] accepted nodes (indices within the request), -1


def _tree_call(v: "Verifier", target_logits, draft_probs, node_tokens, node_parent, cu_num_nodes,
               T, seed, request_offset=0, with_path=True, out: TreeOutput | None = None):
    for t in (target_logits, node_tokens, node_parent, cu_num_nodes):
        if t.device != v.device or not t.is_contiguous():
            raise ValueError("inputs must be contiguous tensors on the verifier's device")
    if draft_probs is not None and (draft_probs.device != v.device
                                    or draft_probs.dtype != torch.float32
                                    or not draft_probs.is_contiguous()):
        raise ValueError("draft_probs must be a contiguous float32 tensor on the device")
    if target_logits.dtype == torch.float32:
        dtype = SPECDEC_F32
    elif target_logits.dtype == torch.bfloat16:
        dtype = SPECDEC_BF16
    else:
        raise TypeError("target_logits must be float32 or bfloat16")
    for t in (node_tokens, node_parent, cu_num_nodes):
        if t.dtype != torch.int32:
            raise TypeError("node_tokens, node_parent and cu_num_nodes must be int32")
    B = cu_num_nodes.numel() - 1
    N = node_tokens.numel()
    V = target_logits.shape[-1]
    if out is None:
        out = TreeOutput(tokens=torch.empty(N, dtype=torch.int32, device=v.device),
                         num_accepted=torch.empty(B, dtype=torch.int32, device=v.device),
                         path=torch.empty(N, dtype=torch.int32, device=v.device)
                         if with_path else None)
    rc = specdec_tree_verify(v.handle, _ptr(target_logits), dtype, _ptr(draft_probs),
                             _ptr(node_tokens), _ptr(node_parent), _ptr(cu_num_nodes), B, V,
                             float(T), int(seed), int(request_offset), _ptr(out.tokens),
                             _ptr(out.num_accepted), _ptr(out.path), _stream_handle(v.device))
    _check(rc, "specdec_tree_verify")
    return out


def uniform(seed: int, b: int, pos: int, stream_id: int, v0: int, n: int,
            device: int | torch.device = 0) -> torch.Tensor:
    """The generator's uniforms U(seed, b, pos, stream_id, v0 .. v0+n-1) (float32)."""
    dev = torch.device("cuda", device) if isinstance(device, int) else torch.device(device)
    out = torch.empty(n, dtype=torch.float32, device=dev)
    _check(specdec_uniform(seed, b, pos, stream_id, v0, n, out.data_ptr(), _stream_handle(dev)),
           "specdec_uniform")
    return out


def selection_mass(z: torch.Tensor, V: int) -> tuple[torch.Tensor, torch.Tensor]:
    """The top-p selection's integer masses (int64 holding the uint64 values,
    all below 2^63) and 2^-z (float32) for float32 distances z on the device."""
    if z.dtype != torch.float32 or not z.is_cuda:
        raise ValueError("z must be a float32 CUDA tensor")
    z = z.contiguous()
    mass = torch.empty(z.numel(), dtype=torch.int64, device=z.device)
    p2 = torch.empty(z.numel(), dtype=torch.float32, device=z.device)
    _check(specdec_selection_mass(z.data_ptr(), z.numel(), V, mass.data_ptr(), p2.data_ptr(),
                                  _stream_handle(z.device)), "specdec_selection_mass")
    return mass, p2


def neg_log_uniform(k0: int, n: int, device: int | torch.device = 0) -> torch.Tensor:
    dev = torch.device("cuda", device) if isinstance(device, int) else torch.device(device)
    out = torch.empty(n, dtype=torch.float32, device=dev)
    _check(specdec_neg_log_uniform(k0, n, out.data_ptr(), _stream_handle(dev)),
           "specdec_neg_log_uniform")
    return out
