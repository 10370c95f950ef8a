"""ctypes view of libspecdec.so: one Python function per C entry point, with
the same name and arguments (plain integers for pointers and streams).

Importing this module loads the in-tree library and raises if it is missing;
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspecdec.so")

SPECDEC_F32 = 0
SPECDEC_BF16 = 1

SPECDEC_OK = 0
SPECDEC_ERR_INVALID_ARG = -1
SPECDEC_ERR_UNSUPPORTED_DTYPE = -2
SPECDEC_ERR_CUDA = -3
SPECDEC_ERR_OOM = -4
SPECDEC_ERR_BAD_DRAFT_ID = -5
SPECDEC_ERR_CAPACITY = -6
SPECDEC_ERR_TIMEOUT = -7

SPECDEC_DEVERR_BAD_DRAFT_ID = 1
SPECDEC_DEVERR_BAD_CU = 2
SPECDEC_DEVERR_CAPACITY = 4
SPECDEC_DEVERR_TIMEOUT = 8
SPECDEC_DEVERR_BAD_TREE = 16

SPECDEC_FAULT_NONE = 0
SPECDEC_FAULT_PAIR_STALL = 1

SPECDEC_NOALLOC_MAX_ROWS = 16384
SPECDEC_NOALLOC_MAX_BATCH = 4096

SPECDEC_PATH_AUTO = 0
SPECDEC_PATH_FUSED = 1
SPECDEC_PATH_TWO_PASS = 2
SPECDEC_PATH_SWEEP = 3
SPECDEC_PATH_GREEDY = 4
SPECDEC_PATH_STREAM = 5
SPECDEC_PATH_PAIR = 6
SPECDEC_PATH_DUAL = 7

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it first (python -m "
        "speculative_decoding_rejection_decode_gb300.build or __graft_entry__.build())")

_lib = ctypes.CDLL(LIB_PATH)

_vp, _i32, _i64, _u32, _u64, _f32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                      ctypes.c_uint32, ctypes.c_uint64, ctypes.c_float)


def _fn(name, restype, *argtypes):
    f = getattr(_lib, name)
    f.restype = restype
    f.argtypes = list(argtypes)
    return f


_create = _fn("specdec_create", _i32, ctypes.POINTER(_vp), _i32)
_reserve = _fn("specdec_reserve", _i32, _vp, _i64, _i32)
_rs = _fn("specdec_rejection_sample", _i32, _vp, _vp, _i32, _vp, _vp, _vp, _i32, _i32, _f32, _u64,
          _vp, _vp, _vp, _vp)
_rs_ex = _fn("specdec_rejection_sample_ex", _i32, _vp, _vp, _i32, _vp, _vp, _vp, _i32, _i32, _f32,
             _u64, _u64, _vp, _vp, _vp, _vp, _vp, _vp, _vp)
_rs_adj = _fn("specdec_rejection_sample_topk_topp", _i32, _vp, _vp, _i32, _vp, _vp, _vp, _i32,
              _i32, _f32, _vp, _vp, _u64, _u64, _vp, _vp, _vp, _vp, _vp, _vp, _vp)
_get_error = _fn("specdec_get_error", _i32, _vp, ctypes.POINTER(_i32), _vp)
_set_path = _fn("specdec_set_path", _i32, _vp, _i32)
_set_events = _fn("specdec_set_timing_events", _i32, _vp, _vp, _vp)
_last_path = _fn("specdec_last_path", _i32, _vp, ctypes.POINTER(_i32), ctypes.POINTER(_i32))
_set_adj_ctr = _fn("specdec_set_adjust_counters", _i32, _vp, _vp)
_set_fault = _fn("specdec_set_fault_injection", _i32, _vp, _i32, _u64)
_uniform = _fn("specdec_uniform", _i32, _u64, _u64, _u64, _u32, _u64, _i64, _vp, _vp)
_neg_log = _fn("specdec_neg_log_uniform", _i32, _u32, _i64, _vp, _vp)
_sel_mass = _fn("specdec_selection_mass", _i32, _vp, _i64, _i32, _vp, _vp, _vp)
_rs_noalloc = _fn("specdec_rejection_sample_noalloc", _i32, _vp, _i32, _vp, _vp, _vp, _i32, _i32,
                  _f32, _u64, _i64, _vp, _vp, _vp, _vp, _vp)
_tree = _fn("specdec_tree_verify", _i32, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _i32, _i32, _f32,
            _u64, _u64, _vp, _vp, _vp, _vp)
_status_string = _fn("specdec_status_string", ctypes.c_char_p, _i32)
_destroy = _fn("specdec_destroy", _i32, _vp)


def specdec_create(device: int) -> tuple[int, int]:
    h = _vp()
    rc = _create(ctypes.byref(h), device)
    return rc, (h.value or 0)


def specdec_reserve(h: int, max_draft_positions: int, max_batch: int) -> int:
    return _reserve(h, max_draft_positions, max_batch)


def specdec_rejection_sample(h, target_logits, dtype, draft_probs, draft_ids, cu_num_draft_tokens,
                             B, V, T, seed, out_tokens, out_num_accepted, out_beta, stream) -> int:
    return _rs(h, target_logits, dtype, draft_probs, draft_ids, cu_num_draft_tokens, B, V, T,
               seed & 0xFFFFFFFFFFFFFFFF, out_tokens, out_num_accepted, out_beta, stream)


def specdec_rejection_sample_ex(h, target_logits, dtype, draft_probs, draft_ids,
                                cu_num_draft_tokens, B, V, T, seed, request_offset, out_tokens,
                                out_num_accepted, out_beta, out_target_prob, out_draft_prob,
                                out_accept, stream) -> int:
    return _rs_ex(h, target_logits, dtype, draft_probs, draft_ids, cu_num_draft_tokens, B, V, T,
                  seed & 0xFFFFFFFFFFFFFFFF, request_offset, out_tokens, out_num_accepted,
                  out_beta, out_target_prob, out_draft_prob, out_accept, stream)


def specdec_rejection_sample_topk_topp(h, target_logits, dtype, draft_probs, draft_ids,
                                       cu_num_draft_tokens, B, V, T, top_k, top_p, seed,
                                       request_offset, out_tokens, out_num_accepted, out_beta,
                                       out_target_prob, out_draft_prob, out_accept, stream) -> int:
    return _rs_adj(h, target_logits, dtype, draft_probs, draft_ids, cu_num_draft_tokens, B, V, T,
                   top_k, top_p, seed & 0xFFFFFFFFFFFFFFFF, request_offset, out_tokens,
                   out_num_accepted, out_beta, out_target_prob, out_draft_prob, out_accept, stream)


def specdec_set_timing_events(h: int, before_rows, after_rows) -> int:
    return _set_events(h, before_rows, after_rows)


def specdec_set_adjust_counters(h: int, device_counters) -> int:
    return _set_adj_ctr(h, device_counters)


def specdec_set_fault_injection(h: int, mode: int, wait_limit_ns: int) -> int:
    return _set_fault(h, mode, wait_limit_ns)


def specdec_get_error(h: int, stream) -> tuple[int, int]:
    e = _i32(0)
    rc = _get_error(h, ctypes.byref(e), stream)
    return rc, e.value


def specdec_set_path(h: int, path: int) -> int:
    return _set_path(h, path)


def specdec_last_path(h: int) -> tuple[int, int, int]:
    p, c = _i32(0), _i32(0)
    rc = _last_path(h, ctypes.byref(p), ctypes.byref(c))
    return rc, p.value, c.value


def specdec_uniform(seed, b, pos, stream_id, v0, n, out, stream) -> int:
    return _uniform(seed & 0xFFFFFFFFFFFFFFFF, b, pos, stream_id, v0, n, out, stream)


def specdec_neg_log_uniform(k0, n, out, stream) -> int:
    return _neg_log(k0, n, out, stream)


def specdec_selection_mass(z, n, V, out_mass, out_pow2, stream) -> int:
    return _sel_mass(z, n, V, out_mass, out_pow2, stream)


def specdec_rejection_sample_noalloc(target_logits, dtype, draft_probs, draft_ids,
                                     cu_num_draft_tokens, B, V, T, seed, n_draft_positions,
                                     out_tokens, out_num_accepted, out_beta, out_device_error,
                                     stream) -> int:
    return _rs_noalloc(target_logits, dtype, draft_probs, draft_ids, cu_num_draft_tokens, B, V, T,
                       seed & 0xFFFFFFFFFFFFFFFF, n_draft_positions, out_tokens, out_num_accepted,
                       out_beta, out_device_error, stream)


def specdec_tree_verify(h, target_logits, dtype, draft_probs, node_tokens, node_parent,
                        cu_num_nodes, B, V, T, seed, request_offset, out_tokens, out_num_accepted,
                        out_path, stream) -> int:
    return _tree(h, target_logits, dtype, draft_probs, node_tokens, node_parent, cu_num_nodes, B,
                 V, T, seed & 0xFFFFFFFFFFFFFFFF, request_offset, out_tokens, out_num_accepted,
                 out_path, stream)


def specdec_status_string(status: int) -> str:
    return _status_string(status).decode()


def specdec_destroy(h: int) -> int:
    return _destroy(h)


EXPORTED = ["specdec_create", "specdec_reserve", "specdec_rejection_sample",
            "specdec_rejection_sample_ex", "specdec_rejection_sample_topk_topp",
            "specdec_get_error", "specdec_set_path",
            "specdec_set_timing_events", "specdec_set_adjust_counters",
            "specdec_set_fault_injection",
            "specdec_last_path", "specdec_uniform", "specdec_neg_log_uniform",
            "specdec_selection_mass", "specdec_rejection_sample_noalloc", "specdec_tree_verify",
            "specdec_status_string", "specdec_destroy"]
