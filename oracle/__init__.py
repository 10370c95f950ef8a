"""CPU oracle of the speculative-sampling verifier (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The product path never does: the CUDA
library fails loudly when its extension is missing instead of falling back
here.

The arithmetic lives in ``specdec_oracle.c`` (double precision, one thread,
one request at a time, following Algorithm 1 and Section 2.3 of Leviathan et
al. as restated on the bloss0m and vllbc reading-notes pages, and the
verification pseudo-code of the timinsight implementation guide).  This module
compiles it with gcc on first use and marshals numpy arrays through ctypes; it
adds no arithmetic of its own.

Parity pins live in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "specdec_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libspecdec_oracle.so")

OK = 0
INVALID_ARG = -1
UNSUPPORTED_DTYPE = -2
OOM = -4
BAD_DRAFT_ID = -5

DTYPE_F32 = 0
DTYPE_BF16 = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compiles the oracle into ``oracle/_build`` (IEEE semantics: no fast-math,
    no contraction into fused multiply-adds, so x86 and Arm agree)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u64, i64, i32, dbl, vp = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int, ctypes.c_double,
                                  ctypes.c_void_p)
        lib.oracle_splitmix64.argtypes = [u64]
        lib.oracle_splitmix64.restype = u64
        lib.oracle_stream_key.argtypes = [u64, u64, u64, u64]
        lib.oracle_stream_key.restype = u64
        lib.oracle_uniform.argtypes = [u64, u64, u64, u64, u64]
        lib.oracle_uniform.restype = dbl
        lib.oracle_uniform_fill.argtypes = [u64, u64, u64, u64, u64, i64, vp]
        lib.oracle_uniform_fill.restype = None
        lib.oracle_verify_request.argtypes = [i64, i32, vp, i32, vp, vp, i32, dbl, u64,
                                              vp, vp, vp, vp, vp, vp, vp, vp]
        lib.oracle_verify_request.restype = i32
        lib.oracle_rejection_sample.argtypes = [vp, i32, vp, vp, vp, i32, i32, dbl, u64,
                                                vp, vp, vp, vp, vp, vp, vp, vp]
        lib.oracle_rejection_sample.restype = i32
        lib.oracle_verify_request_adj.argtypes = [i64, i32, vp, i32, vp, vp, i32, dbl, i32, dbl,
                                                  vp, u64, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                  vp]
        lib.oracle_verify_request_adj.restype = i32
        lib.oracle_rejection_sample_adj.argtypes = [vp, i32, vp, vp, vp, i32, i32, dbl, vp, vp,
                                                    u64, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.oracle_rejection_sample_adj.restype = i32
        lib.oracle_adjusted_probs.argtypes = [vp, i32, i32, dbl, i32, dbl, i32, vp, vp, vp]
        lib.oracle_adjusted_probs.restype = i32
        lib.oracle_tree_verify_request.argtypes = [i64, i32, vp, i32, vp, vp, vp, i32, dbl, u64,
                                                   vp, vp, vp, vp]
        lib.oracle_tree_verify_request.restype = i32
        lib.oracle_tree_verify.argtypes = [vp, i32, vp, vp, vp, vp, i32, i32, dbl, u64, vp, vp,
                                           vp, vp]
        lib.oracle_tree_verify.restype = i32
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def splitmix64(z: int) -> int:
    """SplitMix64 output for state increment + finaliser applied to ``z``."""
    return int(_load().oracle_splitmix64(ctypes.c_uint64(z & 0xFFFFFFFFFFFFFFFF)))


def stream_key(seed: int, b: int, pos: int, stream: int) -> int:
    return int(_load().oracle_stream_key(seed, b, pos, stream))


def uniform(seed: int, b: int, pos: int, stream: int, v0: int = 0, n: int = 1) -> np.ndarray:
    """U(seed, b, pos, stream, v) for v = v0 .. v0+n-1 as float64 (each value is
    an exact float32 as well)."""
    out = np.empty(n, dtype=np.float64)
    _load().oracle_uniform_fill(seed, b, pos, stream, v0, n, _ptr(out))
    return out


def _logits_array(target_logits: np.ndarray, dtype: str | None):
    a = np.ascontiguousarray(target_logits)
    if dtype is None:
        dtype = "bf16" if a.dtype == np.uint16 else "f32"
    if dtype == "f32":
        if a.dtype != np.float32:
            raise TypeError("f32 target logits must be a float32 array")
        return a, DTYPE_F32
    if dtype == "bf16":
        if a.dtype != np.uint16:
            raise TypeError("bf16 target logits must be passed as their uint16 bit patterns")
        return a, DTYPE_BF16
    raise ValueError(f"unknown dtype {dtype!r}")


@dataclass
class OracleResult:
    tokens: np.ndarray          # int32 [N_t]; request b uses slots cu[b]+b .. cu[b+1]+b
    num_accepted: np.ndarray    # int32 [B]
    beta: np.ndarray            # float64 [N_d]
    p_x: np.ndarray             # float64 [N_d]  p_i(x_i)
    q_x: np.ndarray             # float64 [N_d]  q_i(x_i)
    accept: np.ndarray          # int32 [N_d]    accept test at every position
    pos_near_tie: np.ndarray    # int32 [N_d]
    near_tie: np.ndarray        # int32 [B]
    status: int
    edge_lo: np.ndarray | None = None   # int32 [N_t]  reachable top-p cut shifts of each
    edge_hi: np.ndarray | None = None   # int32 [N_t]  target row (0 / 0 without a band)


def _per_request(a, B: int, dtype, name: str):
    if a is None:
        return None
    arr = np.ascontiguousarray(np.broadcast_to(np.asarray(a, dtype=dtype), (B,)))
    if arr.shape != (B,):
        raise ValueError(f"{name} needs one value per request")
    return arr


def rejection_sample(target_logits: np.ndarray, draft_probs: np.ndarray | None,
                     draft_ids: np.ndarray, cu_num_draft_tokens: np.ndarray, T: float, seed: int,
                     dtype: str | None = None, top_k=None, top_p=None) -> OracleResult:
    """Whole batch in the flattened ragged layout (see ``specdec_oracle.c``).
    ``top_k`` / ``top_p``: None, a scalar or one value per request."""
    lib = _load()
    logits, dt = _logits_array(target_logits, dtype)
    cu = np.ascontiguousarray(cu_num_draft_tokens, dtype=np.int32)
    ids = np.ascontiguousarray(draft_ids, dtype=np.int32)
    B = cu.shape[0] - 1
    V = logits.shape[-1]
    n_d = int(cu[-1])
    n_t = n_d + B
    if logits.reshape(-1, V).shape[0] != n_t:
        raise ValueError(f"target logits hold {logits.reshape(-1, V).shape[0]} rows, expected {n_t}")
    q = None
    if draft_probs is not None:
        q = np.ascontiguousarray(draft_probs, dtype=np.float32)
        if q.reshape(-1, V).shape[0] != n_d:
            raise ValueError("draft probs row count does not match cu[B]")
    tk = _per_request(top_k, B, np.int32, "top_k")
    tp = _per_request(top_p, B, np.float64, "top_p")
    tokens = np.empty(n_t, np.int32)
    nacc = np.empty(B, np.int32)
    beta = np.empty(max(n_d, 1), np.float64)
    p_x = np.empty(max(n_d, 1), np.float64)
    q_x = np.empty(max(n_d, 1), np.float64)
    acc = np.empty(max(n_d, 1), np.int32)
    pos_tie = np.empty(max(n_d, 1), np.int32)
    tie = np.empty(B, np.int32)
    elo = np.zeros(n_t, np.int32)
    ehi = np.zeros(n_t, np.int32)
    st = lib.oracle_rejection_sample_adj(_ptr(logits), dt, _ptr(q), _ptr(ids), _ptr(cu), B, V,
                                         float(T), _ptr(tk), _ptr(tp), seed & 0xFFFFFFFFFFFFFFFF,
                                         _ptr(tokens), _ptr(nacc), _ptr(beta), _ptr(p_x), _ptr(q_x),
                                         _ptr(acc), _ptr(pos_tie), _ptr(tie), _ptr(elo), _ptr(ehi))
    return OracleResult(tokens, nacc, beta[:n_d], p_x[:n_d], q_x[:n_d], acc[:n_d], pos_tie[:n_d],
                        tie, int(st), elo, ehi)


def verify_request(b: int, target_rows: np.ndarray, draft_rows: np.ndarray | None,
                   draft_ids: np.ndarray, T: float, seed: int,
                   dtype: str | None = None, top_k: int = 0, top_p: float = 1.0,
                   edge_shift=None) -> OracleResult:
    """One request with global request index ``b`` (the generator key), its
    gamma+1 target rows and gamma draft rows.  ``edge_shift`` (gamma+1 ints or
    None) moves each row's top-p cut by that many groups within the row's
    reachable range (``edge_lo`` / ``edge_hi`` of the result); a shift outside
    it gives status INVALID_ARG."""
    lib = _load()
    logits, dt = _logits_array(target_rows, dtype)
    V = logits.shape[-1]
    gamma = logits.reshape(-1, V).shape[0] - 1
    ids = np.ascontiguousarray(draft_ids, dtype=np.int32)
    if ids.shape[0] != gamma:
        raise ValueError("need gamma draft ids for gamma+1 target rows")
    q = None if draft_rows is None else np.ascontiguousarray(draft_rows, dtype=np.float32)
    shift = None
    if edge_shift is not None:
        shift = np.ascontiguousarray(edge_shift, dtype=np.int32)
        if shift.shape != (gamma + 1,):
            raise ValueError("edge_shift needs one value per target row")
    g1 = max(gamma, 1)
    tokens = np.empty(gamma + 1, np.int32)
    nacc = np.empty(1, np.int32)
    beta, p_x, q_x = (np.empty(g1, np.float64) for _ in range(3))
    acc, pos_tie = np.empty(g1, np.int32), np.empty(g1, np.int32)
    tie = np.empty(1, np.int32)
    elo = np.zeros(gamma + 1, np.int32)
    ehi = np.zeros(gamma + 1, np.int32)
    st = lib.oracle_verify_request_adj(b, gamma, _ptr(logits), dt, _ptr(q), _ptr(ids), V, float(T),
                                       int(top_k), float(top_p), _ptr(shift),
                                       seed & 0xFFFFFFFFFFFFFFFF, _ptr(tokens), _ptr(nacc),
                                       _ptr(beta), _ptr(p_x), _ptr(q_x), _ptr(acc), _ptr(pos_tie),
                                       _ptr(tie), _ptr(elo), _ptr(ehi))
    return OracleResult(tokens, nacc, beta[:gamma], p_x[:gamma], q_x[:gamma], acc[:gamma],
                        pos_tie[:gamma], tie, int(st), elo, ehi)


def adjusted_probs(row: np.ndarray, T: float, top_k: int = 0, top_p: float = 1.0,
                   dtype: str | None = None, shift: int = 0, with_range: bool = False):
    """The adjusted target distribution of one row of logits (temperature,
    then top-k, then top-p), with the top-p cut moved by ``shift`` groups.
    With ``with_range`` also the reachable range (lo, hi) of shifts."""
    lib = _load()
    logits, dt = _logits_array(np.asarray(row).reshape(-1), dtype)
    p = np.empty(logits.shape[0], np.float64)
    lo = np.zeros(1, np.int32)
    hi = np.zeros(1, np.int32)
    st = lib.oracle_adjusted_probs(_ptr(logits), dt, logits.shape[0], float(T), int(top_k),
                                   float(top_p), int(shift), _ptr(p), _ptr(lo), _ptr(hi))
    if st < 0:
        raise ValueError(f"oracle_adjusted_probs failed with status {st}")
    return (p, (int(lo[0]), int(hi[0]))) if with_range else p


@dataclass
class TreeResult:
    tokens: np.ndarray          # int32 [N_nodes]; request b uses slots cu[b] .. cu[b+1]-1
    num_accepted: np.ndarray    # int32 [B]
    path: np.ndarray            # int32 [N_nodes]  accepted node indices (within the request), -1
    near_tie: np.ndarray        # int32 [B]
    status: int


def tree_verify(target_logits: np.ndarray, draft_probs: np.ndarray | None, node_tokens,
                node_parent, cu_num_nodes, T: float, seed: int,
                dtype: str | None = None) -> TreeResult:
    """A batch of token trees in the flattened layout (see ``specdec_oracle.c``,
    oracle_tree_verify): request b owns nodes cu[b] .. cu[b+1]-1, node 0 of a
    request being its context; parents are indices within the request."""
    lib = _load()
    logits, dt = _logits_array(target_logits, dtype)
    cu = np.ascontiguousarray(cu_num_nodes, dtype=np.int32)
    tok = np.ascontiguousarray(node_tokens, dtype=np.int32)
    par = np.ascontiguousarray(node_parent, dtype=np.int32)
    B = cu.shape[0] - 1
    V = logits.shape[-1]
    n = int(cu[-1])
    if logits.reshape(-1, V).shape[0] != n or tok.shape[0] != n or par.shape[0] != n:
        raise ValueError("one target row, token and parent per node")
    q = None
    if draft_probs is not None:
        q = np.ascontiguousarray(draft_probs, dtype=np.float32)
        if q.reshape(-1, V).shape[0] != n:
            raise ValueError("one draft row per node")
    tokens = np.empty(n, np.int32)
    nacc = np.empty(B, np.int32)
    path = np.empty(n, np.int32)
    tie = np.empty(B, np.int32)
    st = lib.oracle_tree_verify(_ptr(logits), dt, _ptr(q), _ptr(tok), _ptr(par), _ptr(cu), B, V,
                                float(T), seed & 0xFFFFFFFFFFFFFFFF, _ptr(tokens), _ptr(nacc),
                                _ptr(path), _ptr(tie))
    return TreeResult(tokens, nacc, path, tie, int(st))


def tree_verify_request(b: int, target_rows: np.ndarray, draft_rows: np.ndarray | None,
                        node_tokens, node_parent, T: float, seed: int,
                        dtype: str | None = None) -> TreeResult:
    """One token tree with global request index ``b`` (the generator key)."""
    lib = _load()
    logits, dt = _logits_array(target_rows, dtype)
    V = logits.shape[-1]
    n = logits.reshape(-1, V).shape[0]
    tok = np.ascontiguousarray(node_tokens, dtype=np.int32)
    par = np.ascontiguousarray(node_parent, dtype=np.int32)
    q = None if draft_rows is None else np.ascontiguousarray(draft_rows, dtype=np.float32)
    tokens = np.empty(n, np.int32)
    nacc = np.empty(1, np.int32)
    path = np.empty(n, np.int32)
    tie = np.empty(1, np.int32)
    st = lib.oracle_tree_verify_request(b, n, _ptr(logits), dt, _ptr(q), _ptr(tok), _ptr(par), V,
                                        float(T), seed & 0xFFFFFFFFFFFFFFFF, _ptr(tokens),
                                        _ptr(nacc), _ptr(path), _ptr(tie))
    return TreeResult(tokens, nacc, path, tie, int(st))
