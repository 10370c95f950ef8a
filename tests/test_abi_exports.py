"""The C-ABI library loads without a GPU and exports every function that
include/specdec.h declares (no compute calls here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_rejection_decode_gb300.build import build
    return ctypes.CDLL(build())


def declared():
    text = open(os.path.join(ROOT, "include", "specdec.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(specdec_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared()
    for required in ("specdec_create", "specdec_rejection_sample", "specdec_destroy",
                     "specdec_reserve", "specdec_get_error", "specdec_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared():
        assert hasattr(lib, name), name


def test_binding_names_match_header():
    from speculative_decoding_rejection_decode_gb300 import _lib
    assert sorted(_lib.EXPORTED) == declared()


def test_host_checks_without_gpu(lib):
    from speculative_decoding_rejection_decode_gb300 import (specdec_rejection_sample,
                                                             specdec_status_string)
    # a null handle is refused before anything touches the device
    assert specdec_rejection_sample(None, 1, 0, 1, 1, 1, 1, 8, 1.0, 0, 1, 1, None, None) == -1
    assert specdec_status_string(-5) == "draft id outside [0, V)"
    assert specdec_status_string(123) == "unknown status"


def test_host_checked_errors_return_before_any_device_work(lib):
    # every documented host check answers with its status code and touches no
    # device (the fake pointer values are never dereferenced on the host)
    import speculative_decoding_rejection_decode_gb300 as sd
    from speculative_decoding_rejection_decode_gb300 import _lib
    INVALID, DTYPE, CAPACITY = -1, -2, -6
    rc, h = _lib.specdec_create(-1)
    assert rc in (INVALID, -3) and h == 0          # bad device (or no CUDA driver at all)
    assert _lib.specdec_reserve(None, 10, 1) == INVALID
    assert _lib.specdec_set_path(None, 0) == INVALID
    assert _lib.specdec_set_timing_events(None, None, None) == INVALID
    assert _lib.specdec_set_adjust_counters(None, None) == INVALID
    assert _lib.specdec_set_fault_injection(None, 0, 0) == INVALID
    assert _lib.specdec_last_path(None)[0] == INVALID
    assert _lib.specdec_get_error(None, None)[0] == INVALID
    assert _lib.specdec_destroy(None) == INVALID
    assert _lib.specdec_rejection_sample_ex(None, 1, 0, 1, 1, 1, 1, 8, 1.0, 0, 0, 1, 1,
                                            None, None, None, None, None) == INVALID
    assert _lib.specdec_rejection_sample_topk_topp(None, 1, 0, 1, 1, 1, 1, 8, 1.0, None, None, 0,
                                                   0, 1, 1, None, None, None, None,
                                                   None) == INVALID
    assert _lib.specdec_tree_verify(None, 1, 0, 1, 1, 1, 1, 1, 8, 1.0, 0, 0, 1, 1, None,
                                    None) == INVALID
    # generator, log and mass diagnostics: bad sizes refused, empty requests are no-ops
    assert _lib.specdec_uniform(0, 0, 0, 0, 0, -1, None, None) == INVALID
    assert _lib.specdec_uniform(0, 0, 0, 0, 0, 0, None, None) == 0
    assert _lib.specdec_neg_log_uniform((1 << 23) - 1, 2, 1, None) == INVALID
    assert _lib.specdec_neg_log_uniform(0, 0, None, None) == 0
    assert _lib.specdec_selection_mass(None, -1, 10, None, None, None) == INVALID
    assert _lib.specdec_selection_mass(1, 4, 10, None, None, None) == INVALID
    assert _lib.specdec_selection_mass(None, 0, 0, None, None, None) == INVALID
    assert _lib.specdec_selection_mass(None, 0, 10, None, None, None) == 0
    # the allocation-free entry point checks dtype, sizes, T, pointers and its limits first
    args = dict(target_logits=1, dtype=sd.SPECDEC_F32, draft_probs=1, draft_ids=1,
                cu_num_draft_tokens=1, B=2, V=8, T=1.0, seed=0, n_draft_positions=4,
                out_tokens=1, out_num_accepted=1, out_beta=None, out_device_error=None,
                stream=None)

    def noalloc(**kw):
        a = dict(args)
        a.update(kw)
        return _lib.specdec_rejection_sample_noalloc(*a.values())

    assert noalloc(dtype=7) == DTYPE
    assert noalloc(B=0) == INVALID and noalloc(V=0) == INVALID
    assert noalloc(n_draft_positions=-1) == INVALID
    assert noalloc(T=-1.0) == INVALID and noalloc(T=float("nan")) == INVALID
    assert noalloc(target_logits=None) == INVALID and noalloc(out_tokens=None) == INVALID
    assert noalloc(B=_lib.SPECDEC_NOALLOC_MAX_BATCH + 1) == CAPACITY
    assert noalloc(n_draft_positions=_lib.SPECDEC_NOALLOC_MAX_ROWS) == CAPACITY
