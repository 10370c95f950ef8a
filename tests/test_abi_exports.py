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
