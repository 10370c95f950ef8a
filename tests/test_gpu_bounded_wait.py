"""The bounded waits of the cluster path (failure handling without a GPU
fault): with the library's test hook, rank 0 of every 2-CTA cluster of the pair
kernel withholds the first work slot from rank 1, whose wait runs out after a
short limit; the call must return, the error word must carry the timeout bit,
and the next call (hook off) must be clean and at parity with the oracle."""
import pytest
import torch

from gpu_helpers import compare, flag_budget_ok, run_gpu, run_oracle
from speculative_decoding_rejection_decode_gb300.inputs import make_config

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def V():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_rejection_decode_gb300 import Verifier
    v = Verifier(0)
    yield v
    v.close()


def test_pair_kernel_wait_runs_out_and_the_next_call_is_clean(V):
    import time

    from speculative_decoding_rejection_decode_gb300 import SPECDEC_PATH_PAIR
    from speculative_decoding_rejection_decode_gb300._lib import (SPECDEC_DEVERR_TIMEOUT,
                                                                  SPECDEC_FAULT_NONE,
                                                                  SPECDEC_FAULT_PAIR_STALL,
                                                                  specdec_set_fault_injection)
    w = make_config(1)                      # 8 requests: the pair path
    V.set_path(SPECDEC_PATH_PAIR)
    assert specdec_set_fault_injection(V.handle, SPECDEC_FAULT_PAIR_STALL, 5_000_000) == 0
    t0 = time.perf_counter()
    run_gpu(V, w)                           # returns; outputs undefined
    elapsed = time.perf_counter() - t0
    assert V.last_path()[0] == SPECDEC_PATH_PAIR
    assert V.get_error() & SPECDEC_DEVERR_TIMEOUT
    assert elapsed < 30.0
    assert specdec_set_fault_injection(V.handle, SPECDEC_FAULT_NONE, 0) == 0
    for _ in range(2):
        g = run_gpu(V, w)
        assert V.get_error() == 0
        st = compare(w, g, run_oracle(w))
        assert flag_budget_ok(st), st
    V.set_path(0)


def test_fault_injection_argument_checks(V):
    from speculative_decoding_rejection_decode_gb300._lib import (SPECDEC_ERR_INVALID_ARG,
                                                                  SPECDEC_FAULT_NONE,
                                                                  SPECDEC_FAULT_PAIR_STALL,
                                                                  specdec_set_fault_injection)
    assert specdec_set_fault_injection(None, SPECDEC_FAULT_NONE, 0) == SPECDEC_ERR_INVALID_ARG
    assert specdec_set_fault_injection(V.handle, 7, 1000) == SPECDEC_ERR_INVALID_ARG
    assert specdec_set_fault_injection(V.handle, SPECDEC_FAULT_PAIR_STALL, 0) == SPECDEC_ERR_INVALID_ARG
    assert specdec_set_fault_injection(V.handle, SPECDEC_FAULT_PAIR_STALL,
                                       3_000_000_000) == SPECDEC_ERR_INVALID_ARG
    assert specdec_set_fault_injection(V.handle, SPECDEC_FAULT_NONE, 0) == 0
