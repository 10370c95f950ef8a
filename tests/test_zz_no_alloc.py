"""The allocation-free entry point against the handle-based one, through the
C ABI.

specdec_rejection_sample_noalloc serves callers that cannot allocate device
memory when they verify: code running inside a memory pool or arena it does not
own, plug-ins that are handed only pre-allocated buffers, hosts that freeze
device allocation after start-up.  Its scratch is a fixed device array shared
by every call, so each check runs two calls in a row: the second must not see
anything the first left behind.  Results must equal those of
specdec_rejection_sample (same kernels) within the tolerance the other parity
tests use (tokens and counts identical, beta within 1e-5), and, once, those of
the CPU oracle."""
import dataclasses

import numpy as np
import pytest
import torch

from speculative_decoding_rejection_decode_gb300.inputs import make_config

pytestmark = pytest.mark.gpu

BETA_TOL = 1e-5


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_rejection_decode_gb300 as sd
    return sd


def _handle_path(sd, w):
    """The handle-based entry point on the path the allocation-free one runs."""
    v = sd.Verifier(0)
    if w.T > 0:
        v.set_path(sd.SPECDEC_PATH_SWEEP)
    wd = w.to("cuda")
    out = v(wd.target_logits, wd.draft_probs, wd.draft_ids, wd.cu, w.T, w.seed, n_draft=w.n_draft)
    torch.cuda.synchronize()
    assert v.get_error() == 0
    res = (out.tokens.cpu().numpy(), out.num_accepted.cpu().numpy(), out.beta.cpu().numpy())
    v.close()
    return res


def _noalloc(sd, w, err, n_draft=None):
    wd = w.to("cuda")
    out_t = torch.full((w.n_target,), -7, dtype=torch.int32, device="cuda")
    out_n = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    out_b = torch.full((w.n_draft,), -7.0, dtype=torch.float32, device="cuda")
    dtype = sd.SPECDEC_BF16 if w.dtype == "bf16" else sd.SPECDEC_F32
    rc = sd.specdec_rejection_sample_noalloc(
        wd.target_logits.data_ptr(), dtype,
        None if wd.draft_probs is None else wd.draft_probs.data_ptr(),
        wd.draft_ids.data_ptr(), wd.cu.data_ptr(), w.B, w.V, w.T, w.seed,
        w.n_draft if n_draft is None else n_draft,
        out_t.data_ptr(), out_n.data_ptr(), out_b.data_ptr(), err.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == 0, sd.specdec_status_string(rc)
    torch.cuda.synchronize()
    return out_t.cpu().numpy(), out_n.cpu().numpy(), out_b.cpu().numpy()


def _same(a, b):
    assert np.array_equal(a[0], b[0])
    assert np.array_equal(a[1], b[1])
    assert np.abs(a[2] - b[2]).max(initial=0.0) <= BETA_TOL


@pytest.mark.parametrize("idx,kw", [(3, dict(B=60, V=20000)), (4, dict(B=40)), (2, dict(B=48)),
                                    (1, {})])
def test_noalloc_matches_handle_entry_point_twice(lib, idx, kw):
    w = make_config(idx, device="cuda", **kw)
    ref = _handle_path(lib, w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        _same(_noalloc(lib, w, err), ref)
    assert int(err.item()) == 0


def test_noalloc_back_to_back_different_batches(lib):
    # a large call, then a smaller one with other inputs: no state carries over
    big = make_config(4, device="cuda", B=300)
    small = make_config(3, device="cuda", B=30, V=12000)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _same(_noalloc(lib, big, err), _handle_path(lib, big))
    _same(_noalloc(lib, small, err), _handle_path(lib, small))
    _same(_noalloc(lib, big, err), _handle_path(lib, big))
    assert int(err.item()) == 0


def test_noalloc_rejects_sizes_beyond_the_limit(lib):
    w = make_config(1, device="cuda")
    wd = w.to("cuda")
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for B, nd in ((lib._lib.SPECDEC_NOALLOC_MAX_BATCH + 1, 0),
                  (8, lib._lib.SPECDEC_NOALLOC_MAX_ROWS)):
        rc = lib.specdec_rejection_sample_noalloc(
            wd.target_logits.data_ptr(), lib.SPECDEC_F32, wd.draft_probs.data_ptr(),
            wd.draft_ids.data_ptr(), wd.cu.data_ptr(), B, w.V, 1.0, 0, nd, dummy.data_ptr(),
            dummy.data_ptr(), None, None, stream)
        assert rc == lib._lib.SPECDEC_ERR_CAPACITY


def test_noalloc_matches_the_oracle(lib):
    # the ragged workload at B = 60 against the CPU oracle, element by element
    from gpu_helpers import compare, flag_budget_ok, run_oracle
    w = make_config(3, device="cuda", B=60)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        tok, nacc, beta = _noalloc(lib, w, err)
        st = compare(w, dict(tokens=tok, num_accepted=nacc, beta=beta), run_oracle(w))
        assert flag_budget_ok(st), st
    assert int(err.item()) == 0


def test_noalloc_one_hot_drafts(lib):
    # draft ids without draft rows at T > 0 (a one-hot drafter): the sweep
    # kernel never reads a draft row
    w = dataclasses.replace(make_config(2, device="cuda", B=48), T=1.0, seed=2)
    assert w.draft_probs is None
    ref = _handle_path(lib, w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        _same(_noalloc(lib, w, err), ref)
    assert int(err.item()) == 0


def test_noalloc_understated_positions_set_the_capacity_bit(lib):
    # n_draft_positions below the real cu[B] passes the host check, but the
    # real rows (16800) pass the limit: the kernels skip the rows past it and
    # report SPECDEC_DEVERR_CAPACITY; a following well-formed call is clean
    from speculative_decoding_rejection_decode_gb300._lib import SPECDEC_DEVERR_CAPACITY
    from speculative_decoding_rejection_decode_gb300.inputs import make_workload
    big = make_workload(name="over the row limit", B=2100, gamma=7, V=64, dtype="f32", T=1.0,
                        seed=5, device="cuda")
    assert big.n_target > lib._lib.SPECDEC_NOALLOC_MAX_ROWS
    for T in (1.0, 0.0):
        w = dataclasses.replace(big, T=T)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        _noalloc(lib, w, err, n_draft=1000)
        assert int(err.item()) & SPECDEC_DEVERR_CAPACITY, T
    w = make_config(1, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _same(_noalloc(lib, w, err), _handle_path(lib, w))
    assert int(err.item()) == 0
