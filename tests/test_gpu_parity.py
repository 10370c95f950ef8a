"""CUDA library vs the CPU oracle, through the C ABI, on seeded synthetic
workloads (the five standard configurations plus edge cases)."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import stat_checks as sc
from gpu_helpers import (compare, flag_budget_ok, numpy_runner, run_gpu, run_oracle,
                         run_oracle_threaded)
from speculative_decoding_rejection_decode_gb300.inputs import (from_rows, make_config,
                                                                make_workload)

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rng_vectors.txt")


@pytest.fixture(scope="module")
def V():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_rejection_decode_gb300 import Verifier
    v = Verifier(0)
    yield v
    v.close()


def _paths():
    from speculative_decoding_rejection_decode_gb300 import (SPECDEC_PATH_DUAL, SPECDEC_PATH_FUSED,
                                                             SPECDEC_PATH_PAIR, SPECDEC_PATH_STREAM,
                                                             SPECDEC_PATH_SWEEP,
                                                             SPECDEC_PATH_TWO_PASS)
    return {"fused": SPECDEC_PATH_FUSED, "sweep": SPECDEC_PATH_SWEEP, "stream": SPECDEC_PATH_STREAM,
            "pair": SPECDEC_PATH_PAIR, "dual": SPECDEC_PATH_DUAL, "two_pass": SPECDEC_PATH_TWO_PASS}


ALL_PATHS = ["dual", "pair", "stream", "fused", "sweep", "two_pass"]


# --------------------------------------------------------------------------
# generator
# --------------------------------------------------------------------------

def test_rng_vectors_bit_exact(V):
    from speculative_decoding_rejection_decode_gb300 import uniform
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        seed, b, pos, stream, v, _h, u = line.split()
        seed, b, pos, stream, v = (int(x, 0) for x in (seed, b, pos, stream, v))
        got = uniform(seed, b, pos, stream, v, 1).cpu().item()
        assert got == float.fromhex(u)


def test_rng_bulk_matches_oracle(V):
    from speculative_decoding_rejection_decode_gb300 import uniform
    for (seed, b, pos, stream) in ((4, 1023, 7, 1), (0, 0, 0, 0), (99, 5, 2, 1)):
        g = uniform(seed, b, pos, stream, 1000, 1 << 18).cpu().numpy().astype(np.float64)
        o = oracle.uniform(seed, b, pos, stream, 1000, 1 << 18)
        assert np.array_equal(g, o)


def test_neg_log_uniform_accuracy(V):
    from speculative_decoding_rejection_decode_gb300 import neg_log_uniform
    n = 1 << 23
    e = neg_log_uniform(0, n).cpu().numpy().astype(np.float64)
    k = np.arange(n, dtype=np.float64)
    ref = -np.log((k + 0.5) / 2 ** 23)
    rel = np.abs(e - ref) / ref
    assert rel.max() < 2e-6, rel.max()


# --------------------------------------------------------------------------
# the five standard workloads
# --------------------------------------------------------------------------

def test_config0_tiny(V):
    w = make_config(0)
    for path in _paths().values():
        V.set_path(path)
        g = run_gpu(V, w)
        assert V.get_error() == 0
        st = compare(w, g, run_oracle(w))
        assert st["flagged"] == 0
    V.set_path(0)


@pytest.mark.parametrize("path", ALL_PATHS)
def test_config1(V, path):
    w = make_config(1)
    V.set_path(_paths()[path])
    g = run_gpu(V, w)
    assert V.get_error() == 0
    assert V.last_path()[0] == _paths()[path]
    st = compare(w, g, run_oracle(w))
    assert flag_budget_ok(st), st
    V.set_path(0)


def test_config2_greedy_bit_exact(V):
    w = make_config(2)
    g = run_gpu(V, w)
    assert V.get_error() == 0
    r = run_oracle(w)
    compare(w, g, r, exact=True)
    # alpha ~ 0.75 by construction
    acc = r.accept.mean()
    assert 0.7 < acc < 0.8


@pytest.mark.parametrize("path", ALL_PATHS)
def test_config3_ragged(V, path):
    w = make_config(3, device="cuda")
    V.set_path(_paths()[path])
    g = run_gpu(V, w)
    assert V.get_error() == 0
    p, c = V.last_path()
    assert p == _paths()[path]
    if path == "fused":
        assert c == 4
    st = compare(w, g, run_oracle(w))
    assert flag_budget_ok(st), st
    V.set_path(0)


def test_config4_full_size(V):
    # the large workload at full size, in the launch configuration the benchmark
    # times, against the oracle on every request (threads over request ranges)
    w = make_config(4, device="cuda")
    g = run_gpu(V, w)
    assert V.get_error() == 0
    assert V.last_path()[0] == _paths()["sweep"]
    cu = w.cu.cpu().numpy()
    sc.check_e_layout(g["tokens"], g["num_accepted"], w.draft_ids.cpu().numpy(), cu, w.V)
    r = run_oracle_threaded(w)
    assert r.status == 0
    st = compare(w, g, r)
    assert st["requests"] == w.B and st["rows"] == w.n_target
    assert flag_budget_ok(st), st


@pytest.mark.parametrize("path", ALL_PATHS)
def test_config4_reduced_full_parity(V, path):
    w = make_config(4, device="cuda", B=24)
    V.set_path(_paths()[path])
    g = run_gpu(V, w)
    assert V.get_error() == 0
    st = compare(w, g, run_oracle(w))
    assert flag_budget_ok(st), st
    V.set_path(0)


def test_deterministic_across_calls(V):
    w = make_config(3, device="cuda", B=40, V=20000)
    a = run_gpu(V, w)
    b = run_gpu(V, w)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


# --------------------------------------------------------------------------
# edge cases
# --------------------------------------------------------------------------

@pytest.mark.parametrize("path", ALL_PATHS)
@pytest.mark.parametrize("Vsz,dtype", [(8, "f32"), (8, "bf16"), (100, "f32"), (4100, "bf16"),
                                       (4099, "f32"), (4097, "bf16"), (12345, "f32"),
                                       (65536, "bf16"), (40000, "f32")])
def test_vocab_sizes_and_tails(V, Vsz, dtype, path):
    # sizes that span several 4096-element chunks with a ragged tail, odd sizes
    # (no vector loads / bulk copies), and sizes below one chunk
    w = make_workload(name="tails", B=7, gamma=(0, 6), V=Vsz, dtype=dtype, T=0.9, seed=17,
                      target_std=2.0, noise_std=0.8, device="cuda")
    V.set_path(_paths()[path])
    g = run_gpu(V, w)
    assert V.get_error() == 0
    st = compare(w, g, run_oracle(w))
    assert flag_budget_ok(st), st
    V.set_path(0)


@pytest.mark.parametrize("T", [0.05, 0.3, 2.5, 10.0])
def test_temperatures(V, T):
    w = make_workload(name="temps", B=16, gamma=5, V=3000, dtype="bf16", T=T, seed=23,
                      target_std=3.0, noise_std=1.0, draft_T=T, device="cuda")
    g = run_gpu(V, w)
    st = compare(w, g, run_oracle(w))
    assert flag_budget_ok(st), st


def test_gamma_zero_and_empty_requests(V):
    w = make_workload(name="zeros", B=9, gamma=(0, 2), V=5000, dtype="f32", T=1.0, seed=31,
                      device="cuda")
    assert (np.diff(w.cu.cpu().numpy()) == 0).any()
    for path in _paths().values():
        V.set_path(path)
        g = run_gpu(V, w)
        st = compare(w, g, run_oracle(w))
        assert flag_budget_ok(st), st
    V.set_path(0)


def test_single_request_bonus_only(V):
    # draft_probs / draft_ids must be real pointers at T > 0 even when cu[B] == 0
    from speculative_decoding_rejection_decode_gb300 import VerifyOutput
    t = torch.randn(1, 4096) * 2
    w = from_rows(t, torch.zeros(1, 4096), torch.zeros(0, dtype=torch.int32), [0], T=1.0, seed=5)
    wd = w.to("cuda")
    ids = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = VerifyOutput(tokens=torch.empty(1, dtype=torch.int32, device="cuda"),
                       num_accepted=torch.empty(1, dtype=torch.int32, device="cuda"), beta=None)
    V(wd.target_logits, wd.draft_probs, ids, wd.cu, w.T, w.seed, out=out)
    g = dict(tokens=out.tokens.cpu().numpy(), num_accepted=out.num_accepted.cpu().numpy())
    w = from_rows(t, torch.zeros(0, 4096), torch.zeros(0, dtype=torch.int32), [0], T=1.0, seed=5)
    r = run_oracle(w)
    assert g["num_accepted"][0] == 0 and g["tokens"][0] == r.tokens[0]


def test_every_request_bonus_only_with_empty_draft_tensors(V):
    # gamma = 0 for every request: the binding passes empty draft tensors (the
    # C ABI then gets a valid dummy address for draft_ids); only bonus tokens
    t = torch.randn(6, 3000, generator=torch.Generator().manual_seed(9)) * 2
    w = from_rows(t, torch.zeros(0, 3000), torch.zeros(0, dtype=torch.int32), [0] * 6, T=0.8,
                  seed=17)
    g = run_gpu(V, w)
    r = run_oracle(w)
    st = compare(w, g, r)
    assert flag_budget_ok(st), st
    assert (g["num_accepted"] == 0).all()


def test_masked_logits_and_zero_draft_probs(V):
    # -inf logits (masked vocabulary) and q(x) = 0 < p(x) (always accepted)
    Vs, gam, B = 2048, 3, 6
    g0 = torch.Generator().manual_seed(3)
    tgt = torch.randn(B * (gam + 1), Vs, generator=g0) * 2
    tgt[:, 100:900] = -float("inf")
    q = torch.softmax(torch.randn(B * gam, Vs, generator=g0), -1)
    q[:, :50] = 0.0
    q = q / q.sum(-1, keepdim=True)
    ids = torch.randint(0, 50, (B * gam,), generator=g0, dtype=torch.int32)   # q(x) = 0
    ids[::4] = 500                                                             # p(x) = 0
    w = from_rows(tgt, q, ids, [gam] * B, T=1.0, seed=8).to("cuda")
    g = run_gpu(V, w)
    r = run_oracle(w)
    compare(w, g, r)
    acc = g["accept"].reshape(B, gam)
    assert (acc[np.arange(B * gam).reshape(B, gam) % 4 == 0] == 0).all()


def test_p_equals_q_accepts_all_and_disjoint_rejects_all(V):
    run = numpy_runner(V)
    same, disjoint = sc.check_d_special(run, n=20000)
    assert same["all_accepted"] and same["beta_min"] > 1 - 1e-6
    assert disjoint["none_accepted"] and disjoint["beta_max"] == 0.0
    assert same["bonus_p"] > sc.P_MIN and disjoint["correction_p"] > sc.P_MIN


def test_bad_draft_ids_flagged_not_trapped(V):
    from speculative_decoding_rejection_decode_gb300._lib import SPECDEC_DEVERR_BAD_DRAFT_ID
    w = make_config(1, B=4, V=4096)
    w.draft_ids[3] = 5000
    w.draft_ids[7] = -1
    for path in _paths().values():
        V.set_path(path)
        g = run_gpu(V, w)
        assert V.get_error() & SPECDEC_DEVERR_BAD_DRAFT_ID
        r = run_oracle(w)
        assert r.status == oracle.BAD_DRAFT_ID
        compare(w, g, r)
        assert V.get_error() == 0        # cleared by the previous read
    V.set_path(0)


def test_bf16_greedy_ties_and_signed_zero(V):
    Vs, gam, B = 3000, 4, 12
    g0 = torch.Generator().manual_seed(9)
    x = (torch.randn(B * (gam + 1), Vs, generator=g0) * 3).to(torch.bfloat16)
    for r_ in range(0, x.shape[0], 2):
        j, k = sorted(torch.randperm(Vs, generator=g0)[:2].tolist())
        top = x[r_].float().abs().max() + 1
        x[r_, j] = top
        x[r_, k] = top
    x[1] = -1.0
    x[1, 7] = -0.0
    x[1, 3] = 0.0
    am = x.float().argmax(-1)
    ids = torch.empty(B * gam, dtype=torch.int32)
    for b in range(B):
        for i in range(gam):
            ids[b * gam + i] = am[b * (gam + 1) + i] if (b + i) % 3 else (am[b * (gam + 1) + i] + 1) % Vs
    w = from_rows(x, None, ids, [gam] * B, T=0.0, seed=0)
    g = run_gpu(V, w)
    r = run_oracle(w)
    compare(w, g, r, exact=True)


def test_greedy_long_drafts(V):
    # more than 32 drafts per request: the finalize scan runs over several chunks
    w = make_workload(name="long", B=5, gamma=(0, 70), V=999, dtype="bf16", T=0.0, seed=41,
                      ids="argmax0.75", device="cuda")
    g = run_gpu(V, w)
    compare(w, g, run_oracle(w), exact=True)


def test_greedy_unaligned_vocab(V):
    w = make_config(2, B=10, V=1001)
    g = run_gpu(V, w)
    compare(w, g, run_oracle(w), exact=True)


def test_host_argument_errors(V):
    from speculative_decoding_rejection_decode_gb300 import specdec_rejection_sample
    from speculative_decoding_rejection_decode_gb300._lib import (SPECDEC_ERR_INVALID_ARG,
                                                                  SPECDEC_ERR_UNSUPPORTED_DTYPE)
    w = make_config(0).to("cuda")
    out = torch.empty(16, dtype=torch.int32, device="cuda")
    base = dict(h=V.handle, target_logits=w.target_logits.data_ptr(), dtype=0,
                draft_probs=w.draft_probs.data_ptr(), draft_ids=w.draft_ids.data_ptr(),
                cu_num_draft_tokens=w.cu.data_ptr(), B=1, V=32, T=1.0, seed=0,
                out_tokens=out.data_ptr(), out_num_accepted=out.data_ptr(), out_beta=None,
                stream=torch.cuda.current_stream().cuda_stream)
    for k, v, want in (("B", 0, SPECDEC_ERR_INVALID_ARG), ("V", 0, SPECDEC_ERR_INVALID_ARG),
                       ("T", -1.0, SPECDEC_ERR_INVALID_ARG), ("T", float("nan"), SPECDEC_ERR_INVALID_ARG),
                       ("T", float("inf"), SPECDEC_ERR_INVALID_ARG), ("dtype", 7, SPECDEC_ERR_UNSUPPORTED_DTYPE),
                       ("h", None, SPECDEC_ERR_INVALID_ARG),
                       ("out_tokens", None, SPECDEC_ERR_INVALID_ARG)):
        args = dict(base)
        args[k] = v
        assert specdec_rejection_sample(**args) == want, k


def test_reserve_then_calls_within_bounds(V):
    from speculative_decoding_rejection_decode_gb300 import Verifier
    v2 = Verifier(0)
    v2.reserve(2000, 300)
    w = make_config(3, device="cuda", B=60, V=8000)
    g = run_gpu(v2, w)
    compare(w, g, run_oracle(w))
    assert v2.get_error() == 0
    v2.close()


# --------------------------------------------------------------------------
# statistical guarantees (a)-(e), as for the oracle, on the CUDA path
# --------------------------------------------------------------------------

@pytest.mark.parametrize("path", ALL_PATHS)
def test_stat_a_b_output_distribution(V, path):
    run = numpy_runner(V, _paths()[path])
    out = sc.check_a_output_distribution(run)
    assert out["slot0"] > sc.P_MIN and out["residual"] > sc.P_MIN and out["bonus"] > sc.P_MIN
    assert out["accept_z"] < 3.0
    assert out["beta_err"] < 1e-6
    V.set_path(0)


def test_stat_a_joint_two_tokens(V):
    assert sc.check_joint_two_tokens(numpy_runner(V)) > sc.P_MIN


def test_stat_c_eq1(V):
    out = sc.check_c_eq1(numpy_runner(V))
    assert out["pvalue"] > sc.P_MIN and out["z"] < 3.0


# --------------------------------------------------------------------------
# one-hot ("greedy") drafts at T > 0: no draft rows
# --------------------------------------------------------------------------

@pytest.mark.parametrize("Vsz,dtype,T", [(32000, "f32", 1.0), (128256, "bf16", 0.8), (5003, "f32", 1.3),
                                         (256000, "bf16", 1.0), (30000, "bf16", 1.0),
                                         (40000, "f32", 0.9)])
def test_onehot_drafts_parity(V, Vsz, dtype, T):
    # 30000 bf16 and 40000 f32 end the race loop of sweep 2 inside a warp
    w = make_workload(name="onehot", B=48, gamma=(0, 7), V=Vsz, dtype=dtype, T=T, seed=61,
                      ids="argmax0.75", device="cuda")
    assert w.draft_probs is None
    g = run_gpu(V, w)
    assert V.get_error() == 0
    r = run_oracle(w)
    st = compare(w, g, r)
    assert flag_budget_ok(st), st
    assert np.all(g["q_x"] == 1.0)
    assert np.abs(g["beta"] - g["p_x"]).max() <= 1e-6      # beta = p(x)


def test_onehot_drafts_output_distribution(V):
    # the emitted token follows p and the acceptance rate is p(x)
    n, Vs, x = 300_000, 8, 2
    lt = np.array([[0.3, -1.0, 1.2, 0.0, 0.7, -0.4, 0.5, -2.0],
                   [1.0, 0.2, -0.5, 0.9, 0.0, -1.5, 0.4, 0.1]], np.float32)
    tgt = torch.from_numpy(np.tile(lt, (n, 1))).cuda()
    ids = torch.full((n,), x, dtype=torch.int32, device="cuda")
    cu = torch.arange(n + 1, dtype=torch.int32, device="cuda")
    out = V(tgt, None, ids, cu, 1.0, 9, extended=True, n_draft=n)
    torch.cuda.synchronize()
    p = sc.softmax64(lt, 1.0)
    tok0 = out.tokens.cpu().numpy().reshape(n, 2)[:, 0]
    assert sc.chi2_ok(np.bincount(tok0, minlength=Vs), p[0]) > sc.P_MIN
    acc = out.accept.cpu().numpy().mean()
    assert abs(acc - p[0, x]) < 3 * np.sqrt(p[0, x] * (1 - p[0, x]) / n)
