"""Top-k / top-p adjusted targets (the vllbc page's Section 2.2 note: top-k and
top-p fold into the adjusted p before the same rejection test): the CUDA
library through specdec_rejection_sample_topk_topp against the CPU oracle."""
import numpy as np
import pytest
import torch

import stat_checks as sc
from gpu_helpers import (compare, flag_budget_ok, run_gpu, run_gpu_adj, run_oracle,
                         run_oracle_threaded)
from speculative_decoding_rejection_decode_gb300.inputs import (from_rows, make_config,
                                                                make_top_k_top_p, make_workload)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def V():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_rejection_decode_gb300 import Verifier
    v = Verifier(0)
    yield v
    v.close()


def _check(V, w, tk, tp, budget=True):
    g = run_gpu_adj(V, w, tk, tp)
    assert V.get_error() == 0
    r = run_oracle(w, tk, tp)
    st = compare(w, g, r, top_k=tk, top_p=tp)
    if budget:
        assert flag_budget_ok(st), st
    return g, r


@pytest.mark.parametrize("vocab", [1, 2, 3, 1000, 32000, 151936, 256000, 262145, 1 << 30])
def test_selection_mass_accuracy(V, vocab):
    # a unit test of the kernel's own top-p masses (the oracle decides the edge
    # from exp in double and takes no part here): 2^-z within 4e-7 relative of
    # 2^-z, exact powers of two at integer z, 0 from z = 64 on and for NaN; the
    # integer mass is 2^-z scaled by 2^F, F = 62 - ceil(log2 V), rounded to the
    # nearest integer, so that V of them never exceed 2^62
    from speculative_decoding_rejection_decode_gb300 import selection_mass
    rng = np.random.default_rng(vocab % 1000)
    ints = np.arange(0, 70, dtype=np.float32)
    z = np.concatenate([
        rng.uniform(0, 70, 200000), rng.uniform(0, 1, 50000), rng.uniform(40, 64, 50000),
        ints, np.nextafter(ints, np.float32(np.inf)), np.nextafter(ints, np.float32(-np.inf))[1:],
        [-0.0, 63.99999, 64.0, 1e30, np.inf, np.nan]]).astype(np.float32)
    got_m, got_p = selection_mass(torch.from_numpy(z).cuda(), vocab)
    got_m = got_m.cpu().numpy().view(np.uint64).astype(np.float64)
    got_p = got_p.cpu().numpy().astype(np.float64)
    F = 62 - int(np.ceil(np.log2(vocab))) if vocab > 1 else 62
    z64 = z.astype(np.float64)
    live = np.isfinite(z64) & (z64 < 64)
    ref = np.exp2(-z64[live])
    assert np.all(np.abs(got_p[live] - ref) <= 4e-7 * ref)
    assert np.all(got_p[~live] == 0) and np.all(got_m[~live] == 0)
    at_int = live & (z64 == np.floor(z64)) & (z64 >= 0)
    assert np.array_equal(got_p[at_int], np.exp2(-z64[at_int]))
    assert np.all(np.abs(got_m[live] - got_p[live] * 2.0 ** F) <= 0.5)
    assert vocab * got_m.max() <= 2.0 ** 62


def test_selection_mass_argument_checks(V):
    from speculative_decoding_rejection_decode_gb300 import specdec_selection_mass
    assert specdec_selection_mass(None, -1, 10, None, None, None) != 0
    assert specdec_selection_mass(None, 4, 10, None, None, None) != 0
    assert specdec_selection_mass(None, 0, 0, None, None, None) != 0
    assert specdec_selection_mass(None, 0, 10, None, None, None) == 0


@pytest.mark.parametrize("idx", [0, 1, 3])
def test_standard_workloads_with_mixed_settings(V, idx):
    w = make_config(idx, device="cuda")
    tk, tp = make_top_k_top_p(w.B, w.V, seed=100 + idx)
    _check(V, w, tk, tp)


@pytest.mark.parametrize("top_k,top_p", [(50, 1.0), (0, 0.9), (20, 0.8), (1, 1.0), (0, 0.0)])
def test_large_vocab_bf16_uniform_settings(V, top_k, top_p):
    w = make_config(4, device="cuda", B=12)
    tk, tp = make_top_k_top_p(w.B, w.V, seed=0, top_k=top_k, top_p=top_p)
    _check(V, w, tk, tp)


def test_full_size_large_workload(V):
    # the large workload at full size with the seeded per-request settings,
    # against the oracle on every request (threads over request ranges)
    w = make_config(4, device="cuda")
    tk, tp = make_top_k_top_p(w.B, w.V, seed=44)
    g = run_gpu_adj(V, w, tk, tp)
    assert V.get_error() == 0
    cu = w.cu.cpu().numpy()
    sc.check_e_layout(g["tokens"], g["num_accepted"], w.draft_ids.cpu().numpy(), cu, w.V)
    r = run_oracle_threaded(w, tk, tp)
    assert r.status == 0
    st = compare(w, g, r, top_k=tk, top_p=tp)
    assert st["requests"] == w.B
    assert flag_budget_ok(st), st


@pytest.mark.parametrize("Vsz,dtype", [(8, "f32"), (8, "bf16"), (100, "f32"), (4097, "bf16"),
                                       (4099, "f32"), (12345, "f32"), (65536, "bf16"),
                                       (151936, "f32")])
def test_vocab_sizes_and_tails(V, Vsz, dtype):
    w = make_workload(name="adj tails", B=24, gamma=(0, 6), V=Vsz, dtype=dtype, T=0.9, seed=71,
                      target_std=2.0, noise_std=0.8, device="cuda")
    tk, tp = make_top_k_top_p(w.B, w.V, seed=Vsz)
    _check(V, w, tk, tp)


@pytest.mark.parametrize("T", [0.05, 0.5, 2.5, 10.0])
def test_temperatures(V, T):
    w = make_workload(name="adj temps", B=24, gamma=5, V=30000, dtype="bf16", T=T, seed=73,
                      target_std=3.0, noise_std=1.0, draft_T=T, device="cuda")
    tk, tp = make_top_k_top_p(w.B, w.V, seed=int(T * 100))
    _check(V, w, tk, tp)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ties_signed_zero_and_masked_entries(V, dtype):
    # integer logits: large tie groups at every cut; -0.0 / +0.0 are one value;
    # -inf entries are never kept and never counted as mass
    g0 = torch.Generator().manual_seed(5)
    B, gam, Vs = 32, 3, 3000
    tgt = torch.randint(-4, 5, (B * (gam + 1), Vs), generator=g0).float()
    neg0 = torch.rand(tgt.shape, generator=g0) < 0.5
    tgt = torch.where((tgt == 0) & neg0, torch.tensor(-0.0), tgt)
    tgt[:, 1000:1500] = -float("inf")
    tgt[::5, 10:] = -float("inf")          # rows with only 10 finite logits (k beyond them)
    if dtype == "bf16":
        tgt = tgt.bfloat16()
    q = torch.softmax(torch.randn(B * gam, Vs, generator=g0), -1)
    ids = torch.multinomial(q, 1, generator=g0).view(-1).int()
    w = from_rows(tgt, q, ids, [gam] * B, T=1.0, seed=12).to("cuda")
    for tk, tp in [make_top_k_top_p(B, Vs, seed=3), make_top_k_top_p(B, Vs, 0, top_k=200),
                   make_top_k_top_p(B, Vs, 0, top_k=20), make_top_k_top_p(B, Vs, 0, top_p=0.5)]:
        _check(V, w, tk, tp)


@pytest.mark.parametrize("spread", [2, 40])
def test_top_k_with_large_tie_groups(V, spread):
    # bf16 integer logits in [-spread, spread]: with spread 2 the top value alone
    # holds ~13000 entries of each row, more than the candidate list of a top-k
    # row takes (the row falls back to sweeping the whole row); with spread 40
    # the list holds the top groups; both must keep every entry of the edge group
    g0 = torch.Generator().manual_seed(spread)
    B, gam, Vs = 8, 3, 65536
    tgt = torch.randint(-spread, spread + 1, (B * (gam + 1), Vs), generator=g0).float().bfloat16()
    q = torch.softmax(torch.randn(B * gam, Vs, generator=g0), -1)
    ids = torch.multinomial(q, 1, generator=g0).view(-1).int()
    w = from_rows(tgt, q, ids, [gam] * B, T=1.0, seed=21).to("cuda")
    for k in (1, 20, 500):
        _check(V, w, *make_top_k_top_p(B, Vs, 0, top_k=k))
    _check(V, w, *make_top_k_top_p(B, Vs, 0, top_k=20, top_p=0.5))


@pytest.mark.parametrize("frac_k,top_p", [(0.999, 1.0), (0.75, 1.0), (0.6, 0.9), (1.0, 0.95)])
def test_top_k_keeping_most_of_the_row(V, frac_k, top_p):
    # 2k > V: the edge lies near the bottom of the row (k = V - 1 drops the
    # smallest value's group only when it holds one entry); with top-p the edge
    # is chosen inside the top-k set
    w = make_workload(name="adj large k", B=16, gamma=3, V=30000, dtype="bf16", T=1.0, seed=23,
                      target_std=3.0, noise_std=0.8, device="cuda")
    k = w.V - 1 if frac_k == 1.0 else int(frac_k * w.V)
    tk, tp = make_top_k_top_p(w.B, w.V, 0, top_k=k, top_p=top_p)
    _check(V, w, tk, tp)


def test_onehot_drafts_with_settings(V):
    w = make_workload(name="adj onehot", B=48, gamma=(0, 7), V=50000, dtype="bf16", T=1.0,
                      seed=77, ids="argmax0.75", device="cuda")
    tk, tp = make_top_k_top_p(w.B, w.V, seed=7)
    g, _ = _check(V, w, tk, tp)
    assert np.abs(g["beta"] - g["p_x"]).max() <= 1e-6


def test_switched_off_matches_the_plain_call(V):
    # adjusted calls run on the sweep path; compare with a plain call on that path
    from speculative_decoding_rejection_decode_gb300 import SPECDEC_PATH_SWEEP
    w = make_config(3, device="cuda", B=40, V=20000)
    V.set_path(SPECDEC_PATH_SWEEP)
    plain = run_gpu(V, w)
    off_k = torch.full((w.B,), 0, dtype=torch.int32)
    off_p = torch.full((w.B,), 1.0)
    for tk, tp in [(None, None), (off_k, None), (None, off_p), (off_k, off_p)]:
        g = run_gpu_adj(V, w, tk, tp)
        for key in plain:
            assert np.array_equal(g[key], plain[key]), key
    V.set_path(0)


def test_top_k_one_reproduces_greedy_tokens(V):
    w = make_workload(name="adj k1", B=64, gamma=(1, 6), V=20000, dtype="f32", T=1.0, seed=79,
                      ids="argmax0.75", device="cuda")
    q = torch.softmax(torch.randn(w.n_draft, w.V, generator=torch.Generator().manual_seed(1)), -1)
    ws = from_rows(w.target_logits.cpu(), q, w.draft_ids.cpu(), np.diff(w.cu.cpu().numpy()).tolist(),
                   T=1.0, seed=79).to("cuda")
    greedy = from_rows(w.target_logits.cpu(), None, w.draft_ids.cpu(),
                       np.diff(w.cu.cpu().numpy()).tolist(), T=0.0, seed=0).to("cuda")
    gg = run_gpu(V, greedy, extended=False)
    tk, tp = make_top_k_top_p(w.B, w.V, 0, top_k=1)
    g = run_gpu_adj(V, ws, tk, tp)
    assert np.array_equal(g["tokens"], gg["tokens"])
    assert np.array_equal(g["num_accepted"], gg["num_accepted"])


def test_deterministic_across_calls(V):
    w = make_config(3, device="cuda", B=40, V=20000)
    tk, tp = make_top_k_top_p(w.B, w.V, seed=9)
    a = run_gpu_adj(V, w, tk, tp)
    b = run_gpu_adj(V, w, tk, tp)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("top_k,top_p", [(3, 1.0), (0, 0.7), (5, 0.8)])
def test_output_distribution_follows_the_adjusted_target(V, top_k, top_p):
    dev = V.device

    def run(tgt, q, ids, cu, T, seed, k, p):
        B = len(cu) - 1
        out = V(torch.from_numpy(tgt).to(dev), torch.from_numpy(q).to(dev),
                torch.from_numpy(ids).to(dev), torch.from_numpy(cu).to(dev), T, seed,
                extended=True, n_draft=int(cu[-1]),
                top_k=torch.full((B,), k, dtype=torch.int32, device=dev),
                top_p=torch.full((B,), p, dtype=torch.float32, device=dev))
        torch.cuda.synchronize(dev)
        return (out.tokens.cpu().numpy(), out.num_accepted.cpu().numpy(),
                out.accept.cpu().numpy(), out.beta.cpu().numpy().astype(np.float64))
    out = sc.check_adjusted_distribution(run, top_k, top_p, n=400_000)
    assert out["slot0"] > sc.P_MIN
    assert out["residual"] > sc.P_MIN
    assert out["bonus"] > sc.P_MIN
    assert out["accept_z"] < 3.0
    assert out["beta_err"] < 1e-6


def test_argument_checks(V):
    w = make_config(1, device="cuda")
    with pytest.raises(ValueError):
        run_gpu_adj(V, w, torch.zeros(w.B + 1, dtype=torch.int32), None)
    with pytest.raises(ValueError):
        run_gpu_adj(V, w, None, torch.ones(w.B, dtype=torch.float64))


def test_greedy_ignores_settings(V):
    # at T = 0 the argmax is always kept, so top-k / top-p change nothing
    w = make_config(2, device="cuda", B=16, V=20000)
    plain = run_gpu(V, w)
    tk, tp = make_top_k_top_p(w.B, w.V, seed=11)
    g = run_gpu_adj(V, w, tk, tp)
    for key in plain:
        assert np.array_equal(g[key], plain[key]), key


def test_request_offset_shards_reproduce_the_whole_batch(V):
    # the generator index of request b is request_offset + b, with settings too
    from speculative_decoding_rejection_decode_gb300.sharding import shard_workload
    w = make_config(3, device="cuda", B=24, V=12000)
    tk, tp = make_top_k_top_p(w.B, w.V, seed=13)
    whole = run_gpu_adj(V, w, tk, tp, extended=False)
    cu = w.cu.cpu().numpy()
    for rank in range(2):
        sub, b0 = shard_workload(w, 2, rank)
        b1 = b0 + sub.B
        out = V(sub.target_logits, sub.draft_probs, sub.draft_ids, sub.cu, sub.T, sub.seed,
                n_draft=sub.n_draft, request_offset=b0, top_k=tk[b0:b1].cuda(),
                top_p=tp[b0:b1].cuda())
        torch.cuda.synchronize()
        t0, t1 = cu[b0] + b0, cu[b1] + b1
        assert np.array_equal(out.tokens.cpu().numpy(), whole["tokens"][t0:t1])
        assert np.array_equal(out.num_accepted.cpu().numpy(), whole["num_accepted"][b0:b1])


def test_selection_counters(V):
    w = make_config(1, device="cuda")
    tk, tp = make_top_k_top_p(w.B, w.V, seed=0, top_k=50, top_p=0.9)
    ctr = torch.zeros(8, dtype=torch.int64, device="cuda")
    V.set_adjust_counters(ctr)
    run_gpu_adj(V, w, tk, tp)
    V.set_adjust_counters(None)
    c = ctr.cpu().tolist()
    # every row that was verified was adjusted; none lacked a threshold
    assert c[0] >= w.B and c[0] <= w.n_target
    assert c[4] == 0
    assert c[5] == 0                   # f32 rows: the general selection
    before = list(c)
    run_gpu_adj(V, w, tk, tp)          # counters off: unchanged
    assert ctr.cpu().tolist() == before


@pytest.mark.parametrize("std,top_k,top_p,value_bins", [
    (3.0, 50, 1.0, "all"),     # bf16, edge a few octaves below the max: one bin per value
    (3.0, 0, 0.9, "all"),      # top-p alone: the bound from the compensated sweep-1 mass
    (0.02, 0, 0.9, "none"),    # logits around 0: the values above the cut span > 2048 keys
])
def test_value_bins_and_general_selection_agree_with_oracle(V, std, top_k, top_p, value_bins):
    w = make_workload(name="adj paths", B=16, gamma=3, V=40000, dtype="bf16", T=1.0, seed=19,
                      target_std=std, noise_std=0.5, device="cuda")
    tk, tp = make_top_k_top_p(w.B, w.V, 0, top_k=top_k, top_p=top_p)
    ctr = torch.zeros(8, dtype=torch.int64, device="cuda")
    V.set_adjust_counters(ctr)
    _check(V, w, tk, tp)
    V.set_adjust_counters(None)
    c = ctr.cpu().tolist()
    assert c[0] > 0 and c[4] == 0
    if value_bins == "all":
        assert c[5] == c[0]
    else:
        assert c[5] == 0
