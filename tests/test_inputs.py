"""Host-side input generators (no GPU): the seeded workloads and per-request
top-k / top-p settings are reproducible and have the documented shapes."""
import torch

from speculative_decoding_rejection_decode_gb300.inputs import (make_config, make_top_k_top_p,
                                                                TOP_K_CHOICES, TOP_P_CHOICES)


def test_top_k_top_p_fixed_values():
    k, p = make_top_k_top_p(5, 100, seed=0, top_k=7)
    assert k.dtype == torch.int32 and p.dtype == torch.float32
    assert k.tolist() == [7] * 5 and p.tolist() == [1.0] * 5
    k, p = make_top_k_top_p(3, 100, seed=0, top_p=0.5)
    assert k.tolist() == [0] * 3 and p.tolist() == [0.5] * 3


def test_top_k_top_p_mix_is_seeded_and_covers_edges():
    V = 1000
    a = make_top_k_top_p(4096, V, seed=3)
    b = make_top_k_top_p(4096, V, seed=3)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    k, p = a
    ks = set(k.tolist())
    ps = set(round(x, 6) for x in p.tolist())
    # off, each listed value and the edge values all occur
    for v in list(TOP_K_CHOICES) + [V - 1, V, V + 7, -1, 0]:
        assert v in ks, v
    for v in list(TOP_P_CHOICES) + [0.0, 1e-6, 1.0, 1.5]:
        assert round(v, 6) in ps, v
    # about a fifth of the requests use neither
    neither = ((k == 0) | (k >= V) | (k < 0)) & (p >= 1.0)
    assert 0.1 < neither.float().mean().item() < 0.45


def test_config_layout():
    w = make_config(3, B=12, V=64)
    cu = w.cu.tolist()
    assert cu[0] == 0 and all(b >= a for a, b in zip(cu, cu[1:]))
    assert w.target_logits.shape == (cu[-1] + 12, 64)
    assert w.draft_probs.shape == (cu[-1], 64)
    assert torch.allclose(w.draft_probs.sum(-1), torch.ones(cu[-1]), atol=1e-5)
    w2 = make_config(3, B=12, V=64)
    assert torch.equal(w.target_logits, w2.target_logits) and torch.equal(w.draft_ids, w2.draft_ids)
