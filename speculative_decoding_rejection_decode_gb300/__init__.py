"""GB300 speculative-sampling verifier.

The verify step of speculative decoding (Algorithm 1 of Leviathan et al.; see
include/specdec.h for the exact contract) runs in hand-written CUDA kernels in
``libspecdec.so``; this package only marshals torch tensors into the C ABI.

    from speculative_decoding_rejection_decode_gb300 import Verifier
    v = Verifier(device=0)
    out = v(target_logits, draft_probs, draft_ids, cu_num_draft_tokens, T=1.0, seed=0)
    out.tokens, out.num_accepted, out.beta

The library is loaded on first use of anything below (``Verifier``,
``uniform``, the ``specdec_*`` functions); that raises ImportError when
libspecdec.so has not been built.  ``inputs`` (synthetic workloads) needs no
library.
"""
from __future__ import annotations

_LAZY = {"Verifier", "VerifyOutput", "SpecdecError", "uniform", "neg_log_uniform",
         "specdec_create", "specdec_reserve", "specdec_rejection_sample",
         "specdec_rejection_sample_ex", "specdec_rejection_sample_topk_topp",
         "specdec_get_error", "specdec_set_path", "specdec_set_timing_events",
         "specdec_set_adjust_counters", "specdec_last_path", "specdec_uniform",
         "specdec_neg_log_uniform", "specdec_selection_mass", "selection_mass",
         "specdec_status_string", "specdec_destroy",
         "specdec_rejection_sample_noalloc", "specdec_tree_verify", "TreeOutput",
         "SPECDEC_F32", "SPECDEC_BF16",
         "SPECDEC_PATH_AUTO", "SPECDEC_PATH_FUSED", "SPECDEC_PATH_TWO_PASS", "SPECDEC_PATH_SWEEP",
         "SPECDEC_PATH_STREAM", "SPECDEC_PATH_PAIR", "SPECDEC_PATH_DUAL", "SPECDEC_PATH_GREEDY"}


def __getattr__(name):
    if name in _LAZY:
        from . import verifier
        return getattr(verifier, name)
    raise AttributeError(name)
