import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library through its C ABI)")
    config.addinivalue_line("markers", "slow: long-running statistical test")


def pytest_terminal_summary(terminalreporter):
    """Near-tie counts of the CUDA-vs-oracle comparisons run in this session:
    requests the oracle flags (exempt from token identity) and their rows, and
    requests whose top-p edge was ambiguous (and how many of those the library
    decided on a reachable cut other than the exact one)."""
    mod = sys.modules.get("gpu_helpers")
    log = getattr(mod, "FLAG_LOG", None) if mod else None
    if not log:
        return
    tr = terminalreporter
    tot = [sum(v[j] for v in log.values()) for j in range(5)]
    tr.write_sep("-", "near ties in the parity comparisons")
    tr.write_line(f"all comparisons: {tot[0]} flagged requests, {tot[1]} of {tot[2]} rows "
                  f"({100.0 * tot[1] / max(tot[2], 1):.4f} %); top-p edge ambiguous in "
                  f"{tot[3]} requests, decided on another reachable cut in {tot[4]}")
    for label, v in sorted(log.items()):
        if v[0] or v[3] or "config" in label:
            tr.write_line(f"  {label}: flagged {v[0]} requests / {v[1]} of {v[2]} rows; "
                          f"edge ambiguous {v[3]}, shifted {v[4]}")
