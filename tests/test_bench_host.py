"""Host logic of bench.py on CPU: the all-cores oracle rate covers every request
once, the clock sampler's parsing and throttle flags, the committed DRAM-traffic
record's validity checks, the top-k / top-p settings of the adjusted lines, and
the reference arm under a two-rank torchrun launch (gloo)."""
import argparse
import os

import pytest
import torch

import bench
from speculative_decoding_rejection_decode_gb300.inputs import make_config


@pytest.mark.parametrize("threads", [1, 3, 12])
def test_threaded_oracle_rate_covers_every_request_once(threads):
    w = make_config(1)            # B=8, gamma=5, V=32000
    rate, nreq, npos, slowest = bench.oracle_threaded_rate(w, 600.0, threads)
    assert nreq == w.B and npos == w.n_draft
    assert rate > 0 and slowest > 0


def test_threaded_oracle_rate_with_top_k_top_p():
    w = make_config(1)
    tk = torch.full((w.B,), 5, dtype=torch.int32)
    tp = torch.full((w.B,), 0.8)
    _, nreq, npos, _ = bench.oracle_threaded_rate(w, 600.0, 4, top_k=tk, top_p=tp)
    assert nreq == w.B and npos == w.n_draft


def test_host_cpu_model_is_named():
    assert isinstance(bench.host_cpu_model(), str) and bench.host_cpu_model()


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler_with(tmp_path, lines):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    s.proc = _Done()
    s.fh = open(tmp_path / "unused.csv", "w")
    return s


def test_clock_sampler_median_and_reasons(tmp_path):
    idle = "0, 2070, 2070, 300.5, 0x0, Not Active, Not Active, Not Active, Not Active"
    capped = "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active"
    hot = "0, 1500, 2070, 1400.0, 0x40, Not Active, Active, Not Active, Not Active"
    r = _sampler_with(tmp_path, [idle, capped, idle, "garbage line"]).stop()
    assert r["sm_mhz"] == 2070 and r["sm_max_mhz"] == 2070 and r["samples"] == 3
    assert r["reasons"] == ["sw_power_cap"] and r["power_w_max"] == 1390.0
    r = _sampler_with(tmp_path, [idle, hot, hot]).stop()
    assert r["sm_mhz"] == 1500 and r["reasons"] == ["hw_thermal_slowdown"]
    r = _sampler_with(tmp_path, ["not,a,sample"]).stop()
    assert r["samples"] == 0 and r["sm_mhz"] is None


def test_recorded_traffic_needs_current_source_and_workload(tmp_path, monkeypatch):
    path = tmp_path / "traffic.txt"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.recorded_traffic("w", "k", 1000) is None          # no record
    h = bench.kernel_source_hash()
    path.write_text("# note: a comment with a colon\n"
                    f"kernel: k\nworkload_key: w\nsource_sha256_16: {h}\n"
                    "traffic_bytes_per_algorithmic_byte: 1.25\n")
    # scaled to the algorithmic bytes of the launch being reported
    assert bench.recorded_traffic("w", "k", 1000) == 1250.0
    assert bench.recorded_traffic("w", "k", 8000) == 10000.0
    assert bench.recorded_traffic("other", "k", 1000) is None
    assert bench.recorded_traffic("w", "other", 1000) is None
    path.write_text(path.read_text().replace(h, "0" * 16))
    assert bench.recorded_traffic("w", "k", 1000) is None          # taken on other kernel code


def test_secondary_workload_defaults():
    # the plain large workload carries the ragged one beside it; anything else
    # runs alone unless asked
    assert bench.parse_args([]).secondary == 3
    assert bench.parse_args(["--secondary", "-1"]).secondary is None
    assert bench.parse_args(["--config", "3"]).secondary is None
    assert bench.parse_args(["--top-k", "50"]).secondary is None
    assert bench.parse_args(["--draft", "onehot"]).secondary is None
    assert bench.parse_args(["--config", "2", "--secondary", "1"]).secondary == 1


def _args(**kw):
    base = dict(top_k=None, top_p=None, adjust_mix=False, config=4)
    base.update(kw)
    return argparse.Namespace(**base)


def test_adjust_settings():
    w = make_config(1)
    assert bench.adjust_settings(w, _args(), "cpu") == (None, None)
    assert bench.adjust_desc(_args()) is None
    tk, tp = bench.adjust_settings(w, _args(top_k=50), "cpu")
    assert tk.dtype == torch.int32 and tk.shape == (w.B,) and bool((tk == 50).all())
    assert tp is None or bool((tp == 1.0).all())
    tk, tp = bench.adjust_settings(w, _args(top_p=0.9), "cpu")
    assert tp.dtype == torch.float32 and bool((tp == torch.tensor(0.9)).all())
    assert bench.adjust_desc(_args(top_k=50, top_p=0.9)) == {"top_k": 50, "top_p": 0.9}
    tk1, tp1 = bench.adjust_settings(w, _args(adjust_mix=True), "cpu")
    tk2, tp2 = bench.adjust_settings(w, _args(adjust_mix=True), "cpu")
    assert torch.equal(tk1, tk2) and torch.equal(tp1, tp2)     # seeded
    assert bench.adjust_desc(_args(adjust_mix=True)) == "seeded per-request mix"


def test_reference_arm_two_ranks_rank0_prints_once():
    # the launch the driver uses for N > 1 (torchrun, one process per rank, gloo
    # here): rank 0 alone times the oracle and prints one line, the other rank
    # exits 0 without work
    import json
    import socket
    import subprocess
    import sys
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--config", "1", "--steps", "2", "--warmup", "1"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=root, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["metric"] == "verified draft positions/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_gpu_local_cpus_from_topology_table():
    topo = ("\tGPU0\tGPU1\tNIC0\tCPU Affinity\tNUMA Affinity\tGPU NUMA ID\n"
            "GPU0\t X \tNV18\tSYS\t0-1,3\t0\t2\n"
            "GPU1\tNV18\t X \tSYS\t100000-100003\t1\t10\n")
    cpus, numa = bench.gpu_local_cpus(0, topo)
    usable = os.sched_getaffinity(0)
    assert cpus == ({0, 1, 3} & usable or None) and numa == "0"
    assert bench.gpu_local_cpus(1, topo) == (None, "1")      # none of those CPUs exist here
    assert bench.gpu_local_cpus(2, topo) == (None, None)
    assert bench.gpu_local_cpus(0, "garbage") == (None, None)
    assert bench.parse_cpu_list("0-3,8,10-11") == {0, 1, 2, 3, 8, 10, 11}


@pytest.mark.parametrize("seed", [0, 1])
def test_adjusted_needed_bytes_by_brute_force(seed):
    # every target row, plus 32 bytes per draft-row sector holding a kept entry;
    # kept sets written out from the definitions, one entry at a time
    import numpy as np
    from speculative_decoding_rejection_decode_gb300.inputs import make_top_k_top_p, make_workload
    w = make_workload(name="t", B=7, gamma=(0, 4), V=40, dtype="bf16", T=0.7, seed=seed,
                      target_std=1.0)
    tk, tp = make_top_k_top_p(w.B, w.V, seed=5 + seed)
    got = bench.adjusted_needed_bytes(w, tk, tp, chunk=3)
    cu, V, sectors = w.cu.tolist(), w.V, 0
    for b in range(w.B):
        for i in range(cu[b + 1] - cu[b]):
            x = w.target_logits[cu[b] + b + i].double().numpy() / w.T
            k, p = int(tk[b]), float(tp[b])
            e = np.exp(x - x.max())
            keep = np.ones(V, bool)
            if 1 <= k < V:
                keep = x >= np.sort(x)[::-1][k - 1]
            s_k = e[keep].sum()
            if not p >= 1.0:
                above = np.array([e[keep & (x > x[v])].sum() for v in range(V)])
                keep &= (above < max(p, 0.0) * s_k) | (above == 0)
            sectors += len(set((np.nonzero(keep)[0] // 8).tolist()))
    assert got == w.n_target * V * 2 + 32 * sectors
    # without settings every kept set is the whole row: every sector of every draft row
    none_k, none_p = make_top_k_top_p(w.B, w.V, 0, top_k=0, top_p=1.0)
    assert bench.adjusted_needed_bytes(w, none_k, none_p) == w.n_target * V * 2 + \
        w.n_draft * 32 * ((V + 7) // 8)
