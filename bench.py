#!/usr/bin/env python
"""Throughput of the GB300 speculative-sampling verifier.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one verify call over the whole synthetic batch (row kernel, first-
rejection scan, deferred-race kernel).  Default workload: the large batch
(B=1024 requests, gamma=7 drafts, V=256000, bf16 target logits, f32 draft
probabilities, T=1), whose 11.5 GB of inputs dwarf the 129 MB L2, so no L2
flush is needed between steps.  Prints one JSON line (rank 0).

--impl reference times the CPU oracle (the plain double-precision C
implementation the tests compare against) on the host cores, on a bounded
sample of the same workload.

Multi-GPU (torchrun, one rank per GPU): requests are independent, so every rank
verifies its own full batch (weak scaling, no collective on the data path); the
barrier and the max over ranks are for timing only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft positions/s"
UNIT = "positions/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["speculative_decoding_rejection_decode_gb300/csrc/kernels.cuh",
                  "speculative_decoding_rejection_decode_gb300/csrc/device_common.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "row_kernel_traffic_large_workload.txt")
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e data-sheet bandwidth (context beside the measured peak)


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=4, help="standard workload 0..4")
    ap.add_argument("--batch", type=int, default=None, help="override B (smaller case)")
    ap.add_argument("--vocab", type=int, default=None, help="override V")
    ap.add_argument("--path", choices=["auto", "fused", "sweep", "stream", "pair", "dual", "two_pass"],
                    default="auto")
    ap.add_argument("--draft", choices=["probs", "onehot"], default="probs",
                    help="onehot: no draft rows (a greedy drafter, q = one-hot at the draft id)")
    ap.add_argument("--top-k", type=int, default=None,
                    help="top-k of every request (adjusted target rows)")
    ap.add_argument("--top-p", type=float, default=None,
                    help="top-p of every request (adjusted target rows)")
    ap.add_argument("--adjust-mix", action="store_true",
                    help="a seeded per-request mix of top-k / top-p settings")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-threads", type=int, default=0,
                    help="threads of the all-cores oracle rate (0: every usable core; 1: skip it)")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-streams", type=int, default=1,
                    help="host-to-device copies of a step split over this many streams")
    ap.add_argument("--e2e-compare", action="store_true",
                    help="also time e2e with the pinned inputs placed by default (no CPU pinning)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--secondary", type=int, default=None,
                    help="a second standard workload timed in the same run and reported as "
                         "'secondary' (default: the ragged workload 3 beside the plain large "
                         "workload 4; -1: none)")
    ap.add_argument("--secondary-steps", type=int, default=200)
    ap.add_argument("--tree", action="store_true",
                    help="token trees (specdec_tree_verify): B=512 requests of V=256000 bf16 "
                         "target rows, f32 draft rows, T=1, every tree 4 root candidates, 2 "
                         "below each, then chains (29 nodes)")
    args = ap.parse_args(argv)
    if args.tree:
        args.secondary = -1
    if args.secondary is None:
        plain = (args.config == 4 and args.batch is None and args.vocab is None
                 and args.draft == "probs" and args.path == "auto" and args.top_k is None
                 and args.top_p is None and not args.adjust_mix)
        args.secondary = 3 if plain else -1
    if args.secondary < 0:
        args.secondary = None
    return args


# ----------------------------------------------------------------------------
# distributed plumbing (timing only)
# ----------------------------------------------------------------------------

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"specdec_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict | None:
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, power, reasons = [], [], [], set()
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "reasons": sorted(reasons), "samples": len(sm)}


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_key: str, kernel: str, alg_bytes: int):
    """DRAM bytes per launch of the row kernel, scaled from the committed ncu
    summary: that record holds the DRAM bytes per algorithmic byte of one
    launch captured on a smaller batch of the same workload (same vocabulary,
    dtypes and draft depth; the batch is left out of the key), taken on the
    current kernel source.  None when no such record exists."""
    try:
        vals = {}
        for line in open(TRAFFIC_FILE):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
        if vals.get("source_sha256_16") != kernel_source_hash():
            return None
        if vals.get("workload_key") != workload_key or vals.get("kernel") != kernel:
            return None
        return float(vals["traffic_bytes_per_algorithmic_byte"]) * alg_bytes
    except (OSError, KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------
# CPU oracle timing (baseline / reference arm)
# ----------------------------------------------------------------------------

def oracle_sample_rate(w, seconds: float, start_request: int = 0, top_k=None, top_p=None):
    """Runs the oracle request by request for about `seconds` of wall time;
    returns (positions/s, requests done, positions done, elapsed)."""
    import oracle
    from speculative_decoding_rejection_decode_gb300.inputs import to_numpy_logits
    cu = w.cu.cpu().numpy().astype("int64")
    tk = None if top_k is None else top_k.cpu().numpy()
    tp = None if top_p is None else top_p.cpu().numpy()
    done_req = done_pos = 0
    elapsed = 0.0
    b = start_request
    while (elapsed < seconds or done_req < 2) and done_req < w.B:
        b = b % w.B
        d0, d1 = cu[b], cu[b + 1]
        tgt = to_numpy_logits(w.target_logits[d0 + b:d1 + b + 1])
        q = None if w.draft_probs is None else w.draft_probs[d0:d1].cpu().numpy()
        ids = w.draft_ids[d0:d1].cpu().numpy()
        t0 = time.perf_counter()
        oracle.verify_request(int(b), tgt, q, ids, w.T, w.seed,
                              top_k=0 if tk is None else int(tk[b]),
                              top_p=1.0 if tp is None else float(tp[b]))
        elapsed += time.perf_counter() - t0
        done_req += 1
        done_pos += int(d1 - d0)
        b += 1
    return done_pos / elapsed, done_req, done_pos, elapsed


def oracle_threaded_rate(w, seconds: float, threads: int, top_k=None, top_p=None):
    """The same oracle call on `threads` host threads, each over its own
    contiguous range of requests (the oracle's C calls release the GIL).  Each
    thread stops after about `seconds` of oracle time or at the end of its range.
    Returns (positions/s over the slowest thread's oracle time, requests done,
    positions done, that time)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    from speculative_decoding_rejection_decode_gb300.inputs import to_numpy_logits
    from speculative_decoding_rejection_decode_gb300.sharding import shard_bounds
    oracle.build()
    oracle.splitmix64(0)          # loads the library once, before the threads start
    cu = w.cu.cpu().numpy().astype("int64")
    tk = None if top_k is None else top_k.cpu().numpy()
    tp = None if top_p is None else top_p.cpu().numpy()

    def work(r):
        b0, b1 = shard_bounds(w.B, threads, r)
        nreq = npos = 0
        el = 0.0
        for b in range(b0, b1):
            if el >= seconds:
                break
            d0, d1 = cu[b], cu[b + 1]
            tgt = to_numpy_logits(w.target_logits[d0 + b:d1 + b + 1])
            q = None if w.draft_probs is None else w.draft_probs[d0:d1].cpu().numpy()
            ids = w.draft_ids[d0:d1].cpu().numpy()
            t0 = time.perf_counter()
            oracle.verify_request(int(b), tgt, q, ids, w.T, w.seed,
                                  top_k=0 if tk is None else int(tk[b]),
                                  top_p=1.0 if tp is None else float(tp[b]))
            el += time.perf_counter() - t0
            nreq += 1
            npos += int(d1 - d0)
        return nreq, npos, el

    with ThreadPoolExecutor(max_workers=threads) as pool:
        parts = list(pool.map(work, range(threads)))
    nreq = sum(p[0] for p in parts)
    npos = sum(p[1] for p in parts)
    slowest = max(p[2] for p in parts)
    return npos / max(slowest, 1e-12), nreq, npos, slowest


def host_cpu_model() -> str:
    """The host CPU's model name (from /proc/cpuinfo, else lscpu), or the
    machine type."""
    import platform
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return f"{platform.machine()} {line.split(':', 1)[1].strip()}"
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine()


def adjust_settings(w, args, device, config=None):
    """Per-request top-k / top-p tensors for the adjusted-target bench lines
    (None, None for the plain verify step)."""
    if args.top_k is None and args.top_p is None and not args.adjust_mix:
        return None, None
    from speculative_decoding_rejection_decode_gb300.inputs import make_top_k_top_p
    if args.adjust_mix:
        cfg = args.config if config is None else config
        return make_top_k_top_p(w.B, w.V, seed=1000 + cfg, device=device)
    return make_top_k_top_p(w.B, w.V, seed=0, top_k=args.top_k, top_p=args.top_p, device=device)


def adjusted_needed_bytes(w, tk, tp, chunk: int = 128) -> int:
    """Bytes an adjusted step must read at the least: every target row once,
    and of each draft row only the 32-byte sectors holding an entry of its
    adjusted target's kept set (p' = 0 elsewhere, so neither beta nor the
    residual needs q there).  The kept sets follow the definitions (top-k keeps
    the ties at the k-th largest logit; top-p keeps v when the mass strictly
    above it is below P times the top-k set's mass, or is 0), computed in
    float64 with torch on the workload's device, outside any timed region."""
    import torch
    esize = 2 if w.dtype == "bf16" else 4
    need = w.n_target * w.V * esize
    if w.draft_probs is None or w.n_draft == 0:
        return need
    dev = w.target_logits.device
    V = w.V
    gam = (w.cu[1:] - w.cu[:-1]).long().to(dev)
    req = torch.repeat_interleave(torch.arange(w.B, device=dev), gam)
    trow = torch.arange(w.n_draft, device=dev) + req
    tk, tp = tk.to(dev), tp.to(dev)
    sectors = 0
    for d0 in range(0, w.n_draft, chunk):
        d1 = min(w.n_draft, d0 + chunk)
        x = w.target_logits[trow[d0:d1]].double() / w.T
        k = tk[req[d0:d1]].long()
        p = tp[req[d0:d1]].double()
        vals, order = torch.sort(x, dim=1, descending=True)
        e = torch.exp(vals - vals[:, :1])
        use_k = (k >= 1) & (k < V)
        thr = vals.gather(1, (k - 1).clamp(0, V - 1)[:, None])[:, 0]
        thr = torch.where(use_k, thr, torch.full_like(thr, -float("inf")))
        keep = vals >= thr[:, None]
        ek = e * keep
        s_k = ek.sum(1)
        neg = (-vals).contiguous()
        first = torch.searchsorted(neg, neg)          # first index of each value's group
        above = (torch.cumsum(ek, 1) - ek).gather(1, first)
        use_p = ~(p >= 1.0)
        in_p = (above < (p.clamp(min=0.0) * s_k)[:, None]) | (above == 0)
        keep &= in_p | ~use_p[:, None]
        sec = torch.zeros(d1 - d0, (V + 7) // 8, dtype=torch.int32, device=dev)
        sec.scatter_add_(1, order // 8, keep.int())
        sectors += int((sec > 0).sum())
        del x, vals, order, e, keep, ek, neg, first, above, sec
    return need + 32 * sectors


def adjust_desc(args):
    if args.adjust_mix:
        return "seeded per-request mix"
    if args.top_k is None and args.top_p is None:
        return None
    return {"top_k": args.top_k, "top_p": args.top_p}


def workload_desc(w, args, flush: bool, in_bytes: int, config=None) -> dict:
    gam = w.meta.get("gamma")
    d = {
        "workload": f"{w.name} (standard workload {args.config if config is None else config})",
        "B": w.B, "gamma": list(gam) if isinstance(gam, tuple) else gam, "V": w.V,
        "target_dtype": w.dtype, "draft_dtype": None if w.draft_probs is None else "f32",
        "T": w.T, "n_draft_positions": w.n_draft, "n_target_rows": w.n_target,
        "input_bytes": in_bytes,
        "l2": ("flushed between steps (256 MB write, then 256 MB read)" if flush else
               f"inputs ({in_bytes / 1e9:.2f} GB) larger than L2 (129 MB); no flush"),
    }
    if adjust_desc(args) is not None:
        d["top_k_top_p"] = adjust_desc(args)
        d["workload"] += " with top-k / top-p"
    return d


class Measured:
    """One workload timed on the GPU: the JSON fields and what the extra legs
    (selection counters, acceptance, e2e, CPU baseline) need."""

    def __init__(self, **kw):
        self.__dict__.update(kw)


def measure(args, dist, dev, sd, config: int, steps: int, warmup: int) -> Measured:
    """Times `steps` verify steps of standard workload `config` (after `warmup`
    untimed ones) with CUDA events on the call's stream, the row kernel timed
    by events the library records around it."""
    import torch
    from speculative_decoding_rejection_decode_gb300.inputs import make_config
    w = make_config(config, device=dev, B=args.batch, V=args.vocab)
    if args.draft == "onehot":
        w.draft_probs = None
        w.name += " one-hot drafts"
    esize = 2 if w.dtype == "bf16" else 4
    tgt_bytes = w.n_target * w.V * esize
    drf_bytes = 0 if w.draft_probs is None else w.n_draft * w.V * 4
    in_bytes = tgt_bytes + drf_bytes
    flush = in_bytes < 4 * L2_BYTES
    alg_bytes_step = w.algorithmic_bytes()       # + one extra target row per request
    alg_bytes_rows = tgt_bytes + drf_bytes       # what the row kernel must read
    workload_key = f"config{config}-V{w.V}-{w.dtype}-{args.draft}"
    tk, tp = adjust_settings(w, args, dev, config)
    if tk is not None:
        workload_key += "-adjusted"

    v = sd.Verifier(dev)
    v.reserve(w.n_draft, w.B)
    if args.path != "auto":
        v.set_path({"fused": sd.SPECDEC_PATH_FUSED, "sweep": sd.SPECDEC_PATH_SWEEP,
                    "stream": sd.SPECDEC_PATH_STREAM, "pair": sd.SPECDEC_PATH_PAIR,
                    "dual": sd.SPECDEC_PATH_DUAL, "two_pass": sd.SPECDEC_PATH_TWO_PASS}[args.path])
    out = sd.VerifyOutput(tokens=torch.empty(w.n_target, dtype=torch.int32, device=dev),
                          num_accepted=torch.empty(w.B, dtype=torch.int32, device=dev),
                          beta=torch.empty(w.n_draft, dtype=torch.float32, device=dev))
    offset = dist.rank * w.B
    # L2 flush between steps: write a 256 MB buffer (twice L2), then read another
    # 256 MB buffer so that the flush's dirty lines are written back during the
    # flush and not while the next step's kernels run
    scratch = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev) if flush else None
    scratch_rd = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev) if flush else None

    def flush_l2():
        scratch.fill_(1.0)
        scratch_rd.amax()

    def step():
        v(w.target_logits, w.draft_probs, w.draft_ids, w.cu, w.T, w.seed, out=out,
          request_offset=offset, top_k=tk, top_p=tp)

    for _ in range(max(3, warmup)):
        if flush:
            flush_l2()
        step()
    torch.cuda.synchronize(dev)
    if v.get_error() != 0:
        raise RuntimeError("device error word set during warm-up")
    path, csize = v.last_path()
    launches_per_step = {sd.SPECDEC_PATH_FUSED: 3, sd.SPECDEC_PATH_TWO_PASS: 4,
                         sd.SPECDEC_PATH_SWEEP: 3, sd.SPECDEC_PATH_STREAM: 3, sd.SPECDEC_PATH_PAIR: 3,
                         sd.SPECDEC_PATH_DUAL: 3,
                         sd.SPECDEC_PATH_GREEDY: 2}[path]
    kernel_name = {sd.SPECDEC_PATH_FUSED: "fused_row_kernel", sd.SPECDEC_PATH_SWEEP: "sweep_row_kernel",
                   sd.SPECDEC_PATH_STREAM: "stream_row_kernel", sd.SPECDEC_PATH_PAIR: "pair_row_kernel",
                   sd.SPECDEC_PATH_DUAL: "dual_row_kernel",
                   sd.SPECDEC_PATH_TWO_PASS: "stats_kernel+verify_kernel",
                   sd.SPECDEC_PATH_GREEDY: "greedy_partial_kernel"}[path]
    path_name = {1: "fused", 2: "two_pass", 3: "sweep", 4: "greedy", 5: "stream", 6: "pair",
                 7: "dual"}[path]

    K = steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    stream = torch.cuda.current_stream(dev)
    for e in ev:               # materialise the CUDA events before handing them over
        for x in e:
            x.record(stream)
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.25)
    dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.perf_counter()
    for k in range(K):
        if flush:
            flush_l2()
        s0, r0, r1, s1 = ev[k]
        v.set_timing_events(r0, r1)
        s0.record(stream)
        step()
        s1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall0
    dist.barrier()
    clocks = sampler.stop()
    v.set_timing_events(None, None)
    if v.get_error() != 0:
        raise RuntimeError("device error word set during the timed steps")

    step_ms = [e[0].elapsed_time(e[3]) for e in ev]
    row_ms = [e[1].elapsed_time(e[2]) for e in ev]
    region_ms = ev[0][0].elapsed_time(ev[-1][3]) if not flush else sum(step_ms)
    total_s = dist.max(region_ms / 1e3)
    ms_per_step = total_s * 1e3 / K
    value = w.n_draft * dist.world * K / total_s
    row_avg_ms = statistics.mean(row_ms)
    peak, peak_kind = measured_peak_gbs()
    achieved = alg_bytes_rows / (row_avg_ms / 1e3) / 1e9
    traffic = recorded_traffic(workload_key, kernel_name, alg_bytes_rows)
    needed = adjusted_needed_bytes(w, tk, tp) if tk is not None else None

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": K,
        "warmup": max(3, warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_desc(w, args, flush, in_bytes, config),
        "requests_per_s": w.B * dist.world * K / total_s,
        "achieved_gbps_step": alg_bytes_step / (ms_per_step / 1e3) / 1e9,
        "algorithmic_bytes_per_step": alg_bytes_step,
        "frac_step_of_peak": alg_bytes_step / (ms_per_step / 1e3) / 1e9 / peak,
        "roofline": {"bound": "hbm", "kernel": kernel_name,
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": alg_bytes_rows,
                     "avg_launch_ms": row_avg_ms, "min_launch_ms": min(row_ms),
                     "median_launch_ms": statistics.median(row_ms),
                     "share_of_step": row_avg_ms / statistics.mean(step_ms)},
        "step_ms_median": statistics.median(step_ms), "step_ms_min": min(step_ms),
        "path": path_name, "cluster_size": csize,
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
        "wall_s_timed_region": t_wall,
    }
    if needed is not None:
        # adjusted rows need q only where p' > 0: rows that keep few entries
        # (top-k) read far less than a whole draft row, so the row kernel can
        # exceed the roofline of the every-row figure above; this is its rate
        # against the bytes such a step must read at the least
        result["roofline"]["needed_bytes_per_launch"] = needed
        result["roofline"]["frac_of_needed"] = needed / (row_avg_ms / 1e3) / 1e9 / peak
    return Measured(result=result, v=v, w=w, out=out, stream=stream, offset=offset, tk=tk, tp=tp,
                    step=step)


TREE_SHAPE = [4, 2, 1, 1]


def measure_tree(args, dist, dev, sd):
    """Times the token-tree entry point: the kernel walks every request from
    its root, so the bytes it must read are the target rows of the nodes it
    visits and the draft rows of those that have children (counted from the
    accepted paths); reported against that."""
    import torch
    from speculative_decoding_rejection_decode_gb300.inputs import make_tree_workload
    B = args.batch or 512
    Vv = args.vocab or 256000
    w = make_tree_workload(name=f"token trees B={B} V={Vv} bf16 T=1 shape {TREE_SHAPE}", B=B, V=Vv,
                           dtype="bf16", T=1.0, seed=7, shape=TREE_SHAPE, device=dev)
    v = sd.Verifier(dev)
    out = None

    def step():
        nonlocal out
        out = v.tree(w.target_logits, w.draft_probs, w.node_tokens, w.node_parent, w.cu, w.T,
                     w.seed, request_offset=dist.rank * B, out=out)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if v.get_error() != 0:
        raise RuntimeError("device error word set during warm-up")
    # rows the walk must read: every visited node's target row, and the draft
    # row of each visited node that has children
    nacc = out.num_accepted.cpu()
    path = out.path.cpu()
    cu = w.cu.cpu()
    par = w.node_parent.cpu()
    visited = int(nacc.sum()) + B
    with_children = 0
    for b in range(B):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        nodes = [0] + [int(x) for x in path[s0:s0 + int(nacc[b])]]
        kids = set(int(x) for x in par[s0 + 1:s1])
        with_children += sum(1 for u in nodes if u in kids)
    alg = visited * Vv * 2 + with_children * Vv * 4
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.25)
    dist.barrier()
    torch.cuda.synchronize(dev)
    for k in range(K):
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    dist.barrier()
    clocks = sampler.stop()
    if v.get_error() != 0:
        raise RuntimeError("device error word set during the timed steps")
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_s = dist.max(ev[0][0].elapsed_time(ev[-1][1]) / 1e3)
    ms = total_s * 1e3 / K
    n_draft = w.n_nodes - B
    peak, peak_kind = measured_peak_gbs()
    achieved = alg / (statistics.mean(step_ms) / 1e3) / 1e9
    in_bytes = w.n_nodes * Vv * 6
    res = {
        "metric": "verified draft nodes/s", "value": n_draft * dist.world * K / total_s,
        "unit": "nodes/s", "n_gpus": dist.world, "steps": K, "warmup": max(3, args.warmup),
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "B": B, "V": Vv, "target_dtype": "bf16",
                   "draft_dtype": "f32", "T": 1.0, "tree_shape": TREE_SHAPE,
                   "nodes": w.n_nodes, "input_bytes": in_bytes,
                   "l2": f"inputs ({in_bytes / 1e9:.2f} GB) larger than L2 (129 MB); no flush"},
        "requests_per_s": B * dist.world * K / total_s,
        "accepted_per_request": float(nacc.double().mean()),
        "roofline": {"bound": "hbm", "kernel": "tree_walk_kernel", "achieved": achieved,
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "algorithmic_bytes_per_launch": alg,
                     "algorithmic_bytes_rule": "target row of every visited node + draft row "
                                               "of every visited node with children",
                     "avg_launch_ms": statistics.mean(step_ms)},
        "step_ms_median": statistics.median(step_ms), "step_ms_min": min(step_ms),
        "gpu_launches": K, "clocks": clocks,
    }
    v.close()
    return res


def main():
    args = parse_args()
    dist = Dist()
    import torch

    if args.impl == "reference":
        run_reference(args, dist)
        dist.close()
        return

    from speculative_decoding_rejection_decode_gb300.build import build
    build()
    import speculative_decoding_rejection_decode_gb300 as sd

    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    if args.tree:
        res = measure_tree(args, dist, dev, sd)
        if dist.rank == 0:
            print(json.dumps(res), flush=True)
        dist.close()
        return
    # the second workload the roofline target names (the ragged batch), timed in
    # the same run and reported beside the headline as "secondary"
    secondary = None
    if args.secondary is not None and args.secondary != args.config:
        m2 = measure(args, dist, dev, sd, args.secondary, args.secondary_steps, args.warmup)
        r2 = m2.result
        secondary = {k: r2[k] for k in ("value", "unit", "ms_per_step", "steps", "warmup", "config",
                                        "requests_per_s", "achieved_gbps_step",
                                        "algorithmic_bytes_per_step", "frac_step_of_peak",
                                        "roofline", "step_ms_median", "step_ms_min", "path",
                                        "cluster_size", "gpu_launches", "clocks")}
        m2.v.close()
        del m2
        torch.cuda.empty_cache()
    m = measure(args, dist, dev, sd, args.config, args.steps, args.warmup)
    result, v, w, out, stream = m.result, m.v, m.w, m.out, m.stream
    offset, tk, tp, step = m.offset, m.tk, m.tp, m.step
    if secondary is not None:
        result["secondary"] = secondary

    if tk is not None:
        # one more step with the selection counters on (outside the timed region)
        ctr = torch.zeros(8, dtype=torch.int64, device=dev)
        v.set_adjust_counters(ctr)
        step()
        torch.cuda.synchronize(dev)
        v.set_adjust_counters(None)
        c = ctr.cpu().tolist()
        result["adjust_selection_per_step"] = {
            "adjusted_rows": c[0], "sample_edge_in_tail": c[1], "edge_past_cut": c[2],
            "key_refinement_passes": c[3], "rows_without_threshold": c[4],
            "resolved_on_value_bins": c[5]}
    nacc = out.num_accepted.double()
    result["acceptance"] = {
        # accepted drafts / proposed drafts (the timinsight guide's definition)
        "draft_acceptance_rate": float(nacc.sum()) / max(w.n_draft, 1),
        # 1 + accepted per verify step and request (vLLM's mean acceptance length; Eq. (1)'s E[N])
        "mean_acceptance_length": 1.0 + float(nacc.mean()),
        # alpha = E[beta] (Corollary 3.6)
        "alpha_mean_beta": float(out.beta.double().mean()),
    }
    if not args.no_e2e:
        result["e2e"] = measure_e2e(v, w, out, dev, stream, args.e2e_steps, dist, offset, tk, tp,
                                    copy_streams=args.e2e_streams)
        if args.e2e_compare:
            d = measure_e2e(v, w, out, dev, stream, args.e2e_steps, dist, offset, tk, tp,
                            local=False, copy_streams=args.e2e_streams)
            result["e2e_default_placement"] = {k: d[k] for k in ("value", "ms_per_step",
                                                                 "h2d_gbps", "host_placement")}
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        rate, nreq, npos, el = oracle_sample_rate(w, args.cpu_seconds, top_k=tk, top_p=tp)
        cpu = host_cpu_model()
        result["cpu_baseline"] = {
            "value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {nreq} requests ({npos} draft positions) of the same workload, "
                      f"one thread, {el:.1f} s of oracle time",
            "cpu": cpu}
        if args.cpu_threads != 1:
            nthr = args.cpu_threads or len(os.sched_getaffinity(0))
            rate_n, nreq_n, npos_n, el_n = oracle_threaded_rate(w, args.cpu_seconds / 3, nthr,
                                                                top_k=tk, top_p=tp)
            result["cpu_baseline_all_cores"] = {
                "value": rate_n, "unit": UNIT, "cores": nthr,
                "kind": f"oracle, {nthr} threads over requests",
                "sample": f"{nreq_n} requests ({npos_n} draft positions) of the same workload in "
                          f"{nthr} contiguous request ranges; rate over the slowest thread's "
                          f"{el_n:.1f} s of oracle time",
                "cpu": cpu}
    if dist.rank == 0:
        print(json.dumps(result), flush=True)
    v.close()
    dist.close()


def parse_cpu_list(text: str) -> set[int]:
    """'0-3,8,10-11' -> {0, 1, 2, 3, 8, 10, 11}."""
    cpus = set()
    for part in text.split(","):
        part = part.strip()
        if not part:
            continue
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        else:
            cpus.add(int(part))
    return cpus


def gpu_local_cpus(index: int, topo: str | None = None):
    """The host CPUs nvidia-smi reports as local to GPU `index` ('CPU Affinity'
    of `nvidia-smi topo -m`) and its NUMA node, or (None, None)."""
    try:
        if topo is None:
            topo = subprocess.run(["nvidia-smi", "topo", "-m"], capture_output=True, text=True,
                                  timeout=30).stdout
        lines = [ln for ln in topo.splitlines() if ln.strip()]
        head = next(ln for ln in lines if "CPU Affinity" in ln)
        cols = [c.strip() for c in head.split("\t")]
        row = next(ln for ln in lines if ln.split("\t")[0].strip() == f"GPU{index}")
        cells = [c.strip() for c in row.split("\t")]
        cpus = parse_cpu_list(cells[cols.index("CPU Affinity")])
        numa = cells[cols.index("NUMA Affinity")] if "NUMA Affinity" in cols else None
        usable = cpus & os.sched_getaffinity(0)
        return (usable or None), numa
    except (OSError, StopIteration, ValueError, IndexError, subprocess.SubprocessError):
        return None, None


def measure_e2e(v, w, out, dev, stream, steps, dist, offset, tk=None, tp=None, local=True,
                copy_streams=1):
    """Same metric through the public API with the step's inputs in pinned host
    memory: every step copies them to the device, verifies, and reads the
    tokens, counts and beta back.  With `local`, the process runs on the CPUs
    local to the GPU while the pinned buffers are allocated and filled, so
    that their pages sit in the GPU's own NUMA node (a GB300 reaches its own
    Grace's memory over the chip-to-chip link)."""
    import torch
    placement = "default (the process's CPUs)"
    old_aff = os.sched_getaffinity(0)
    if local:
        cpus, numa = gpu_local_cpus(dev.index if dev.index is not None else 0)
        if cpus:
            os.sched_setaffinity(0, cpus)
            placement = (f"CPUs local to the GPU ({len(cpus)} of {len(old_aff)}; NUMA node "
                         f"{numa}) while the pinned buffers were allocated and filled")
    host = {}
    for name in ("target_logits", "draft_probs", "draft_ids", "cu"):
        t = getattr(w, name)
        if t is None:
            continue
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        host[name] = h
    adj = {}
    for name, t in (("top_k", tk), ("top_p", tp)):
        if t is not None:
            adj[name] = (t, torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t))
    h_out = {k: torch.empty(getattr(out, k).shape, dtype=getattr(out, k).dtype, pin_memory=True)
             for k in ("tokens", "num_accepted", "beta")}
    h2d = sum(h.numel() * h.element_size() for h in host.values())
    h2d += sum(h.numel() * h.element_size() for _, h in adj.values())
    d2h = sum(h.numel() * h.element_size() for h in h_out.values())

    # the step's host-to-device copies in `copy_streams` pieces on as many
    # streams (each piece waits for the previous step's verify, the verify
    # waits for every piece)
    nstreams = max(1, int(copy_streams))
    cstreams = [torch.cuda.Stream(dev) for _ in range(nstreams)] if nstreams > 1 else []
    free_ev = torch.cuda.Event()
    free_ev.record(stream)

    def one():
        if cstreams:
            done = []
            pieces = []
            for name, h in host.items():
                d = getattr(w, name)
                rows = d.shape[0] if d.dim() else 1
                step_rows = max(1, (rows + nstreams - 1) // nstreams) if d.dim() else rows
                for r0 in range(0, rows, step_rows):
                    pieces.append((d[r0:r0 + step_rows] if d.dim() else d,
                                   h[r0:r0 + step_rows] if d.dim() else h))
            for d, h in adj.values():
                pieces.append((d, h))
            for i, (d, h) in enumerate(pieces):
                cs = cstreams[i % nstreams]
                cs.wait_event(free_ev)
                with torch.cuda.stream(cs):
                    d.copy_(h, non_blocking=True)
            for cs in cstreams:
                ev = torch.cuda.Event()
                ev.record(cs)
                done.append(ev)
            for ev in done:
                stream.wait_event(ev)
        else:
            for name, h in host.items():
                getattr(w, name).copy_(h, non_blocking=True)
            for d, h in adj.values():
                d.copy_(h, non_blocking=True)
        v(w.target_logits, w.draft_probs, w.draft_ids, w.cu, w.T, w.seed, out=out,
          request_offset=offset, top_k=tk, top_p=tp)
        free_ev.record(stream)
        for k, h in h_out.items():
            h.copy_(getattr(out, k), non_blocking=True)

    one()
    torch.cuda.synchronize(dev)
    dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    total_s = dist.max(e0.elapsed_time(e1) / 1e3)
    os.sched_setaffinity(0, old_aff)
    return {"value": w.n_draft * dist.world * steps / total_s, "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": total_s * 1e3 / steps, "host_placement": placement,
            "h2d_gbps": h2d / (total_s / steps) / 1e9, "copy_streams": max(1, int(copy_streams))}


def run_reference(args, dist):
    """CPU oracle arm: rank 0 only; each step is the oracle over a bounded
    sample of the workload (about 2 s of CPU work)."""
    if dist.rank != 0:
        return
    import torch
    from speculative_decoding_rejection_decode_gb300.inputs import make_config
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = make_config(args.config, device=dev, B=args.batch, V=args.vocab)
    if args.draft == "onehot":
        w.draft_probs = None
        w.name += " one-hot drafts"
    tk, tp = adjust_settings(w, args, "cpu")
    per_step_s = 2.0
    for k in range(args.warmup):
        oracle_sample_rate(w, 0.0, start_request=k, top_k=tk, top_p=tp)
    rates, pos, el = [], 0, 0.0
    t0 = time.perf_counter()
    for k in range(args.steps):
        r, _, p, e = oracle_sample_rate(w, per_step_s, start_request=k * 7, top_k=tk, top_p=tp)
        rates.append(r)
        pos += p
        el += e
        if time.perf_counter() - t0 > 150:     # keep the arm within a few minutes
            break
    value = pos / el
    steps_done = len(rates)
    esize = 2 if w.dtype == "bf16" else 4
    in_bytes = w.n_target * w.V * esize + (0 if w.draft_probs is None else w.n_draft * w.V * 4)
    res = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": dist.world, "steps": steps_done, "warmup": args.warmup,
        "ms_per_step": el * 1e3 / max(steps_done, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_desc(w, args, False, in_bytes),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{pos} draft positions over {steps_done} steps of ~{per_step_s:.0f} s "
                                   "(consecutive requests of the same workload), one thread"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
