#!/usr/bin/env python3
"""Benchmark of batched speculative-decoding verification on GB300.

Default workload: chain verification at B=256, gamma=7, V=128256, bf16 logits, fp32
draft probabilities (Zipf-biased synthetic logits), the configuration the throughput
target is stated on.  One step = one specdec_verify_chain call over one batch: each
sequence evaluated left to right over rows 0..J (temperature softmax statistics, accept
tests up to the first rejection, residual/bonus draw).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--rule chain|block]

--rule block times block verification (specdec_verify_block: the draft judged jointly,
every row and q row read) on the same workload instead of the chain rule.
--rule tree times the Medusa candidate-tree walk (specdec_verify_tree) on
tree_b32_n64_v32000 (the Medusa sparse tree of 64 nodes, half the sequences greedy); rows
are B*(N+1) candidate rows per call.
--rule tree_recursive times sampled tree verification by recursive rejection
(specdec_verify_tree_recursive) on tree_rr_b32_n64_v32000 (the Medusa sparse tree's
topology, tokens drafted i.i.d. per node); rows are B*(N+1) candidate rows per call.
--rule chain_varlen times chain verification with a per-request number of verified
drafts (specdec_verify_chain_varlen), gamma_b ~ U{0..gamma} seeded per batch; rows are the
candidate rows sum(gamma_b + 1).
--rule kv_compact times accepted-branch KV compaction (specdec_compact_kv) of 128 KB cache
slots along the recursive-rejection walks of tree_rr_b32_n64_v32000; the metric is bytes
moved per second.
--rule gumbel times Gumbel-coupled verification (specdec_verify_gumbel) on the same
workload as the chain rule, with drafts from the drafter's shared-noise sampler (made
before the timed region).

Prints one JSON line (rank 0).  Metric: verified vocab rows per second, B*(gamma+1)
rows per call, whole job over all ranks.  Several GPUs run independent replicas
(sequences are independent; no collective is needed), scaling "weak".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "verified vocab rows/s (B*(gamma+1)) and achieved HBM GB/s vs GB300 peak"
UNIT = "rows/s"
DEFAULT_WORKLOAD = "chain_b256_v128256"
FALLBACK_HBM_GBS = 6800.0

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the dominant kernel, from
# one ncu capture of one workload and rule, keyed by the sha256 of that kernel's source
# files (KERNEL_SOURCES) it was taken on; reported only for that workload and rule, and
# as null once the sources differ.
NCU_TRAFFIC = {
    # all-rows chain kernels (the test hook): 525.37 MB read + 4.59 MB written
    "chain_stats": {"bytes": 529_954_816, "src_sha": "39194e10996fabbe", "workload": "chain_b256_v128256", "rule": "chain"},
    # left-to-right chain kernel: 310.02 MB read + 5.20 MB written (batch seed 0)
    "chain_seq": {"bytes": 315_212_288, "src_sha": "130ed97f2e6a85c6", "workload": "chain_b256_v128256", "rule": "chain"},
    # one-launch block kernel: 1445.90 MB read + 4.92 MB written (batch seed 0)
    "block_fused": {"bytes": 1_450_814_720, "src_sha": "baf5f641c6f7d206", "workload": "chain_b256_v128256",
                    "rule": "block"},
    # Medusa walk on a cluster: 2.30 MB read, 0 written (batch seed 0)
    "tree_walk": {"bytes": 2_304_000, "src_sha": "247e250351458bee", "workload": "tree_b32_n64_v32000", "rule": "tree"},
    # recursive rejection on a cluster: 17.88 MB read, 0 written (batch seed 0)
    "tree_rr": {"bytes": 17_883_648, "src_sha": "3bd0966d0b64712e", "workload": "tree_rr_b32_n64_v32000",
                "rule": "tree_recursive"},
}


# The translation unit of each profiled kernel and the headers it includes.
KERNEL_SOURCES = {
    "chain_seq": ("chain_seq.cu", "specdec_device.cuh", "specdec_internal.h"),
    "chain_stats": ("chain_stream.cu", "stream_common.cuh", "specdec_device.cuh", "specdec_internal.h"),
    "block_fused": ("block_fused.cu", "stream_common.cuh", "specdec_device.cuh", "specdec_internal.h"),
    "tree_walk": ("tree_walk_cluster.cu", "specdec_device.cuh", "specdec_internal.h"),
    "tree_rr": ("tree_rr_cluster.cu", "specdec_device.cuh", "specdec_internal.h"),
}


def kernel_source_sha(kernel: str | None = None) -> str:
    """sha256 (16 hex digits) of a kernel's source files, or of every CUDA source."""
    h = hashlib.sha256()
    csrc = ROOT / "speculative_decoding_token_temperature_gb300" / "csrc"
    files = ([csrc / f for f in KERNEL_SOURCES[kernel]] if kernel in KERNEL_SOURCES else
             sorted(p for p in csrc.iterdir() if p.suffix in (".cu", ".cuh", ".h")))
    for p in files:
        h.update(p.read_bytes())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, rule: str):
    """ncu traffic per launch recorded for this kernel, workload and rule, or None."""
    t = NCU_TRAFFIC.get(kernel)
    if not t or t["workload"] != workload or t["rule"] != rule or t["src_sha"] != kernel_source_sha(kernel):
        return None
    return t["bytes"]


def replica_round(rank: int, s: int) -> int:
    """The workload round (seed) of batch s on rank `rank`: replicas verify different data."""
    return 100 * rank + s


def max_over_ranks(elapsed_ms: float, dist=None, device="cpu") -> float:
    """The timed interval of the whole job: the maximum over ranks (after the barriers that
    bracket the timed region).  dist: torch.distributed or None for one process."""
    if dist is None:
        return float(elapsed_ms)
    import torch
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t)


def job_value(units_per_step: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank's units (weak scaling) over the slowest rank's time."""
    return units_per_step * world / (ms_per_step / 1e3)


def graph_timed(step, steps: int, dev, dist=None):
    """Capture `steps` calls of step(i, stream) into one CUDA graph and time one replay with
    CUDA events on the replay stream (barriers and synchronisation on both sides).  For
    launch-bound rules, whose kernels finish sooner than the host issues the next call,
    this measures the device work of exactly `steps` steps.  Returns milliseconds."""
    import torch
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for i in range(steps):
                step(i, side)
    torch.cuda.current_stream(dev).wait_stream(side)
    g.replay()  # untimed: first replay uploads the graph
    torch.cuda.synchronize()
    run = torch.cuda.current_stream(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    ev0.record(run)
    g.replay()
    ev1.record(run)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return ev0.elapsed_time(ev1)


def measured_peaks() -> dict:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            return json.loads(p.read_text())
        except Exception:
            pass
    return {}


class ClockSampler:
    """SM clock and clock-event reasons sampled every ~1 ms through NVML (ctypes, read
    only) on a background thread while the timed region runs."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, gpu_uuid: str | None):
        self.index = device_index
        self.uuid = gpu_uuid
        self.samples = []
        self.max_mhz = None
        self._stop = None
        self._thread = None
        self._nvml = None
        self._handle = None

    def _open_nvml(self):
        import ctypes
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                lib = None
        if lib is None or lib.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        ok = False
        if self.uuid:
            ok = lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) == 0
        if not ok:
            ok = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) == 0
        if not ok:
            return False
        self._nvml, self._handle = lib, h
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        return True

    def _poll(self):
        import ctypes
        lib, h = self._nvml, self._handle
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        while not self._stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                r = rs.value if get_reasons(h, ctypes.byref(rs)) == 0 else 0
                self.samples.append((float(clk.value), int(r)))
            time.sleep(0.001)

    def __enter__(self):
        import threading
        if self._open_nvml():
            self._stop = threading.Event()
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
            t0 = time.time()
            while not self.samples and time.time() - t0 < 1.0:
                time.sleep(0.001)
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=2)
        return False

    def summary(self) -> dict:
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"], "samples": 0}
        sm = [c for c, _ in self.samples]
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": min(sm), "reasons": sorted(reasons), "samples": len(sm), "source": "nvml"}


def workload_shape(name):
    import workloads
    w = workloads.CHAIN_WORKLOADS[name]
    return w["B"], w["gamma"], w["V"], w["dtype"]


def oracle_rule(rule: str):
    from oracle import specdec_oracle as so
    return so.verify_block_sequence if rule == "block" else so.verify_chain_sequence


def cpu_oracle_rate(inputs_cpu: dict, target_seconds: float, max_seqs: int | None = None, rule: str = "chain"):
    """Time the fp64 oracle (as it stands, one process) on the sequences of one batch, in
    order and again from the start, until about target_seconds of work (at most max_seqs
    sequences, or 64 passes); returns (rows/s, sequences, seconds)."""
    verify = oracle_rule(rule)
    L = inputs_cpu["logits"]
    L = L.float().numpy() if str(L.dtype) == "torch.bfloat16" else L.numpy()
    q = inputs_cpu["draft_probs"].numpy()
    d = inputs_cpu["draft_tokens"].numpy()
    T = inputs_cpu["temperatures"].numpy()
    u = inputs_cpu["uniforms"].numpy()
    B, g1 = u.shape
    n, t0 = 0, time.perf_counter()
    while n < (max_seqs or 64 * B):
        i = n % B
        verify(L[i], q[i], d[i], float(T[i]), u[i])
        n += 1
        if time.perf_counter() - t0 >= target_seconds:
            break
    dt = time.perf_counter() - t0
    return n * g1 / dt, n, dt


_ORACLE_WORKER = {}


def _oracle_worker_init(folder: str, rule: str):
    import numpy as np
    sys.path.insert(0, str(ROOT))
    for k in ("L", "q", "d", "T", "u"):
        _ORACLE_WORKER[k] = np.load(os.path.join(folder, k + ".npy"), mmap_mode="r")
    _ORACLE_WORKER["verify"] = oracle_rule(rule)


def _oracle_worker_run(job):
    """Worker w of n: sequences w, w + n, ... of the batch (cycling) for `seconds`."""
    import numpy as np
    w, n, seconds = job
    W = _ORACLE_WORKER
    B = W["u"].shape[0]
    done, i, t0 = 0, w, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        b = i % B
        W["verify"](np.asarray(W["L"][b]), np.asarray(W["q"][b]), np.asarray(W["d"][b]), float(W["T"][b]),
                    np.asarray(W["u"][b]))
        done += 1
        i += n
    return done


def cpu_oracle_rate_all_cores(inputs_cpu: dict, target_seconds: float, rule: str = "chain"):
    """The same oracle, one process per host core (a spawn-started pool over memory-mapped
    inputs: this process holds a CUDA context), sequences split round-robin, for about
    target_seconds; returns (rows/s, sequences, seconds, processes)."""
    import multiprocessing as mp
    import tempfile
    import numpy as np
    n = os.cpu_count() or 1
    L = inputs_cpu["logits"]
    L = L.float().numpy() if str(L.dtype) == "torch.bfloat16" else L.numpy()
    arrays = {"L": L, "q": inputs_cpu["draft_probs"].numpy(), "d": inputs_cpu["draft_tokens"].numpy(),
              "T": inputs_cpu["temperatures"].numpy(), "u": inputs_cpu["uniforms"].numpy()}
    g1 = arrays["u"].shape[1]
    with tempfile.TemporaryDirectory() as folder:
        for k, v in arrays.items():
            np.save(os.path.join(folder, k + ".npy"), np.ascontiguousarray(v))
        with mp.get_context("spawn").Pool(n, initializer=_oracle_worker_init, initargs=(folder, rule)) as pool:
            pool.map(_oracle_worker_run, [(w, n, 0.05) for w in range(n)])  # workers up and warm
            t0 = time.perf_counter()
            done = pool.map(_oracle_worker_run, [(w, n, target_seconds) for w in range(n)])
            dt = time.perf_counter() - t0
    nseq = int(sum(done))
    return nseq * g1 / dt, nseq, dt, n


def run_reference(args, rank):
    """The oracle as it stands, on the host cores, on the same workload and metric."""
    if rank != 0:
        return 0
    import torch
    import workloads
    torch.set_num_threads(1)
    B, g, V, dtype = workload_shape(args.workload)
    per_step = args.ref_sequences
    x = workloads.chain_workload(args.workload, 0, "cpu", B=per_step)
    verify = oracle_rule(args.rule)
    L = x["logits"].float().numpy() if dtype == "bf16" else x["logits"].numpy()
    q, d, T, u = (x[k].numpy() for k in ("draft_probs", "draft_tokens", "temperatures", "uniforms"))

    def step():
        for b in range(per_step):
            verify(L[b], q[b], d[b], float(T[b]), u[b])

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = per_step * (g + 1) / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "rule": args.rule, "B": B, "gamma": g, "V": V,
                   "logits_dtype": dtype, "step_sample_sequences": per_step},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{per_step} sequences ({per_step * (g + 1)} rows) of {args.workload} per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


TREE_RR_WORKLOAD = "tree_rr_b32_n64_v32000"
TREE_WORKLOAD = "tree_b32_n64_v32000"
KV_SLOT_BYTES = 128 * 1024  # one cache slot: 32 layers x 8 KV heads x 128 x (K, V) x bf16
KV_PREFIX = 64
KV_ROTATE = 24  # tree-slot windows rotated between steps (about 24 x 10 MB moved, over L2)


def run_kv_compact(args, rank, world, local_rank):
    """Accepted-branch KV compaction along the recursive-rejection walks of the tree
    workload: the timing contract, metric = cache bytes moved (read + written) per second."""
    import numpy as np
    import torch
    import workloads
    from oracle import specdec_oracle as so  # the tree topology only
    import speculative_decoding_token_temperature_gb300 as sd
    from speculative_decoding_token_temperature_gb300 import build as _build

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps({"impl": "reference", "unavailable": "the KV compaction rule has no CPU arm"}))
        return 0
    w = workloads.TREE_RR_WORKLOADS[TREE_RR_WORKLOAD]
    B, D = w["B"], w["depth"]
    parents, _, _ = so.medusa_sparse_tree(workloads.medusa_workload_accuracies(), 64)
    N = len(parents)
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    _build.ensure_built()
    sd.load_library()
    x = workloads.tree_rr_workload(TREE_RR_WORKLOAD, parents, replica_round(rank, 0), dev)
    walk = sd.verify_tree_recursive(*(x[k] for k in ("logits", "draft_probs", "node_tokens", "parents",
                                                     "temperatures", "uniforms")), D)
    # Step i compacts the tree slots that follow prefix KV_PREFIX + (i mod KV_ROTATE) * (N + 1):
    # the slots the steps touch add up to well over L2, so no step finds its rows there.
    cache = torch.zeros(B, KV_PREFIX + KV_ROTATE * (N + 1), KV_SLOT_BYTES // 2, dtype=torch.bfloat16, device=dev)
    prefixes = [torch.full((B,), KV_PREFIX + r * (N + 1), dtype=torch.int32, device=dev) for r in range(KV_ROTATE)]
    stream = torch.cuda.current_stream(dev)

    def step(i, st=stream):
        sd.compact_kv(cache, prefixes[i % KV_ROTATE], walk["path"], walk["num_accepted"], stream=st)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    J = walk["num_accepted"].cpu().numpy()
    moves = int(sum(sum(1 for d in range(max(j, 0)) if int(walk["path"][b, d]) != d) for b, j in enumerate(J)))
    moved = 2 * moves * KV_SLOT_BYTES
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    with ClockSampler(local_rank, uuid) as clocks:  # one short kernel per step: timed as a CUDA graph
        elapsed = graph_timed(step, args.steps, dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    eager_ms = ev0.elapsed_time(ev1) / args.steps
    ms = elapsed / args.steps
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs") or FALLBACK_HBM_GBS
    gbs = moved / (ms / 1e3) / 1e9
    line = {"metric": "KV cache bytes moved/s", "value": gbs * 1e9 * world, "unit": "B/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": TREE_RR_WORKLOAD, "rule": "kv_compact", "B": B, "N": N,
                       "slot_bytes": KV_SLOT_BYTES, "prefix": KV_PREFIX, "moves_per_step": moves,
                       "l2": f"{KV_ROTATE} slot windows rotated between steps (touched bytes larger than L2)",
                       "launch": f"CUDA graph of the {args.steps} steps; eager Python calls: {eager_ms * 1e3:.1f} us per step"},
            "roofline": {"kernel": "kv_compact", "bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                         "frac": gbs / peak, "algorithmic_bytes_per_launch": moved, "traffic": None},
            "gpu_launches": args.steps, "clocks": clocks.summary(), "kernel_src_sha": kernel_source_sha()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_tree_rr(args, rank, world, local_rank):
    """Token-tree verification on the Medusa sparse tree's topology: the recursive-rejection
    walk (rule tree_recursive, every node drafted i.i.d. from q) or the Medusa walk (rule
    tree: sample from the target at each node, descend on a matching child).  The same
    timing contract as the chain rule; rows are B*(N+1) candidate rows per call."""
    import numpy as np
    import torch
    import workloads
    from oracle import specdec_oracle as so  # the tree topology and the CPU baseline only

    medusa = args.rule == "tree"
    name = TREE_WORKLOAD if medusa else TREE_RR_WORKLOAD
    w = (workloads.TREE_WORKLOADS if medusa else workloads.TREE_RR_WORKLOADS)[name]
    B, V, D = w["B"], w["V"], w["depth"]
    parents, paths, _ = so.medusa_sparse_tree(workloads.medusa_workload_accuracies(), 64)
    N = len(parents)
    rows = B * (N + 1)
    keys = (("logits", "node_tokens", "parents", "temperatures", "uniforms") if medusa else
            ("logits", "draft_probs", "node_tokens", "parents", "temperatures", "uniforms"))
    kernel = "tree_walk" if medusa else "tree_rr"
    base = {"metric": METRIC, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "data": "synthetic"}
    cfg = {"workload": name, "rule": args.rule, "B": B, "N": N, "V": V, "max_depth": D,
           "logits_dtype": w["dtype"]}
    wor = bool(getattr(args, "without_replacement", False)) and not medusa
    if not medusa:
        cfg["draft_probs_dtype"] = "fp32"
        cfg["children"] = "drawn without replacement" if wor else "drafted i.i.d."

    def make(round_idx, device):
        if medusa:
            return workloads.tree_workload(name, parents, paths, round_idx, device)
        return workloads.tree_rr_workload(name, parents, round_idx, device, without_replacement=wor)

    def oracle_rate(x, seconds, max_seqs):
        L = x["logits"].float().numpy() if w["dtype"] == "bf16" else x["logits"].numpy()
        t, T, u = (x[k].numpy() for k in ("node_tokens", "temperatures", "uniforms"))
        q = None if medusa else x["draft_probs"].numpy()
        n, t0 = 0, time.perf_counter()
        while n < max_seqs:
            i = n % B
            if medusa:
                so.verify_tree_sequence(L[i], t[i], parents, float(T[i]), u[i], D)
            else:
                so.verify_tree_rr_sequence(L[i], q[i], t[i], parents, float(T[i]), u[i], D,
                                           without_replacement=wor)
            n += 1
            if time.perf_counter() - t0 >= seconds:
                break
        dt = time.perf_counter() - t0
        return n * (N + 1) / dt, n, dt

    if args.impl == "reference":
        if rank != 0:
            return 0
        torch.set_num_threads(1)
        x = make(0, "cpu")
        per_step = args.ref_sequences
        for _ in range(args.warmup):
            oracle_rate(x, 1e9, per_step)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            oracle_rate(x, 1e9, per_step)
        dt = (time.perf_counter() - t0) / args.steps
        value = per_step * (N + 1) / dt
        line = dict(base, impl="reference", value=value, ms_per_step=dt * 1e3, dtype="f64",
                    config=dict(cfg, step_sample_sequences=per_step),
                    cpu_baseline={"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                                  "sample": f"{per_step} sequences of {name} per step"},
                    e2e={"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0})
        print(json.dumps(line), flush=True)
        return 0

    import speculative_decoding_token_temperature_gb300 as sd
    from speculative_decoding_token_temperature_gb300 import build as _build
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    _build.ensure_built()
    sd.load_library()
    sets = [make(replica_round(rank, s), dev) for s in range(args.sets)]
    outs = [{"tokens": torch.empty(B, D + 1, dtype=torch.int32, device=dev),
             "path": torch.empty(B, D, dtype=torch.int32, device=dev),
             "num_accepted": torch.empty(B, dtype=torch.int32, device=dev),
             "status": torch.empty(B, dtype=torch.int32, device=dev)} for _ in sets]
    stream = torch.cuda.current_stream(dev)

    verify = sd.verify_tree if medusa else sd.verify_tree_recursive
    flags = {} if medusa else {"without_replacement": wor}

    def step(i, st=stream):
        x = sets[i % len(sets)]
        verify(*(x[k] for k in keys), D, out=outs[i % len(sets)], stream=st, **flags)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    # One kernel per step, shorter than the Python call that issues it: the K steps are
    # captured into a CUDA graph and its replay is timed.
    with ClockSampler(local_rank, uuid) as clocks:
        elapsed_ms = max_over_ranks(graph_timed(step, args.steps, dev, dist), dist, dev)
    ms_per_step = elapsed_ms / args.steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    eager_ms = ev0.elapsed_time(ev1) / args.steps
    per_kernel = {kernel: (elapsed_ms, args.steps)}
    k_ms, k_n = per_kernel[kernel]
    # a lower bound on the bytes the walk must read: every visited node's logits row once,
    # and (recursive rejection) the q row of every node where the walk ended with children
    es = 2 if w["dtype"] == "bf16" else 4
    has_kids = np.zeros(N + 1, dtype=bool)
    for j, a in enumerate(parents):
        has_kids[0 if a < 0 else 1 + a] = True
    alg = []
    for o in outs:
        J = o["num_accepted"].cpu().numpy()
        path = o["path"].cpu().numpy()
        tot = 0
        for b in range(B):
            if J[b] < 0:
                continue
            tot += (J[b] + 1) * V * es
            last = 0 if J[b] == 0 else 1 + int(path[b][J[b] - 1])
            if has_kids[last] and not medusa:
                tot += V * 4
        alg.append(tot)
    alg_bytes = float(np.mean(alg))
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs") or FALLBACK_HBM_GBS
    achieved = alg_bytes / (k_ms / k_n / 1e3) / 1e9 if k_n else None
    line = dict(base, value=job_value(rows, world, ms_per_step), ms_per_step=ms_per_step, dtype="f32", config=dict(
        cfg, parallelism=f"replicas x{world}", l2=f"{args.sets} seeded batches rotated (inputs larger than L2)",
        launch=f"CUDA graph of the {args.steps} steps; eager Python calls: {eager_ms * 1e3:.1f} us per step"),
        roofline={"kernel": kernel, "bound": "latency", "achieved": achieved,
                  "peak": peak, "peak_source": "measured" if peaks.get("hbm_gbs") else "fallback", "unit": "GB/s",
                  "frac": (achieved / peak) if achieved else None, "algorithmic_bytes_per_launch": alg_bytes,
                  "traffic": recorded_traffic(kernel, name, args.rule + ("_without_replacement" if wor else ""))},
        kernels_ms_per_launch={k: v[0] / v[1] for k, v in per_kernel.items() if v[1]},
        gpu_launches=int(round(sum(v[1] for v in per_kernel.values()))),
        mean_accepted=float(np.mean([o["num_accepted"].float().mean().item() for o in outs])),
        clocks=clocks.summary(), kernel_src_sha=kernel_source_sha())
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        x0 = {k: v.cpu() for k, v in sets[0].items()}
        rate, nseq, secs = oracle_rate(x0, args.cpu_seconds, 10 ** 9)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"{nseq} sequences ({nseq / B:.1f} passes over one batch of {B}), {secs:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--sets", type=int, default=3, help="input batches rotated between steps")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-sequences", type=int, default=2)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--all-rows", action="store_true",
                    help="chain rules: the all-rows streaming kernels instead of the left-to-right kernel "
                         "(the library's test hook; for comparison)")
    ap.add_argument("--without-replacement", action="store_true",
                    help="rule tree_recursive: every node's children drawn without replacement (Sequoia)")
    ap.add_argument("--rule", choices=["chain", "block", "tree", "tree_recursive", "gumbel", "chain_varlen",
                                       "kv_compact"],
                    default="chain")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.rule in ("tree", "tree_recursive"):
        return run_tree_rr(args, rank, world, local_rank)
    if args.rule == "kv_compact":
        return run_kv_compact(args, rank, world, local_rank)
    if args.impl == "reference":
        return run_reference(args, rank)

    import numpy as np
    import torch
    import workloads
    import speculative_decoding_token_temperature_gb300 as sd
    from speculative_decoding_token_temperature_gb300 import build as _build

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    _build.ensure_built()
    sd.load_library()
    if args.all_rows:
        sd.set_test_hook(sd.HOOK_CHAIN_ALL_ROWS, 1)

    B, g, V, dtype = workload_shape(args.workload)
    esize = 2 if dtype == "bf16" else 4
    rows = B * (g + 1)
    sets = [workloads.chain_workload(args.workload, replica_round(rank, s), dev) for s in range(args.sets)]
    keys = ("logits", "draft_probs", "draft_tokens", "temperatures", "uniforms")
    outs = [{"tokens": torch.empty(B, g + 1, dtype=torch.int32, device=dev),
             "num_accepted": torch.empty(B, dtype=torch.int32, device=dev),
             "status": torch.empty(B, dtype=torch.int32, device=dev),
             "p_draft": torch.empty(B, g, dtype=torch.float32, device=dev)} for _ in sets]
    stream = torch.cuda.current_stream(dev)

    verify = sd.verify_block if args.rule == "block" else sd.verify_chain
    if args.rule == "chain_varlen":
        for si, x in enumerate(sets):  # counts chosen without looking at the drafts
            gen = torch.Generator(device="cpu").manual_seed(7000 + si)
            x["gammas"] = torch.randint(0, g + 1, (B,), generator=gen, dtype=torch.int32).to(dev)

        def verify(logits, draft_probs, draft_tokens, temperatures, uniforms, out=None, stream=None, _sets=sets):
            # (host copies of the first batch in the end-to-end pass use its counts)
            gm = next((x["gammas"] for x in _sets if x["logits"] is logits), _sets[0]["gammas"])
            return sd.verify_chain_varlen(logits, draft_probs, draft_tokens, temperatures, uniforms, gm, out=out,
                                          stream=stream)
        rows = float(np.mean([float((x["gammas"] + 1).sum()) for x in sets]))
    if args.rule == "gumbel":
        gseed = 20241202
        for x in sets:  # the drafter's proposals under the shared noise
            x["draft_tokens"] = sd.gumbel_draft(x["draft_probs"], gseed)
        for o in outs:
            o.pop("p_draft")

        def verify(logits, draft_probs, draft_tokens, temperatures, uniforms, out=None, stream=None):
            return sd.verify_gumbel(logits, draft_tokens, temperatures, gseed, out=out, stream=stream)

    def step(i):
        x = sets[i % len(sets)]
        verify(*(x[k] for k in keys), out=outs[i % len(sets)], stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    accepted = [float(o["num_accepted"].float().mean()) for o in outs]

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    # Timed region: K steps bracketed by a barrier and a synchronize on both sides, CUDA
    # events on the launching stream, clocks sampled throughout.
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank, uuid) as clocks:
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        ev0.record(stream)
        for i in range(args.steps):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
    elapsed_ms = max_over_ranks(ev0.elapsed_time(ev1), dist, dev)
    ms_per_step = elapsed_ms / args.steps
    value = job_value(rows, world, ms_per_step)

    # Per-kernel durations: the same K steps again with every library launch bracketed
    # by CUDA events on the launching stream.
    with sd.KernelTimer(max_launches=8 * args.steps + 16) as kt:
        torch.cuda.synchronize()
        for i in range(args.steps):
            step(i)
        torch.cuda.synchronize()
        per_kernel = kt.read()
    launches_per_step = sum(v[1] for v in per_kernel.values()) / args.steps

    # roofline of the dominant kernel
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or FALLBACK_HBM_GBS
    # rows a left-to-right verifier must read: 0..J of every sequence (the bonus row too
    # when all gamma drafts are accepted), and the draft row q_J of each rejection
    gcap = [x["gammas"] if "gammas" in x else torch.full((B,), g, dtype=torch.int32, device=dev) for x in sets]
    n_rej = sum(float((o["num_accepted"] < gc).float().sum()) for o, gc in zip(outs, gcap)) / len(outs)
    rows_read = sum(float((torch.minimum(o["num_accepted"], gc) + 1).float().sum())
                    for o, gc in zip(outs, gcap)) / len(outs)
    seq_bytes = rows_read * V * esize + n_rej * V * 4
    if args.rule == "gumbel":
        # rows 0..J of every sequence (no q row: the race needs only the target's logits)
        seq_bytes = rows_read * V * esize
        kname, alg_bytes = "gumbel", seq_bytes
    elif args.rule == "block":
        # block verification reads every logits row and every q row: the statistics pass
        # reads the logits, the mass pass both
        seq_bytes = rows * V * esize + B * g * V * 4
        per_kernel_bytes = {"chain_stats": rows * V * esize, "chain_sample": seq_bytes, "block_fused": seq_bytes}
        kname = max(per_kernel_bytes, key=lambda k: per_kernel.get(k, (0.0, 0))[0])
        alg_bytes = per_kernel_bytes[kname]
    elif per_kernel.get("chain_seq", (0.0, 0))[1]:
        kname, alg_bytes = "chain_seq", seq_bytes
    else:
        kname, alg_bytes = "chain_stats", rows * V * esize   # every logits row read once
    k_ms, k_n = per_kernel[kname]
    achieved = alg_bytes / (k_ms / k_n / 1e3) / 1e9 if k_n else None
    traffic_val = recorded_traffic(kname, args.workload, args.rule)
    # bytes one whole call must move (the same left-to-right count for either chain
    # kernel set; every row and q row for the block rule)
    call_bytes = seq_bytes
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "rule": args.rule, "B": B, "gamma": g, "V": V,
                   "logits_dtype": dtype, "draft_probs_dtype": "fp32", "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2, {args.sets} seeded batches rotated",
                   **({"path": "all-rows kernels (library test hook)"} if args.all_rows else {})},
        "hbm_gbs_call": call_bytes / (ms_per_step / 1e3) / 1e9,
        "roofline": {"kernel": kname, "bound": "hbm", "achieved": achieved, "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s",
                     "frac": (achieved / peak) if achieved else None,
                     "algorithmic_bytes_per_launch": alg_bytes, "traffic": traffic_val},
        "rows_read_per_step": rows_read,
        "kernels_ms_per_launch": {k: (v[0] / v[1] if v[1] else None) for k, v in per_kernel.items() if v[1]},
        # the Gumbel call is one timed scope of 2 launches per wave of two rows
        # (a left-to-right call also launches the one-block kernel that clears its counters)
        "gpu_launches": int(round(launches_per_step * args.steps)) * (2 * ((g + 2) // 2) if args.rule == "gumbel" else 1)
                        + (args.steps if kname == "chain_seq" else 0),
        "mean_accepted": statistics.mean(accepted),
        "clocks": clocks.summary(),
        "kernel_src_sha": kernel_source_sha(kname),
    }

    if not args.no_e2e:
        host = {k: sets[0][k].cpu().pin_memory() for k in keys}
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = sum(t.numel() * t.element_size() for t in outs[0].values())
        rows_in_place = args.rule in ("chain", "chain_varlen") and per_kernel.get("chain_seq", (0.0, 0))[1] > 0
        if rows_in_place:
            # The chain calls leave pinned logits and draft probabilities where they are
            # and the kernel reads the rows the round needs over the host link: count the
            # other inputs' copies plus those rows (rows 0..J and q row J of this batch).
            o0, gc0 = outs[0], gcap[0]
            read0 = float((torch.minimum(o0["num_accepted"], gc0) + 1).float().sum()) * V * esize
            read0 += float((o0["num_accepted"] < gc0).float().sum()) * V * 4
            h2d = sum(host[k].numel() * host[k].element_size() for k in keys[2:]) + int(read0)
        for _ in range(2):
            verify(*(host[k] for k in keys))
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            res = verify(*(host[k] for k in keys))
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = e0.elapsed_time(e1) / args.e2e_steps
        assert res["tokens"].device.type == "cpu"
        line["e2e"] = {"value": rows * world / (e_ms / 1e3), "unit": UNIT, "ms_per_step": e_ms,
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
        if rows_in_place:
            line["e2e"]["host_rows"] = "read in place from pinned host memory (rows 0..J, q row J)"

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        x0 = {k: sets[0][k].cpu() for k in keys}
        rate, nseq, secs = cpu_oracle_rate(x0, args.cpu_seconds, rule=args.rule)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"{nseq} sequences ({nseq * (g + 1)} rows; {nseq / B:.1f} passes over the "
                                          f"{B} sequences of one batch), {secs:.1f} s"}
        prate, pseq, psecs, procs = cpu_oracle_rate_all_cores(x0, args.cpu_seconds / 2, rule=args.rule)
        line["cpu_baseline"]["all_cores"] = {
            "value": prate, "unit": UNIT, "cores": procs, "kind": "oracle",
            "sample": f"{pseq} sequences of the same batch ({pseq * (g + 1)} rows), one process per host core "
                      f"(os.cpu_count() = {procs}), {psecs:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
