"""Benchmark of the Block AttnRes aggregation hot path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-e2e]

Workload (one step): long-context chunked prefill, 131072 tokens in 8 chunks of 16384,
d = 7168, bf16 storage with fp32 arithmetic, a resident block-representation cache
[10, 131072, 7168] whose slots 0..8 are the embedding and 8 completed blocks.  For every
chunk the step runs the whole hot path:
  query prep (u = w ⊙ gamma_key, once per step), phase 1 over the 9 sources for the block's
  24 queries, 24 phase-2 merges (fused partial update and input RMSNorm), the block close
  into slot 9, and the final aggregation over the 10 slots.
Inputs are synthetic (seeded); every launch streams >= 235 MB, far more than the 126 MB L2,
so no flush is needed between steps.

Prints one JSON line.  ``value`` is tokens/s over all ranks (each rank runs its own step on its
own GPU: tokens are independent, no collective on the data path, weak scaling).  The
reference arm (``--impl reference``) times the fp64 CPU oracle on a bounded token sample.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import queue
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from depth_wise_softmax_block_b300 import cost as C  # noqa: E402
from synth import inputs as I  # noqa: E402

METRIC = "AttnRes tokens/s per block and achieved HBM GB/s (% of B300 peak), 1 GPU"
CSRC = os.path.join(ROOT, "depth_wise_softmax_block_b300", "csrc")


def csrc_hash(files=None) -> str:
    """Hash of the kernel sources (all of them, or the named files of csrc/)."""
    h = hashlib.sha256()
    for f in sorted(files if files is not None else os.listdir(CSRC)):
        h.update(f.encode())
        h.update(open(os.path.join(CSRC, f), "rb").read())
    return h.hexdigest()[:16]


# The source files that make up each kernel kind of the step (for matching a committed ncu
# capture to the code it measured).
KERNEL_SOURCES = {
    "phase1": ["phase1_tc.cu", "tc.cuh", "tma.cuh", "tmap.cu", "common.cuh", "kernels.h"],
    "rowwise": ["rowwise.cu", "common.cuh", "kernels.h"],
    "final": ["rowwise.cu", "fullring.cu", "tma.cuh", "common.cuh", "kernels.h"],
}


def kernel_hash(kind: str) -> str:
    return csrc_hash(KERNEL_SOURCES[kind if kind in ("phase1", "final") else "rowwise"])


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return float(j["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


# --------------------------------------------------------------------------------------------
class LongContextStep:
    """The bench step.  Allocates everything once; ``run()`` allocates nothing."""

    def __init__(self, wl: I.Workload, dev, timer=None, heads: int = 1):
        from depth_wise_softmax_block_b300 import attnres_query_prep
        from depth_wise_softmax_block_b300.schedule import BlockRunner
        self.wl, self.dev, self.heads = wl, dev, heads
        self.n = 9                                   # embedding + 8 completed blocks
        T, d, S, ch = wl.T, wl.d, wl.S, wl.chunk
        self.nchunks = T // ch
        assert self.nchunks * ch == T
        self.reps = torch.empty((self.n + 1, T, d), dtype=torch.bfloat16, device=dev)
        for j in range(self.n):
            I.fill_block_rep(self.reps[j], j, wl.seed)
        self.reps[self.n].zero_()                    # slot 9 receives the closed block
        self.vbuf = I.make_outputs(wl, 1, S, dev, T=ch)   # stand-ins for f_i, shared by chunks
        self.P = I.block_params(wl, dev)
        self.U = torch.empty_like(self.P.W)
        self.U_split = torch.empty((2 * S, d), dtype=torch.bfloat16, device=dev)
        self.uf = torch.empty((1, d), device=dev)
        self.out = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
        self.timer = timer
        self.runner = BlockRunner(ch, d, S, torch.bfloat16, dev, timer=timer, heads=heads)
        self._prep = attnres_query_prep

    def chunk_views(self, c):
        sl = slice(c * self.wl.chunk, (c + 1) * self.wl.chunk)
        return (self.reps[:self.n, sl], self.reps[self.n, sl], self.reps[:self.n + 1, sl],
                self.out[sl])

    def prep(self):
        from depth_wise_softmax_block_b300.schedule import _call
        _call(self.timer, "query_prep", self._prep, self.P.W, self.P.G_key, self.U, self.U_split)
        _call(self.timer, "query_prep", self._prep, self.P.w_final.view(1, -1),
              self.P.g_final.view(1, -1), self.uf)

    def sublayer(self, i, y):
        """Stand-in for the sublayer f_i: returns the synthetic output v_i."""
        return self.vbuf[i - 1]

    def run_chunk(self, c, on_call=None):
        from depth_wise_softmax_block_b300.schedule import final_aggregation
        reps_c, close_c, all_c, out_c = self.chunk_views(c)
        self.runner.run_block(reps_c, self.U, self.P.G_in, self.sublayer, close_c, self.wl.eps,
                              self.wl.eps, on_call=on_call, U_split=self.U_split)
        final_aggregation(all_c, self.uf[0], out_c, self.wl.eps, timer=self.timer,
                          heads=self.heads)

    def run(self):
        self.prep()
        for c in range(self.nchunks):
            self.run_chunk(c)

    # algorithmic bytes, per step, per kernel kind
    def bytes_per_launch(self):
        d, E, ch, S, n, H = self.wl.d, 2, self.wl.chunk, self.wl.S, self.n, self.heads
        return {
            "phase1": C.phase1_bytes(n, S, d, E, heads=H) * ch,
            "phase2_first": C.phase2_bytes(d, E, False, False) * ch,
            "phase2": C.phase2_bytes(d, E, True, False, heads=H) * ch,
            "phase2_fused": C.phase2_bytes(d, E, True, True, heads=H) * ch,
            "close": C.partial_update_bytes(d, E) * ch,
            "final": C.phase1_bytes(n + 1, 1, d, E, with_lse=False) * ch,
        }

    def launches_per_step(self):
        return 2 + self.nchunks * (1 + self.wl.S + 1 + 1)

    def step_bytes(self):
        per_tok = C.block_step_bytes(self.n, self.wl.S, self.wl.d, 2, self.n + 1,
                                     heads=self.heads).total
        return per_tok * self.wl.T


# --------------------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples (every 100 ms) of the SM clock and throttle reasons."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except FileNotFoundError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------------------------
def oracle_sample(wl: I.Workload, k: int, seed_offset: int = 0):
    """Host inputs of a k-token sample of the long-context block (CPU-generated)."""
    n, d, S = 9, wl.d, wl.S
    T = k
    reps = torch.empty((n, T, d), dtype=torch.bfloat16)
    for j in range(n):
        I.fill_block_rep(reps[j], j, wl.seed + 1000 + seed_offset)
    v = I.make_outputs(wl, 1, S, "cpu", T=T)
    P = I.block_params(wl, "cpu")
    f = lambda t: t.float().numpy().astype("float64")  # noqa: E731
    return (f(reps), f(v), f(P.W), f(P.G_key), f(P.G_in), f(P.w_final), f(P.g_final))


def time_oracle(wl: I.Workload, k: int, seed_offset: int = 0):
    """Run the fp64 oracle (as it stands) over a k-token sample of one block; seconds."""
    import oracle.attnres_oracle as O
    args = oracle_sample(wl, k, seed_offset)
    t0 = time.perf_counter()     # elementwise numpy and reductions only: one thread
    O.single_block(args[0], args[1], args[2], args[3], args[4], args[5], args[6], wl.eps,
                   wl.eps)
    return time.perf_counter() - t0


def _oracle_worker(wl, k, seed_offset, rounds, barrier, out):
    """One host core's share of the all-cores oracle timing (a spawned process): build the
    sample once, then for every round wait for all workers and time the oracle on it."""
    torch.set_num_threads(1)
    import oracle.attnres_oracle as O
    args = oracle_sample(wl, k, seed_offset)
    for r in range(rounds):
        barrier.wait(timeout=600)
        t0 = time.perf_counter()
        O.single_block(args[0], args[1], args[2], args[3], args[4], args[5], args[6], wl.eps,
                       wl.eps)
        out.put((r, k, time.perf_counter() - t0))


def time_oracle_all_cores(wl: I.Workload, k: int, procs: int, rounds: int = 1):
    """The oracle on every host core at once: ``procs`` spawned processes (spawn, so nothing
    is forked from a process that holds a CUDA context), each timing its own k-token sample
    after a common barrier, ``rounds`` times.  Returns one (tokens, seconds of the slowest
    worker) pair per round."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(procs)
    out = ctx.Queue()
    env_keep = {v: os.environ.get(v) for v in ("OMP_NUM_THREADS", "MKL_NUM_THREADS",
                                               "OPENBLAS_NUM_THREADS")}
    for v in env_keep:
        os.environ[v] = "1"
    try:
        ps = [ctx.Process(target=_oracle_worker,
                          args=(wl, k, 500 + i, rounds, barrier, out))
              for i in range(procs)]
        for p in ps:
            p.start()
        res, deadline = [], time.time() + 900 + 60 * rounds
        while len(res) < procs * rounds:
            try:
                res.append(out.get(timeout=1.0))
            except queue.Empty:
                failed = [p.exitcode for p in ps if p.exitcode not in (None, 0)]
                if failed or time.time() > deadline:
                    for p in ps:
                        p.terminate()
                    raise RuntimeError(f"all-cores oracle timing failed (exit codes {failed})")
        for p in ps:
            p.join()
    finally:
        for v, old in env_keep.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
    return [(sum(x[1] for x in res if x[0] == r), max(x[2] for x in res if x[0] == r))
            for r in range(rounds)]


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def host_memory_bytes() -> int:
    try:
        return os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError, AttributeError):
        return 8 << 30


def oracle_procs(wl: I.Workload, k: int) -> int:
    """Host cores to time the oracle on, capped so that the workers' fp64 arrays (about three
    copies of a k-token sample of 9 sources and 24 sublayer outputs each) fit in half of the
    free host memory."""
    per_worker = 3 * k * wl.d * 8 * (9 + 1 + wl.S)
    return max(1, min(host_cores(), host_memory_bytes() // 2 // per_worker))


def cpu_baseline_line(wl: I.Workload, k1: int, k_all: int):
    """cpu_baseline: the oracle on all host cores (the reported value) and on one core."""
    secs1 = time_oracle(wl, k1)
    cores = oracle_procs(wl, k_all)
    tok, secs = time_oracle_all_cores(wl, k_all, cores)[0]
    return {"value": tok / secs, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{k_all} tokens per core x {cores} cores (one process each) of one "
                      f"24-sublayer block over 9 sources + final aggregation, fp64 numpy; "
                      f"{secs:.1f} s for the slowest core",
            "single_core": {"value": k1 / secs1, "unit": "tokens/s", "cores": 1,
                            "sample": f"{k1} tokens, {secs1:.1f} s"}}


# --------------------------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reference_arm(args, world, rank):
    """The fp64 oracle on the host cores, on a bounded sample of the same workload."""
    if rank != 0:
        return None
    wl = I.LONGCTX_PREFILL_BF16
    k = args.ref_tokens
    cores = oracle_procs(wl, k)
    rounds = time_oracle_all_cores(wl, k, cores, args.warmup + args.steps)[args.warmup:]
    step = sum(r[1] for r in rounds) / len(rounds)      # seconds per step (slowest core)
    val = rounds[0][0] / step
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
        "n_gpus": getattr(args, "gpus", 1), "runs_on": "host cores (the oracle uses no GPU)",
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": wl.name, "tokens_per_step": k * cores, "d": wl.d, "sources": 9,
                   "S": wl.S},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{k} tokens per core x {cores} cores (one process each) "
                                   "of one 24-sublayer block over 9 sources + final "
                                   "aggregation, fp64 numpy, per step"},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    return line


def traffic_for(kernel: str, heads: int = 1):
    """dram bytes per launch from a committed ncu summary, if it matches the current source."""
    tag = "" if heads == 1 else f"_heads{heads}"
    p = os.path.join(ROOT, "profiles", f"dram_traffic_longctx{tag}_T4096.json")
    if not os.path.exists(p):
        return None
    j = json.load(open(p))
    e = j.get(kernel)
    if not e or e.get("src_hash") != kernel_hash(kernel):
        return None
    return e.get("bytes_per_launch")


# ncu metric units -> bytes or nanoseconds
_NCU_UNITS = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12,
              "ns": 1.0, "nsecond": 1.0, "us": 1e3, "usecond": 1e3, "ms": 1e6, "msecond": 1e6}


def import_traffic(csv_path: str, tokens: int, heads: int = 1, scale_to: int = 16384,
                   out_dir: str = ""):
    """Turn an ncu capture of the step at ``tokens`` tokens (one chunk; metrics
    dram__bytes_read.sum and dram__bytes_write.sum of this library's kernels, in launch order)
    into the per-kernel DRAM traffic that ``traffic_for`` reads: bytes per launch scaled to a
    ``scale_to``-token launch (traffic grows with the tokens), stamped with the hash of each
    kernel's source files.  The launches of a chunk come in the step's order: phase 1, the S
    phase-2 calls (the first, the one with the partial given, then the fused ones), the close,
    the final aggregation.  Values are converted from the unit ncu printed them in; the JSON
    goes to ``out_dir`` (default: profiles/)."""
    import csv
    import collections
    rows = list(csv.reader(open(csv_path)))
    hdr = None
    launches = collections.OrderedDict()
    for r in rows:
        if "Kernel Name" in r:
            hdr = r
            continue
        if hdr is None or len(r) != len(hdr):
            continue
        rec = dict(zip(hdr, r))
        lid = int(rec["ID"])
        e = launches.setdefault(lid, {"name": rec["Kernel Name"]})
        unit = rec.get("Metric Unit", "byte") or "byte"
        if unit not in _NCU_UNITS:
            raise ValueError(f"unknown ncu unit {unit!r} for {rec['Metric Name']}")
        e[rec["Metric Name"]] = float(rec["Metric Value"].replace(",", "")) * _NCU_UNITS[unit]
    step_kernels = ("phase1_tc_kernel", "phase1_kernel", "phase2_kernel", "phase2_heads_kernel",
                    "add_kernel", "full_ring_kernel", "full_hold_kernel", "full_kernel",
                    "full_heads_kernel")
    ours = [e for e in launches.values()  # a template's name is followed by '<', others by '('
            if any(k + "<" in e["name"] or k + "(" in e["name"] for k in step_kernels)]
    S = I.LONGCTX_PREFILL_BF16.S
    per_chunk = ["phase1"] + ["phase2_first", "phase2"] + ["phase2_fused"] * (S - 2) + ["close",
                                                                                      "final"]
    assert len(ours) % len(per_chunk) == 0, (len(ours), len(per_chunk))
    acc = collections.defaultdict(lambda: [0, 0.0, 0.0, 0.0, ""])
    for k, e in enumerate(ours):
        kind = per_chunk[k % len(per_chunk)]
        a = acc[kind]
        a[0] += 1
        a[1] += e.get("dram__bytes_read.sum", 0.0)
        a[2] += e.get("dram__bytes_write.sum", 0.0)
        a[3] += e.get("gpu__time_duration.sum", 0.0)
        a[4] = e["name"]
    tag = "" if heads == 1 else f"_heads{heads}"
    out_path = os.path.join(out_dir or os.path.join(ROOT, "profiles"),
                            f"dram_traffic_longctx{tag}_T{tokens}.json")
    out = {}
    for kind, (cnt, rd, wr, dur, name) in acc.items():
        files = KERNEL_SOURCES[kind if kind in ("phase1", "final") else "rowwise"]
        out[kind] = {"src_hash": kernel_hash(kind), "src_files": files, "kernel": name[:120],
                     "heads": heads, "captured_tokens": tokens, "scaled_to_tokens": scale_to,
                     "launches_captured": cnt, "read_bytes_captured": rd,
                     "write_bytes_captured": wr,
                     "bytes_per_launch": (rd + wr) / cnt * scale_to / tokens,
                     "ncu_duration_ns_captured": dur / cnt}
    with open(out_path, "w") as f:
        json.dump(out, f, indent=1)
    print(json.dumps({k: round(v["bytes_per_launch"] / 1e9, 4) for k, v in out.items()}))
    return 0


def run_e2e(step: LongContextStep, iters: int):
    """The same step through the public API from pinned HOST buffers: per step, copy the
    block-representation cache (slots 0..8), the sublayer stand-ins and the parameters to the
    device, run, and read the final output back."""
    wl = step.wl
    h_reps = torch.empty(step.reps[:step.n].shape, dtype=torch.bfloat16, pin_memory=True)
    h_v = torch.empty(step.vbuf.shape, dtype=torch.bfloat16, pin_memory=True)
    params = [step.P.W, step.P.G_key, step.P.G_in, step.P.w_final, step.P.g_final]
    h_params = [torch.empty(p.shape, dtype=p.dtype, pin_memory=True) for p in params]
    h_out = torch.empty(step.out.shape, dtype=torch.bfloat16, pin_memory=True)
    h_reps.copy_(step.reps[:step.n])
    h_v.copy_(step.vbuf)
    for h, p in zip(h_params, params):
        h.copy_(p)
    torch.cuda.synchronize()
    h2d = h_reps.numel() * 2 + h_v.numel() * 2 + sum(h.numel() * 4 for h in h_params)
    d2h = h_out.numel() * 2

    # Copies overlap the kernels: host-to-device on one stream, device-to-host on another,
    # the kernels on the current stream; events order each chunk's copies and compute.
    compute = torch.cuda.current_stream()
    up = torch.cuda.Stream()
    down = torch.cuda.Stream()

    def one():
        with torch.cuda.stream(up):
            for h, p in zip(h_params, params):
                p.copy_(h, non_blocking=True)
            step.vbuf.copy_(h_v, non_blocking=True)
        ch = wl.chunk
        for c in range(step.nchunks):
            sl = slice(c * ch, (c + 1) * ch)
            with torch.cuda.stream(up):
                for j in range(step.n):
                    step.reps[j, sl].copy_(h_reps[j, sl], non_blocking=True)
                landed = torch.cuda.Event()
                landed.record(up)
            compute.wait_event(landed)
            if c == 0:
                step.prep()
            step.run_chunk(c)
            done = torch.cuda.Event()
            done.record(compute)
            with torch.cuda.stream(down):
                down.wait_event(done)
                h_out[sl].copy_(step.out[sl], non_blocking=True)
        for s in (up, compute, down):
            s.synchronize()

    one()
    t0 = time.perf_counter()
    for _ in range(iters):
        one()
    el = (time.perf_counter() - t0) / iters
    return {"value": wl.T / el, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": el * 1e3, "h2d_gbs": h2d / el / 1e9}


def full_grouped_bytes(L: int, S: int, d: int, E: int) -> int:
    """Algorithmic bytes per token of a whole Full AttnRes depth by the grouped two-phase
    schedule: per group starting at layer l0 + 1 with Sg layers, phase 1 reads the l0 + 1
    history rows and writes Sg outputs o (+ 4 B of lse each); layer l0 + i reads o, its i - 1
    in-group rows, the lse, and writes y."""
    total = 0
    for l0 in range(0, L, S):
        Sg = min(S, L - l0)
        total += (l0 + 1 + Sg) * d * E + 4 * Sg
        for i in range(1, Sg + 1):
            total += (1 + (i - 1) + 1) * d * E + 4
    return total


def full_direct_bytes(L: int, d: int, E: int) -> int:
    """The same depth one layer at a time (the naive path): layer l reads l rows, writes y."""
    return sum((l + 1) * d * E for l in range(1, L + 1))


def run_full_grouped(args):
    """Full AttnRes interpolation workload (54 sublayers, 8192 tokens, d = 2048, bf16, every
    sublayer output its own source): one whole depth by the grouped two-phase schedule (groups
    of --group sublayers), timed against the direct path (one single-pass aggregation per
    layer over all its sources).  Prints one JSON line."""
    from depth_wise_softmax_block_b300 import build as B
    B.build()
    import depth_wise_softmax_block_b300 as ar
    from depth_wise_softmax_block_b300.schedule import FullGroupedRunner, KernelTimer
    dev = torch.device("cuda", 0)
    wl = I.FULL_INTERP_BF16
    T, d, L, S = wl.T, wl.d, wl.L, args.group
    hist = torch.empty((L + 1, T, d), dtype=torch.bfloat16, device=dev)
    hist[0].copy_(I.normal((T, d), 1.0, wl.seed, "v0", dev, torch.bfloat16))
    v = torch.stack([I.normal((T, d), 1.0 + wl.v_growth * l, wl.seed, f"v{l}", dev,
                              torch.bfloat16) for l in range(1, L + 1)])
    W = I.queries(L, d, wl.seed, "w", dev)
    U = torch.empty_like(W)
    Us = torch.empty((2 * L, d), dtype=torch.bfloat16, device=dev)
    ar.attnres_query_prep(W, None, U, Us)
    G_in = I.gains(L, d, 0.0, wl.seed, "gin", dev)
    ys = torch.empty((L, T, d), dtype=torch.bfloat16, device=dev)
    timer = KernelTimer()
    runner = FullGroupedRunner(T, d, S, torch.bfloat16, dev, timer=timer)

    def grouped():
        runner.run(hist, U, G_in, ys, lambda l, y: v[l - 1], wl.eps, wl.eps, U_split=Us)

    def direct():
        for l in range(1, L + 1):
            ar.attnres_full_reference_path([hist[j] for j in range(l)], U[l - 1], G_in[l - 1],
                                           y_out=ys[l - 1], eps_key=wl.eps, eps_in=wl.eps)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        timer.clear()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    ms_g_eager = timed(grouped)
    kern = {k: {"launches_per_step": c // args.steps, "avg_ms": t / c}
            for k, (t, c) in timer.totals_ms().items()}
    runner.timer = None
    ms_d_eager = timed(direct)

    def graphed(fn):
        """The same calls captured once as a CUDA graph and replayed (the library launches on the
        caller's stream and allocates nothing); None if the capture fails."""
        try:
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                fn()
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            with torch.cuda.graph(g):
                fn()
            return timed(g.replay)
        except Exception:  # noqa: BLE001 - the eager time stands
            return None

    ms_g_graph, ms_d_graph = graphed(grouped), graphed(direct)
    ms_g = min(x for x in (ms_g_eager, ms_g_graph) if x is not None)
    ms_d = min(x for x in (ms_d_eager, ms_d_graph) if x is not None)
    bg, bd = full_grouped_bytes(L, S, d, 2) * T, full_direct_bytes(L, d, 2) * T
    peak, kind = peaks()
    line = {
        "metric": "Full AttnRes whole-depth tokens/s and achieved HBM GB/s, grouped two-phase "
                  "vs direct, 1 GPU",
        "value": T / (ms_g / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_g, "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name + f"_grouped_S{S}", "tokens": T, "d": d, "layers": L,
                   "group": S},
        "launch": {"grouped": "cuda_graph" if ms_g == ms_g_graph else "eager",
                   "direct": "cuda_graph" if ms_d == ms_d_graph else "eager",
                   "eager_ms": {"grouped": ms_g_eager, "direct": ms_d_eager},
                   "graph_ms": {"grouped": ms_g_graph, "direct": ms_d_graph}},
        "grouped": {"ms": ms_g, "bytes": bg, "achieved_gbs": bg / (ms_g / 1e3) / 1e9,
                    "frac_of_peak": bg / (ms_g / 1e3) / 1e9 / peak,
                    "d_elements_per_layer": bg / T / L / d / 2, "kernels": kern},
        "direct": {"ms": ms_d, "bytes": bd, "achieved_gbs": bd / (ms_d / 1e3) / 1e9,
                   "d_elements_per_layer": bd / T / L / d / 2},
        "speedup_grouped_over_direct": ms_d / ms_g, "peak_gbs": peak, "peak_source": kind,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_backward(args):
    """Backward of one sublayer's aggregation at the long-context shape: 16384 tokens,
    d = 7168, bf16, 10 sources (the embedding, 8 completed blocks and a partial sum).  Prints
    one JSON line: tokens/s and algorithmic GB/s ((2 n + 1) rows of d per token: the sources and
    g_y read, the source gradients written)."""
    from depth_wise_softmax_block_b300 import build as B
    B.build()
    import depth_wise_softmax_block_b300 as ar
    dev = torch.device("cuda", 0)
    T, d, n = 16384, 7168, 10
    srcs = [I.normal((T, d), 1.0 + 0.1 * j, 9, f"v{j}", dev, torch.bfloat16) for j in range(n)]
    U = (I.queries(1, d, 9, "w", dev)[0] * 3.0).contiguous()
    Gi = I.gains(1, d, 0.02, 9, "gi", dev)[0]
    gy = I.normal((T, d), 1.0, 9, "gy", dev, torch.bfloat16)
    dsrcs = [torch.empty_like(s) for s in srcs]
    du = torch.zeros((d,), device=dev)
    dgi = torch.zeros((d,), device=dev)

    def step():
        ar.attnres_backward(srcs, U, Gi, gy, dsrcs, du, dgi)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    byt = (2 * n + 1) * d * 2 * T
    peak, kind = peaks()
    line = {"metric": "AttnRes aggregation backward tokens/s and achieved HBM GB/s, 1 GPU",
            "value": T / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"backward_bf16_T{T}_d{d}_n{n}", "tokens": T, "d": d,
                       "sources": n},
            "achieved_gbs": byt / (ms / 1e3) / 1e9, "frac_of_peak": byt / (ms / 1e3) / 1e9 / peak,
            "peak_gbs": peak, "peak_source": kind}
    print(json.dumps(line), flush=True)
    return 0


def run_backward_block(args):
    """Backward of one whole block at the long-context chunk shape: 16384 tokens, d = 7168,
    bf16, n = 9 completed sources (the embedding and 8 blocks), S = 24 sublayers
    (attnres_backward_block: phase 1 recomputed for the 24 queries, the merge backward per
    token, then the sources' and parameters' gradients).  Next to it, in the same run, the same
    block by the per-sublayer backward (attnres_backward once per sublayer over its explicit
    sources: the 9 completed ones and, from the second sublayer on, the partial sum).  Prints one
    JSON line: tokens/s of the block backward and its achieved GB/s against the algorithmic
    bytes (read the sources, v_1 .. v_{S-1} and the S upstream gradients; write the sources' and
    the v's gradients)."""
    from depth_wise_softmax_block_b300 import build as B
    B.build()
    import depth_wise_softmax_block_b300 as ar
    dev = torch.device("cuda", 0)
    T, d, n, S = args.tokens or 16384, 7168, 9, 24
    dt = torch.bfloat16
    reps = torch.empty((n, T, d), dtype=dt, device=dev)
    for j in range(n):
        I.fill_block_rep(reps[j], j, 11)
    v = torch.stack([I.normal((T, d), 1.0, 11, f"v{k}", dev, dt) for k in range(S - 1)])
    W = I.queries(S, d, 11, "w", dev)
    Gk = I.gains(S, d, 0.02, 11, "gk", dev)
    Gi = I.gains(S, d, 0.02, 11, "gi", dev)
    U = torch.empty_like(W)
    Us = torch.empty((2 * S, d), dtype=dt, device=dev)
    ar.attnres_query_prep(W, Gk, U, Us)
    gy = torch.stack([I.normal((T, d), 1.0, 11, f"gy{i}", dev, dt) for i in range(S)])
    d_reps = torch.empty_like(reps)
    d_v = torch.empty_like(v)
    du = torch.zeros((S, d), device=dev)
    dgi = torch.zeros((S, d), device=dev)
    ws = torch.empty((ar.attnres_backward_block_workspace_size(n, S, T, d, dt),),
                     dtype=torch.uint8, device=dev)

    def block():
        ar.attnres_backward_block(reps, v, U, Gi, gy, d_reps, d_v, du, dgi, u_split=Us,
                                  workspace=ws)

    part = v[0].clone()             # stands in for the partial sum of every sublayer
    dsrcs = [torch.empty((T, d), dtype=dt, device=dev) for _ in range(n + 1)]

    def per_sublayer():
        for i in range(1, S + 1):
            srcs = [reps[j] for j in range(n)] + ([part] if i >= 2 else [])
            ar.attnres_backward(srcs, U[i - 1], Gi[i - 1], gy[i - 1], dsrcs[:len(srcs)],
                                du[i - 1], dgi[i - 1])

    def timed(fn, k):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(k):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / k

    with ClockSampler(0) as clk:
        ms = timed(block, args.steps)
    ms_sub = timed(per_sublayer, max(1, args.steps // 4))
    ar.attnres_poll_device_errors()
    byt = (2 * n + 3 * S - 2) * d * 2 * T
    ws_bytes = ws.numel()
    sub_bytes = sum((2 * (n + (1 if i >= 2 else 0)) + 1) * d * 2 * T for i in range(1, S + 1))
    peak, kind = peaks()
    line = {"metric": "AttnRes block backward (24 sublayers over 9 sources) tokens/s and "
                      "achieved HBM GB/s, 1 GPU",
            "value": T / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"backward_block_bf16_T{T}_d{d}_n{n}_S{S}", "tokens": T,
                       "d": d, "sources": n, "sublayers": S,
                       "l2": "no flush: every launch streams more than the 126 MB L2"},
            "algorithmic_bytes": byt, "achieved_gbs": byt / (ms / 1e3) / 1e9,
            "frac_of_peak": byt / (ms / 1e3) / 1e9 / peak, "peak_gbs": peak,
            "peak_source": kind, "workspace_bytes": ws_bytes,
            "per_sublayer_backward": {"ms": ms_sub, "algorithmic_bytes": sub_bytes,
                                      "achieved_gbs": sub_bytes / (ms_sub / 1e3) / 1e9},
            "speedup_over_per_sublayer": ms_sub / ms,
            "gpu_launches": 4 * args.steps, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)
    return 0


def walk_bytes(wl: I.Workload) -> int:
    """Algorithmic bytes of one Block AttnRes depth walk: every block's phase 1 over the
    sources before it, its phase-2 calls and close, then the final aggregation."""
    d, T, S, L = wl.d, wl.T, wl.S, wl.L
    E = 4 if wl.dtype == "f32" else 2
    total = 0
    for n in range(1, wl.n_blocks + 1):
        Sn = min(S, L - (n - 1) * S)
        b = C.block_step_bytes(n, Sn, d, E, 0)
        total += b.phase1 + b.phase2 + b.close
    total += C.phase1_bytes(wl.n_blocks + 1, 1, d, E, with_lse=False)
    return total * T


def run_block_walk(args, wl: I.Workload):
    """A whole Block AttnRes depth walk of one workload: every block's phase 1 (tensor-core
    logits for bf16), its phase-2 calls with the fused partial update and input RMSNorm, the
    block close into the next source slot, then the final aggregation.  Timed eager (each call
    launched from Python through the C ABI) and as one CUDA graph of the same calls, captured
    once and replayed.  Prints one JSON line; ``value`` is tokens/s of the faster launch mode."""
    from depth_wise_softmax_block_b300 import attnres_poll_device_errors, attnres_query_prep
    from depth_wise_softmax_block_b300 import build as B
    from depth_wise_softmax_block_b300.schedule import BlockRunner, KernelTimer, final_aggregation
    B.build()
    dev = torch.device("cuda", 0)
    T, d, S, L, N = wl.T, wl.d, wl.S, wl.L, wl.n_blocks
    bf16 = wl.dtype == "bf16"
    reps = I.make_reps(wl, N + 1, dev)           # slot 0 = b_0; slot n receives block n
    P = I.block_params(wl, dev)
    U = torch.empty_like(P.W)
    Us = torch.empty((2 * L, d), dtype=torch.bfloat16, device=dev) if bf16 else None
    uf = torch.empty((1, d), device=dev)
    attnres_query_prep(P.W, P.G_key, U, Us)
    attnres_query_prep(P.w_final.view(1, -1), P.g_final.view(1, -1), uf)
    vbuf = I.make_outputs(wl, 1, S, dev)        # stand-ins for f_i, shared by the blocks
    runner = BlockRunner(T, d, S, wl.torch_dtype, dev)
    fin = torch.empty((T, d), dtype=wl.torch_dtype, device=dev)
    timer = None

    def walk():
        for n in range(1, N + 1):
            l0 = (n - 1) * S
            Sn = min(S, L - l0)
            runner.run_block(reps[:n], U[l0:l0 + Sn], P.G_in[l0:l0 + Sn],
                             lambda i, y: vbuf[i - 1], reps[n], wl.eps, wl.eps,
                             U_split=None if Us is None else Us[2 * l0:2 * (l0 + Sn)])
        final_aggregation(reps[:N + 1], uf[0], fin, wl.eps, timer=timer)

    def timed(fn, k):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(k):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / k

    for _ in range(args.warmup):
        walk()
    torch.cuda.synchronize()
    eager_ms = timed(walk, args.steps)
    # per-kernel device times: one more eager walk with CUDA events around every launch
    timer = KernelTimer()
    runner.timer = timer
    walk()
    torch.cuda.synchronize()
    per_kernel = {k: {"launches": c, "total_us": t * 1e3, "avg_us": t * 1e3 / c}
                  for k, (t, c) in timer.totals_ms().items()}
    runner.timer = None
    timer = None
    graph_ms, graph_err = None, None
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            walk()                                # warm the side stream before capture
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            walk()
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        graph_ms = timed(g.replay, args.steps)
    except Exception as e:  # noqa: BLE001 - reported in the JSON line
        graph_err = f"{type(e).__name__}: {e}"
    attnres_poll_device_errors()
    byt = walk_bytes(wl)
    E = 4 if wl.dtype == "f32" else 2
    launches = 2 * N + L + 1 - sum(1 for n in range(1, N + 1) if min(S, L - (n - 1) * S) == 1)
    peak, kind = peaks()
    best = eager_ms if graph_ms is None else min(eager_ms, graph_ms)
    n_last = N                                   # sources of the last block's phase 1
    line = {"metric": f"Block AttnRes whole-depth walk ({L} sublayers, {T} tokens): tokens/s "
                      "and achieved HBM GB/s, 1 GPU",
            "value": T / (best / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": best, "higher_is_better": True,
            "dtype": wl.dtype, "data": "synthetic",
            "config": {"workload": wl.name, "tokens": T, "d": d, "sublayers": L, "S": S,
                       "blocks": N, "launch": "cuda_graph" if best == graph_ms else "eager",
                       "l2": "no flush" if byt / L < 126e6 else
                             "no flush: launches stream more than the 126 MB L2"},
            "eager_ms": eager_ms, "graph_ms": graph_ms,
            "us_per_sublayer": {"eager": eager_ms * 1e3 / L,
                                "graph": None if graph_ms is None else graph_ms * 1e3 / L},
            "bytes_per_step": byt, "achieved_gbs": byt / (best / 1e3) / 1e9,
            "frac_of_peak": byt / (best / 1e3) / 1e9 / peak, "peak_gbs": peak,
            "peak_source": kind, "gpu_launches": launches * args.steps,
            "d_elements_per_sublayer": byt / T / L / d / E,
            "pages_formula_d_elements": {"(N/S + 5) d, last block": n_last / S + 5},
            "kernels_eager_one_walk": per_kernel}
    if graph_err:
        line["graph_error"] = graph_err
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=2)
    ap.add_argument("--cpu-tokens", type=int, default=512,
                    help="oracle sample for the one-core cpu_baseline (about 10 s)")
    ap.add_argument("--cpu-tokens-per-core", type=int, default=256,
                    help="oracle sample per core for the all-cores cpu_baseline")
    ap.add_argument("--ref-tokens", type=int, default=32,
                    help="oracle sample per core and step of the reference arm (about 2 s)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the token count (profiling a smaller case)")
    ap.add_argument("--chunk", type=int, default=0, help="override the chunk size")
    ap.add_argument("--workload", default="longctx",
                    choices=["longctx", "full_grouped", "backward", "backward_block", "decode",
                             "prefill_chunk", "tiny"],
                    help="full_grouped: the Full AttnRes depth, grouped two-phase vs direct; "
                         "backward: one sublayer's aggregation backward; decode, "
                         "prefill_chunk, tiny: the whole Block AttnRes depth walk of the "
                         "256-token decode, 16384-token prefill-chunk or tiny fp32 workload, "
                         "eager and as a CUDA graph")
    ap.add_argument("--group", type=int, default=8, help="group size of --workload full_grouped")
    ap.add_argument("--heads", type=int, default=1,
                    help="depth-attention heads of the longctx step (Table 4 multi-head: 16)")
    ap.add_argument("--import-traffic", default="",
                    help="write profiles/dram_traffic_longctx_T<tokens>.json from an ncu CSV of "
                         "dram__bytes_read.sum / dram__bytes_write.sum of the step at --tokens")
    args = ap.parse_args(argv)
    if args.import_traffic:
        return import_traffic(args.import_traffic, args.tokens or 4096, args.heads)
    world, rank, local = dist_setup()

    if args.workload == "full_grouped" and args.impl == "ours":
        return run_full_grouped(args)
    if args.workload == "backward" and args.impl == "ours":
        return run_backward(args)
    if args.workload == "backward_block" and args.impl == "ours":
        return run_backward_block(args)
    walks = {"decode": I.DECODE_BF16, "prefill_chunk": I.PREFILL_CHUNK_BF16,
             "tiny": I.TINY_BLOCK_F32}
    if args.workload in walks and args.impl == "ours":
        return run_block_walk(args, walks[args.workload])
    if args.impl == "reference":
        line = reference_arm(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0

    assert torch.cuda.is_available(), "the bench needs a CUDA device"
    assert world == args.gpus or world == 1, "--gpus must match the launcher's world size"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from depth_wise_softmax_block_b300 import build as B
    from depth_wise_softmax_block_b300.schedule import KernelTimer
    B.build()
    wl = I.LONGCTX_PREFILL_BF16
    if args.tokens or args.chunk:
        import dataclasses
        T = args.tokens or wl.T
        ch = args.chunk or min(wl.chunk, T)
        wl = dataclasses.replace(wl, T=T, chunk=ch,
                                 name=f"longctx_prefill_bf16_T{T}_chunk{ch}_d7168_S24_n9")
    timer = KernelTimer()
    if args.heads != 1:
        import dataclasses
        wl = dataclasses.replace(wl, name=f"{wl.name}_heads{args.heads}")
    step = LongContextStep(wl, dev, timer=None, heads=args.heads)
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()

    def timed_steps():
        barrier(world)
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record()
        for _ in range(args.steps):
            step.run()
        end.record()
        torch.cuda.synchronize()
        barrier(world)
        return start.elapsed_time(end) / args.steps

    from depth_wise_softmax_block_b300 import attnres_poll_device_errors
    with ClockSampler(local) as clk:
        # The step as a caller runs it: nothing between the launches.
        ms = timed_steps()
        # The same number of steps again with an event pair around every launch, for the
        # per-kernel durations.  An event between two launches keeps the second from being
        # scheduled early (programmatic dependent launch), so this pass runs a little slower.
        step.timer = step.runner.timer = timer
        step.run()
        torch.cuda.synchronize()
        timer.clear()
        ms_events = timed_steps()
    attnres_poll_device_errors()      # raises if a kernel's bounded wait gave up
    ms = reduce_max(ms, world)
    tokens = wl.T * world
    value = tokens / (ms / 1e3)

    # per-kernel live durations (events on the launching stream, inside the second timed pass)
    tot = timer.totals_ms()
    bpl = step.bytes_per_launch()
    per_kernel = {}
    for k, (t_ms, cnt) in tot.items():
        avg = t_ms / cnt
        e = {"launches_per_step": cnt // args.steps, "avg_ms": avg,
             "share_of_step": t_ms / args.steps / ms_events}
        if k in bpl:
            e["achieved_gbs"] = bpl[k] / (avg / 1e3) / 1e9
        per_kernel[k] = e
    dom = max((k for k in per_kernel if k in bpl), key=lambda k: tot[k][0])
    peak, peak_kind = peaks()
    ach = per_kernel[dom]["achieved_gbs"]
    step_gbs = step.step_bytes() / (ms / 1e3) / 1e9

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": wl.name, "tokens": wl.T, "chunk": wl.chunk, "d": wl.d,
                   "sources": step.n, "S": wl.S, "heads": args.heads, "accumulate": "f32",
                   "l2": "no flush: every launch streams >= 235 MB (> 126 MB L2)",
                   "parallelism": f"replicas x{world} (tokens independent)"},
        "achieved_gbs_step": step_gbs, "frac_of_peak_step": step_gbs / peak,
        "ms_per_step_with_kernel_events": ms_events,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": peak,
                     "peak_source": peak_kind, "unit": "GB/s", "frac": ach / peak,
                     "traffic": traffic_for(dom, args.heads)},
        "kernels": per_kernel,
        "gpu_launches": step.launches_per_step() * args.steps,
        "clocks": clk.summary(),
    }
    del timer
    step.timer = None
    step.runner.timer = None
    if not args.no_e2e and rank == 0:
        line["e2e"] = run_e2e(step, args.e2e_steps)
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline_line(wl, args.cpu_tokens, args.cpu_tokens_per_core)
        print(json.dumps(line), flush=True)
    barrier(world)
    return 0


if __name__ == "__main__":
    sys.exit(main())
