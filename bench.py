#!/usr/bin/env python3
"""Benchmark of one continuous-batching attention step over a paged KV cache on GB300.

A step is the whole hot path over one batch: pa_cache_append of the step's new tokens through
the slot mapping, then pa_attention of every query token over its sequence's paged K/V.  The
headline workload is the 7B-class MHA decode step (32 heads x 128, block 16, 64 sequences
with contexts uniform in [512, 4096], bf16 K/V); by default every named workload (1-6) is also
timed the same way and reported under `per_config`, and --config C times workload C alone.

Prints one JSON line.  `value` is achieved HBM GB/s of the step (algorithmic bytes: every unique
K/V block touched once, q read, out written, metadata, plus the append's reads and writes,
divided by the device time of the step); attended tokens/s is reported beside it.  Inputs are
resident in HBM and larger than L2.  The timed steps are replays of one CUDA graph capturing the
step's library calls (every kernel runs every replay; the eager per-step time is reported
beside it as `eager_ms_per_step`).  `e2e` is the same metric through the public API with the
step's inputs copied from pinned host memory and the output copied back inside the timed
region.  `roofline` reports the main attention kernel alone, timed with CUDA events recorded
around it by the library.  `cpu_baseline` times the fp64 oracle on bounded samples of the
workload, on every host core (one process each) and on one core.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl ours|reference]

With N > 1 (launched by torchrun) every rank runs an independent replica of the workload on
its own GPU; there is no collective on the data path ("replicas only").
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-attn step: achieved HBM GB/s (% of peak), attended tokens/s"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=0, choices=[0, 1, 2, 3, 4, 5, 6],
                    help="one named workload only (0: the 7B-class MHA decode headline plus "
                         "every named workload under per_config)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seqs", type=int, default=0,
                    help="keep only the first N sequences of the workload (small profiling "
                         "cases; 0 = all)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the workload's runs that go to the tensor-core prefill "
                         "tiles (with --config)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="budget of the oracle CPU-baseline sample")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def max_over_ranks(x: float, dist, device) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------------------------
# peaks, clocks
# ---------------------------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured", j
    except Exception:
        return FALLBACK_HBM_GBS, "fallback", {}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "", 1).isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------------------------
# the workload on the device
# ---------------------------------------------------------------------------------------------
class DeviceWorkload:
    """Pools filled with the workload's prior context, plus the step's inputs, on one GPU."""

    def __init__(self, w, device):
        import torch
        import paged_kv_cache_286_gb300 as pa
        self.pa, self.torch, self.w, self.device = pa, torch, w, device

        def dev(bits):
            bits = np.ascontiguousarray(bits)
            t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16) \
                if bits.dtype == np.uint16 else torch.from_numpy(bits)
            return t.to(device)

        # The step's inputs packed into one pinned host buffer and one device buffer (256-byte
        # aligned pieces), so that the end-to-end leg moves them with a single copy each way.
        arrays = {
            "q": (w.q_bits, torch.bfloat16), "k": (w.k_new_bits, torch.bfloat16),
            "v": (w.v_new_bits, torch.bfloat16), "slots": (w.slot_mapping, torch.int64),
            "tables": (w.block_tables, torch.int32), "ctx": (w.context_lens, torch.int32),
            "qsl": (w.query_start_loc, torch.int32),
        }
        layout, off = {}, 0
        for name, (a, _) in arrays.items():
            a = np.ascontiguousarray(a)
            layout[name] = (off, a.nbytes, a.shape)
            off += (a.nbytes + 255) // 256 * 256
        self.host_buf = torch.zeros(off, dtype=torch.uint8).pin_memory()
        hb = self.host_buf.numpy()
        for name, (a, _) in arrays.items():
            o, n, _shape = layout[name]
            hb[o:o + n] = np.frombuffer(np.ascontiguousarray(a).tobytes(), dtype=np.uint8)
        self.dev_buf = self.host_buf.to(device)

        def views(buf):
            return {name: buf[o:o + n].view(arrays[name][1]).view(shape)
                    for name, (o, n, shape) in layout.items()}

        self.host = views(self.host_buf)
        self.dev = views(self.dev_buf)
        # a second set for the pipelined end-to-end leg (step i+1's inputs arrive while step i
        # computes; step i's output is read back while step i+1 computes)
        self.dev_buf2 = torch.empty_like(self.dev_buf)
        self.dev2 = views(self.dev_buf2)
        fp8 = w.cache_dtype == "fp8_e4m3"
        self.k_cache = torch.zeros(w.pool_shape, dtype=torch.uint8 if fp8 else torch.bfloat16,
                                   device=device)
        self.v_cache = torch.zeros_like(self.k_cache)
        self.out = torch.empty((w.num_tokens, w.num_q_heads, w.head_dim), dtype=torch.float32,
                               device=device)
        self.out_host = torch.empty(self.out.shape, dtype=torch.float32).pin_memory()
        self.out2 = torch.empty_like(self.out)
        self.out_host2 = torch.empty(self.out.shape, dtype=torch.float32).pin_memory()
        self.copy_stream = torch.cuda.Stream(device)
        nbytes = pa.attention_workspace_size(w.num_seqs, w.num_tokens, w.num_q_heads,
                                             w.num_kv_heads, w.head_dim, w.max_context_len,
                                             w.max_query_len)
        self.ws = pa.new_workspace(nbytes, device)
        P = w.slot_prior.shape[0]
        for a in range(0, P, 1 << 16):   # set-up: the context cached before the step
            b = min(P, a + (1 << 16))
            pa.cache_append(dev(w.k_prior_bits[a:b]), dev(w.v_prior_bits[a:b]),
                            torch.from_numpy(w.slot_prior[a:b]).to(device), self.k_cache,
                            self.v_cache, self.ws, k_scale=w.k_scale, v_scale=w.v_scale)
        torch.cuda.synchronize(device)
        self.h2d_bytes = self.host_buf.numel()       # the packed inputs, padding included
        self.d2h_bytes = self.out.numel() * self.out.element_size()

    def step(self, t=None, out=None):
        """pa_cache_append + pa_attention on tensors `t` (device copies by default)."""
        t = self.dev if t is None else t
        out = self.out if out is None else out
        w, pa = self.w, self.pa
        pa.cache_append(t["k"], t["v"], t["slots"], self.k_cache, self.v_cache, self.ws,
                        k_scale=w.k_scale, v_scale=w.v_scale)
        pa.attention(t["q"], self.k_cache, self.v_cache, t["tables"], t["ctx"], t["qsl"],
                     self.ws, scale=w.scale, max_context_len=w.max_context_len,
                     max_query_len=w.max_query_len, out=out, k_scale=w.k_scale,
                     v_scale=w.v_scale)

    def steps_from_host(self, n: int, stream) -> None:
        """n steps as a serving loop with inputs in host memory runs them: every step's packed
        inputs go host-to-device in one copy and its output comes back device-to-host, on a
        copy stream, double-buffered so that step i+1's inputs and step i's output move while
        a step computes on `stream`.  Enqueues everything; `stream` ends after the last
        read-back."""
        torch = self.torch
        copy = self.copy_stream
        bufs = [(self.dev_buf, self.dev), (self.dev_buf2, self.dev2)]
        outs = [(self.out, self.out_host), (self.out2, self.out_host2)]
        ready = [torch.cuda.Event() for _ in range(n)]
        free = [torch.cuda.Event() for _ in range(n)]

        def h2d(i):
            with torch.cuda.stream(copy):
                if i >= 2:
                    copy.wait_event(free[i - 2])      # step i-2 is done with this buffer
                bufs[i % 2][0].copy_(self.host_buf, non_blocking=True)
                ready[i].record(copy)

        copy.wait_stream(stream)
        h2d(0)
        for i in range(n):
            if i + 1 < n:
                h2d(i + 1)
            stream.wait_event(ready[i])
            out, out_host = outs[i % 2]
            self.step(bufs[i % 2][1], out)
            free[i].record(stream)
            with torch.cuda.stream(copy):
                copy.wait_event(free[i])
                out_host.copy_(out, non_blocking=True)
        stream.wait_stream(copy)

    def has_prefill(self) -> bool:
        """Whether the step launches the tensor-core prefill-tile kernel: query runs of more than
        16 tokens or of more than 16 (token x head) rows, over a bf16 pool with head_dim 128 or
        64 or an E4M3 pool with head_dim 128, and a group that divides 128."""
        w = self.w
        g = w.num_q_heads // w.num_kv_heads
        built = ((w.cache_dtype == "bf16" and w.head_dim in (64, 128))
                 or (w.cache_dtype == "fp8_e4m3" and w.head_dim == 128))
        return ((w.max_query_len > 16 or w.max_query_len * g > 16) and built
                and g <= 8 and 128 % g == 0)

    def launches_per_step(self) -> int:
        """Our kernels one step launches: the append, the plan, the split-KV attention, the LSE
        merge when the workspace carries split partials, and the tensor-core prefill kernel
        when the step holds chunks it serves (has_prefill)."""
        w = self.w
        size = self.pa.attention_workspace_size(w.num_seqs, w.num_tokens, w.num_q_heads,
                                                w.num_kv_heads, w.head_dim, w.max_context_len,
                                                w.max_query_len)

        def up(x):
            return (x + 255) // 256 * 256
        # the header and the four per-sequence arrays: more means split partials
        no_partials = 256 + 3 * up(4 * (w.num_seqs + 1)) + up(4 * max(w.num_seqs, 1))
        return 3 + (1 if size > no_partials else 0) + (1 if self.has_prefill() else 0)


def prefill_flops(w) -> int:
    """Algorithmic flops of the prefill-tile kernel: every query of a run it serves (more than
    16 tokens, or more than 16 token x head rows) against the keys it attends, QK^T and PV at
    2 flops per multiply-add each."""
    total = 0
    g = w.num_q_heads // w.num_kv_heads
    for L, n in zip(w.context_lens.tolist(), w.query_lens.tolist()):
        if n > 16 or n * g > 16:
            total += n * (L - n) + n * (n + 1) // 2
    return 4 * w.head_dim * w.num_q_heads * total


def src_sha(files=None) -> str:
    """sha256 (first 16 hex digits) over names and contents of kernel source files under csrc/:
    the named ones in the given order, or all of them sorted by name."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_286_gb300", "csrc")
    for name in (files if files is not None else sorted(os.listdir(csrc))):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def decode_src_sha() -> str:
    """Hash of all kernel sources (the label the profile summaries carry)."""
    return src_sha()


def traffic_from_profiles(config_id: int):
    """DRAM bytes per launch of the step's dominant kernel from a committed ncu summary, if the
    source files that define that kernel (its entry's src_files) are unchanged since the
    counters were taken (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            j = json.load(f)
        e = j.get(f"cfg{config_id}")
        if e and e.get("src_sha") == src_sha(e.get("src_files")):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ---------------------------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and reference arm)
# ---------------------------------------------------------------------------------------------
def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part", "processor\t: arm")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def _sub_workload(config_id: int, first: int, k: int):
    """k sequences of a named workload (its length recipe, from sequence `first` on, wrapping
    around), drawn with a seed of their own: a bounded sample of the same workload."""
    from synthetic.workloads import config_lengths, make_workload
    ctx, ql, kw = config_lengths(config_id)
    S = len(ctx)
    idx = [(first + i) % S for i in range(k)]
    kw = dict(kw)
    kw.pop("num_blocks", None)
    return make_workload([ctx[i] for i in idx], [ql[i] for i in idx],
                         seed=1000 + config_id + 7919 * first,
                         name=f"cfg{config_id}-sample{first}+{k}", **kw)


_SHARDS = {}


def _shard_run(args):
    """In a spawned oracle worker: the oracle's whole step (set-up append, step append,
    attention) on shard `shard` of k sequences; returns (seconds, bytes, attended tokens)."""
    config_id, shard, k = args
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    from oracle import run_step
    key = (config_id, shard, k)
    if key not in _SHARDS:
        _SHARDS.clear()
        _SHARDS[key] = _sub_workload(config_id, shard * k, k)
    w = _SHARDS[key]
    t0 = time.perf_counter()
    run_step(w)
    dt = time.perf_counter() - t0
    return dt, w.algorithmic_bytes() + w.append_bytes(), w.attended_tokens()


class OracleRunner:
    """The fp64 oracle, as it stands, on `cores` host processes (spawned, one BLAS thread
    each); a step is one shard of k sequences per process, timed as the wall time of all."""

    def __init__(self, config_id: int, cores: int):
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        self.config_id, self.cores = config_id, cores
        self.pool = mp.get_context("spawn").Pool(cores)

    def close(self):
        self.pool.close()
        self.pool.join()

    def one_core(self, seconds: float):
        """Grow one process's shard until it takes >= seconds/4; (seconds, bytes, tokens, k)."""
        from synthetic.workloads import config_lengths
        S = len(config_lengths(self.config_id)[0])
        k = 1
        while True:
            dt, nbytes, toks = self.pool.apply(_shard_run, ((self.config_id, 0, k),))
            if dt >= seconds / 4 or k >= S:
                return dt, nbytes, toks, k
            k = min(S, max(k + 1, int(k * min(4.0, (seconds / 4) / max(dt, 1e-3)))))

    def step(self, k: int):
        """All processes at once, shard i each; returns (wall seconds, bytes, tokens)."""
        t0 = time.perf_counter()
        res = self.pool.map(_shard_run, [(self.config_id, i, k) for i in range(self.cores)],
                            chunksize=1)
        wall = time.perf_counter() - t0
        return wall, sum(r[1] for r in res), sum(r[2] for r in res)


def cpu_baseline(config_id: int, seconds: float):
    """One-core and all-core throughput of the oracle on bounded samples of the workload."""
    cores = host_cores()
    run = OracleRunner(config_id, cores)
    try:
        dt1, b1, t1, k = run.one_core(seconds)
        run.step(k)                       # every process builds its shard
        wall, nbytes, toks = run.step(k)
    finally:
        run.close()
    return {"value": nbytes / wall / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{cores} processes (one per host core, one BLAS thread each), each the "
                      f"fp64 oracle step (set-up append, step append, attention) on its own "
                      f"{k} sequences of the workload's recipe; wall time {wall:.1f} s",
            "tokens_per_s": toks / wall, "cpu": cpu_model(),
            "value_1core": b1 / dt1 / 1e9, "tokens_per_s_1core": t1 / dt1,
            "sample_1core": f"{k} sequences in one process, {dt1:.1f} s"}


def reference_sample_size(num_seqs: int, cores: int, budget_s: float, seq_s: float) -> int:
    """Sequences per process for one reference-arm step: as many as fit 0.8 of the step's
    budget at the contended per-sequence time, and no more than twice the workload's sequences
    over all processes (a larger sample only repeats its sequences and multiplies the memory
    every process builds); at least one."""
    return max(1, min(max(1, 2 * num_seqs // max(1, cores)), int(0.8 * budget_s / max(seq_s, 1e-3))))


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from synthetic.workloads import CONFIG_NAMES
    cores = host_cores()
    budget = 150.0 / max(1, args.steps + args.warmup)   # whole run within a few minutes
    run = OracleRunner(args.config, cores)
    try:
        # one sequence per process with every process busy (the per-sequence time under
        # contention, after a first pass that builds the shards), then as many sequences per
        # process as fit the step's budget, and no more than twice the workload's sequences
        # over all processes (a larger sample only repeats its sequences and multiplies the
        # memory every process builds)
        from synthetic.workloads import config_lengths
        S = len(config_lengths(args.config)[0])
        run.step(1)
        dt1 = run.step(1)[0]
        k = reference_sample_size(S, cores, budget, dt1)
        times, nbytes, toks = [], 0, 0
        for i in range(args.warmup + args.steps):
            wall, nb, tk = run.step(k)
            if i >= args.warmup:
                times.append(wall)
                nbytes, toks = nb, tk
    finally:
        run.close()
    total = sum(times)
    value = nbytes * len(times) / total / 1e9
    sample = (f"{cores} processes (one per host core), each the fp64 oracle step (set-up "
              f"append, step append, attention) on its own {k} sequences of the workload's "
              "recipe per step")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"cfg{args.config}: {CONFIG_NAMES[args.config]}",
                       "sample_seqs_per_core": k},
            "attended_tokens_per_s": toks * len(times) / total,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample, "cpu": cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------------
def workload_for(config_id: int, seqs: int = 0):
    from synthetic.workloads import config_lengths, make_config, make_workload
    if seqs:
        ctx, ql, kw = config_lengths(config_id)
        return make_workload(ctx[:seqs], ql[:seqs], seed=1000 + config_id,
                             name=f"cfg{config_id}-first{seqs}", **kw)
    return make_config(config_id)


def prefill_only(config_id: int):
    """The sequences of a named workload whose query runs go to the tensor-core tiles, alone
    (same lengths and recipe), or None when it has none."""
    from synthetic.workloads import config_lengths, make_workload
    ctx, ql, kw = config_lengths(config_id)
    g = kw["num_q_heads"] // kw["num_kv_heads"]
    if kw.get("cache_dtype", "bf16") != "bf16" or kw["head_dim"] != 128 or 128 % g:
        return None
    idx = [i for i, n in enumerate(ql) if n > 16 or n * g > 16]
    if not idx or len(idx) == len(ql):
        return None
    kw = dict(kw)
    kw.pop("num_blocks", None)
    return make_workload([ctx[i] for i in idx], [ql[i] for i in idx], seed=1000 + config_id,
                         name=f"cfg{config_id}-chunks", **kw)


def measure(w, args, device, dist, world, sample_clocks=True):
    """Times one workload's step: graph replays (value), eager steps with the library's kernel
    events (roofline, prefill), and the end-to-end serving loop.  Returns a dict."""
    import torch
    import paged_kv_cache_286_gb300 as pa
    dw = DeviceWorkload(w, device)
    algo_attn = w.algorithmic_bytes()
    algo_step = algo_attn + w.append_bytes()
    # the split-KV kernel's own bytes: chunks on the tensor-core prefill path are not its work
    g = w.num_q_heads // w.num_kv_heads
    decode_seqs = [s for s in range(w.num_seqs)
                   if not (dw.has_prefill() and (int(w.query_lens[s]) > 16
                                                 or int(w.query_lens[s]) * g > 16))]
    algo_decode = w.algorithmic_bytes(seqs=decode_seqs)
    prefill_seqs = [s for s in range(w.num_seqs) if s not in set(decode_seqs)]
    algo_prefill = w.algorithmic_bytes(seqs=prefill_seqs) if prefill_seqs else 0
    stream = torch.cuda.current_stream(device)

    # warm-up (also checks the device error word once)
    for _ in range(max(3, args.warmup)):
        dw.step()
    assert pa.check_error(dw.ws) == 0

    # The same step captured once as a CUDA graph: replaying it gives the device time of the
    # step without host-side launch gaps (every kernel of the step still runs every replay).
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        dw.step()
    torch.cuda.synchronize(device)
    with torch.cuda.graph(graph, stream=cap):
        dw.step()
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize(device)

    K = args.steps
    kb = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ka = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    pfb = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    pfa = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for e in kb + ka + pfb + pfa:   # create the events before handing them to the library
        e.record(stream)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(device.index) if sample_clocks else None
    torch.cuda.synchronize(device)
    barrier(dist, device)
    if clocks:
        clocks.start()
    # The sampler reads the clocks every 200 ms and the timed regions below last milliseconds:
    # replay the same step for about a second first, so that the samples are taken under this
    # load, which runs on into the timed regions without a pause.
    t_end = time.monotonic() + (1.0 if clocks else 0.1)
    while time.monotonic() < t_end:
        for _ in range(20):
            graph.replay()
        torch.cuda.synchronize(device)
    # (1) eager steps with the library's span hook: the global-timer start and end of the
    # split-KV and prefill-tile kernels as they run in the step (overlapping each other)
    spans = torch.tensor([-1, 0, -1, 0] * K, dtype=torch.int64, device=device)
    torch.cuda.synchronize(device)
    start.record(stream)
    for i in range(K):
        pa.set_kernel_span_buffer(spans[4 * i:4 * i + 4])
        dw.step()
    stop.record(stream)
    torch.cuda.synchronize(device)
    pa.set_kernel_span_buffer(None)
    sp = spans.view(K, 4).cpu().numpy().astype(np.uint64)
    # (2) eager steps with events around each of the two kernels: the events make each
    # kernel wait for the one before it, so these time every kernel alone
    for i in range(K):
        pa.set_kernel_timing_events(kb[i], ka[i])
        pa.set_prefill_timing_events(pfb[i], pfa[i])
        dw.step()
    torch.cuda.synchronize(device)
    pa.set_kernel_timing_events(None, None)
    pa.set_prefill_timing_events(None, None)
    # (2) graph replays: the timed steps of `value`
    barrier(dist, device)
    torch.cuda.synchronize(device)
    g0.record(stream)
    for _ in range(K):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize(device)
    barrier(dist, device)
    clk = clocks.stop() if clocks else None
    assert pa.check_error(dw.ws) == 0
    def span_ms(col):
        v = [float(sp[i, col + 1] - sp[i, col]) * 1e-6 for i in range(K)
             if sp[i, col] != np.uint64(2 ** 64 - 1) and sp[i, col + 1] >= sp[i, col]]
        return statistics.mean(v) if v else None

    kern_ms = span_ms(0) if decode_seqs else None
    kern_alone_ms = statistics.mean(kb[i].elapsed_time(ka[i]) for i in range(K)) \
        if decode_seqs else None
    pf_flops = prefill_flops(w) if dw.has_prefill() else 0
    pf_ms = span_ms(2) if pf_flops else None
    pf_alone_ms = statistics.mean(pfb[i].elapsed_time(pfa[i]) for i in range(K)) \
        if pf_flops else None
    step_ms = max_over_ranks(g0.elapsed_time(g1) / K, dist, device)
    eager_ms = max_over_ranks(start.elapsed_time(stop) / K, dist, device)

    # end to end: inputs from pinned host memory, output back, every step
    dw.steps_from_host(2, stream)
    torch.cuda.synchronize(device)
    barrier(dist, device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    dw.steps_from_host(K, stream)
    e1.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / K, dist, device)
    assert pa.check_error(dw.ws) == 0

    peak, peak_kind, peaks = load_peaks()
    value = world * algo_step / (step_ms * 1e-3) / 1e9
    r = {
        "workload": w.name, "dtype": "e4m3" if w.cache_dtype == "fp8_e4m3" else "bf16",
        "ms_per_step": step_ms, "value": value, "unit": UNIT,
        "hbm_frac_of_peak": value / world / peak, "eager_ms_per_step": eager_ms,
        "attended_tokens_per_s": world * w.attended_tokens() / (step_ms * 1e-3),
        "algorithmic_bytes_per_step": algo_step,
        "e2e": {"value": world * algo_step / (e2e_ms * 1e-3) / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": dw.h2d_bytes, "d2h_bytes_per_step": dw.d2h_bytes,
                "ms_per_step": e2e_ms},
        "gpu_launches_per_step": dw.launches_per_step(),
        "clocks": clk,
    }
    if decode_seqs:
        achieved = algo_decode / (kern_ms * 1e-3) / 1e9
        alone = algo_decode / (kern_alone_ms * 1e-3) / 1e9
        r["roofline"] = {"bound": "hbm", "kernel": "decode_kernel (split-KV paged attention)",
                         "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
                         "traffic": None, "algorithmic_bytes_per_launch": algo_decode,
                         "kernel_ms": kern_ms,
                         "timing": "span of the kernel in the step (first CTA start to last "
                                   "CTA end, device global timer)",
                         "kernel_ms_alone": kern_alone_ms, "achieved_alone": alone,
                         "frac_alone": alone / peak}
    if pf_flops:
        pf_peak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
        pf_tf = pf_flops / (pf_ms * 1e-3) / 1e12
        pf_tf_alone = pf_flops / (pf_alone_ms * 1e-3) / 1e12
        r["prefill"] = {
            "bound": "tensor", "kernel": "prefill tiles (tcgen05 causal tiles)",
            "achieved": pf_tf, "peak": pf_peak, "unit": "TFLOP/s", "frac": pf_tf / pf_peak,
            "peak_source": ("measured" if "bf16_tflops" in peaks else "fallback")
                           + " bf16_tflops (burst)",
            "flops_per_launch": pf_flops, "kernel_ms": pf_ms,
            "timing": "span of the kernel in the step (device global timer)",
            "kernel_ms_alone": pf_alone_ms, "achieved_alone": pf_tf_alone,
            "frac_alone": pf_tf_alone / pf_peak,
            "algorithmic_bytes_per_launch": algo_prefill,
            "achieved_gbs": algo_prefill / (pf_ms * 1e-3) / 1e9,
            "flops": "algorithmic: 4 * head_dim * q heads * attended keys of the chunk "
                     "queries (QK^T and PV); masked tile parts and the second (lo) half of P's "
                     "bf16 split are extra MMA work not counted"}
        if not decode_seqs:
            # every run of the step is on the tensor-core tiles (e.g. speculative verify with
            # GQA): that kernel is the dominant one, and it streams each K/V tile once
            pf_gbs = algo_prefill / (pf_ms * 1e-3) / 1e9
            r["roofline"] = {
                "bound": "hbm", "kernel": "prefill_kernel (tcgen05 causal tiles)",
                "achieved": pf_gbs, "peak": peak, "unit": "GB/s", "frac": pf_gbs / peak,
                "peak_source": f"{peak_kind} hbm_gbs", "traffic": None,
                "algorithmic_bytes_per_launch": algo_prefill, "kernel_ms": pf_ms}
    if pf_flops:
        # the plan's SM budget for the prefill tiles (workspace header word 3)
        r["prefill"]["ctas"] = int(dw.ws[12:16].cpu().view(torch.int32).item())
    del graph, dw
    torch.cuda.synchronize(device)
    torch.cuda.empty_cache()
    return r


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if args.gpus != world and world > 1:
        print(f"--gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist = dist_init(world, "nccl")
    from paged_kv_cache_286_gb300 import build
    if rank == 0:
        build.build()
    barrier(dist, device)
    from synthetic.workloads import CONFIG_NAMES

    headline = args.config if args.config else 2
    w = prefill_only(headline) if args.prefill_only else workload_for(headline, args.seqs)
    r = measure(w, args, device, dist, world)
    r["roofline"]["traffic"] = None if args.seqs else traffic_from_profiles(headline)
    per_config = None
    if not args.config and not args.seqs:
        # every named workload, one after the other, timed the same way
        per_config = {}
        for c in range(1, 7):
            rc = r if c == headline else measure(workload_for(c), args, device, dist, world)
            if "roofline" in rc:
                rc["roofline"]["traffic"] = traffic_from_profiles(c)
            if c == 1:
                rc["note"] = ("launch-bound: 0.15 MB of K/V per step, a few microseconds of "
                              "HBM time against the launch and plan latency of four kernels")
            per_config[f"cfg{c}"] = rc
        cfg4 = prefill_only(4)
        if cfg4 is not None:
            pr = measure(cfg4, args, device, dist, world, sample_clocks=False)
            per_config["cfg4"]["prefill_alone"] = dict(
                pr["prefill"], workload=cfg4.name, ms_per_step=pr["ms_per_step"],
                note="the two prompt chunks of the mixed step without its decodes: the "
                     "tensor-core kernel's own speed")
    result = None
    if rank == 0:
        cpu = None if args.no_cpu_baseline else cpu_baseline(headline, args.cpu_seconds)
        result = {
            "metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": r["dtype"], "data": "synthetic",
            "config": {"workload": f"cfg{headline}: {CONFIG_NAMES[headline]}"
                                   + (f" (first {args.seqs} sequences)" if args.seqs else ""),
                       "l2": f"no flush: each step streams "
                             f"{r['algorithmic_bytes_per_step'] / 1e9:.2f} GB of K/V and q/out, "
                             "far above the 129 MB L2",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "hbm_frac_of_peak": r["hbm_frac_of_peak"],
            "timing": "CUDA graph of one step, replayed K times between CUDA events",
            "eager_ms_per_step": r["eager_ms_per_step"],
            "attended_tokens_per_s": r["attended_tokens_per_s"],
            "algorithmic_bytes_per_step": r["algorithmic_bytes_per_step"],
            "e2e": dict(r["e2e"], copies="one packed host-to-device copy of each step's inputs "
                        "and one device-to-host copy of its output, on a copy stream, double-"
                        "buffered against the steps' compute"),
            "gpu_launches": args.steps * r["gpu_launches_per_step"],
            "roofline": r["roofline"],
            "cpu_baseline": cpu,
            "clocks": r["clocks"],
        }
        if "prefill" in r:
            result["prefill"] = r["prefill"]
        if per_config is not None:
            result["per_config"] = per_config
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        if not args.config:
            args.config = 2
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
