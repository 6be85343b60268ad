#!/usr/bin/env python3
"""Benchmark of one continuous-batching attention step over a paged KV cache on GB300.

A step is the whole hot path over one batch: pa_cache_append of the step's new tokens through
the slot mapping, then pa_attention of every query token over its sequence's paged K/V.  The
default workload is the 7B-class MHA decode step (32 heads x 128, block 16, 64 sequences with
contexts uniform in [512, 4096], bf16 K/V); --config picks another of the five named workloads.

Prints one JSON line.  `value` is achieved HBM GB/s of the step (algorithmic bytes: every unique
K/V block touched once, q read, out written, metadata, plus the append's reads and writes,
divided by the device time of the step); attended tokens/s is reported beside it.  Inputs are
resident in HBM and larger than L2.  The timed steps are replays of one CUDA graph capturing the
step's library calls (every kernel runs every replay; the eager per-step time is reported
beside it as `eager_ms_per_step`).  `e2e` is the same metric through the public API with the
step's inputs copied from pinned host memory and the output copied back inside the timed
region.  `roofline` reports the main attention kernel alone, timed with CUDA events recorded
around it by the library.  `cpu_baseline` times the fp64 oracle on a bounded sample.

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
    ap.add_argument("--config", type=int, default=2, choices=[1, 2, 3, 4, 5, 6])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seqs", type=int, default=0,
                    help="keep only the first N sequences of the workload (small profiling "
                         "cases; 0 = all)")
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
        16 tokens or of more than 16 (token x head) rows, over a bf16 pool with head_dim 128
        and a group that divides 128."""
        w = self.w
        g = w.num_q_heads // w.num_kv_heads
        return ((w.max_query_len > 16 or w.max_query_len * g > 16) and w.cache_dtype == "bf16"
                and w.head_dim == 128 and 128 % g == 0)

    def launches_per_step(self) -> int:
        """Our kernels one step launches: the append, the plan, the split-KV attention, the LSE
        merge when the workspace carries split partials, and the tensor-core prefill kernel
        when the step holds chunks of more than 16 queries over a bf16 pool with head_dim 128."""
        w = self.w
        size = self.pa.attention_workspace_size(w.num_seqs, w.num_tokens, w.num_q_heads,
                                                w.num_kv_heads, w.head_dim, w.max_context_len,
                                                w.max_query_len)
        no_partials = 256 + 2 * (((4 * (w.num_seqs + 1) + 255) // 256) * 256)
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
def _oracle_sample_worker(args):
    """Runs in a spawned process with one BLAS thread: the oracle's whole step (append of the
    prior context and the new tokens, then attention) on the first `k` sequences."""
    config_id, k = args
    sys.path.insert(0, ROOT)
    from oracle import run_step
    from synthetic.workloads import config_lengths, make_workload
    ctx, ql, kw = config_lengths(config_id)
    w = make_workload(ctx[:k], ql[:k], seed=1000 + config_id, name=f"cfg{config_id}-sample",
                      **kw)
    t0 = time.perf_counter()
    run_step(w)
    dt = time.perf_counter() - t0
    return dt, w.algorithmic_bytes() + w.append_bytes(), w.attended_tokens(), k


def oracle_sample(config_id: int, seconds: float):
    """Time the oracle on growing sub-batches of the workload until one takes >= `seconds`/4,
    then report the largest; returns dict(value GB/s, tokens/s, seqs, seconds)."""
    from synthetic.workloads import config_lengths
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    ctx, _, _ = config_lengths(config_id)
    S = len(ctx)
    ctxmp = mp.get_context("spawn")
    k, best = 1, None
    with ctxmp.Pool(1) as pool:
        while True:
            dt, nbytes, toks, k = pool.apply(_oracle_sample_worker, ((config_id, k),))
            best = (dt, nbytes, toks, k)
            if dt >= seconds / 4 or k >= S:
                break
            k = min(S, max(k + 1, int(k * min(4.0, (seconds / 4) / max(dt, 1e-3)))))
    dt, nbytes, toks, k = best
    return {"value": nbytes / dt / 1e9, "tokens_per_s": toks / dt, "seqs": k, "of_seqs": S,
            "seconds": dt}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from synthetic.workloads import CONFIG_NAMES, config_lengths
    ctx, _, _ = config_lengths(args.config)
    budget = 150.0 / max(1, args.steps + args.warmup)   # whole run within a few minutes
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    ctxmp = mp.get_context("spawn")
    with ctxmp.Pool(1) as pool:
        # size the per-step sample from a one-sequence calibration
        dt1, _, _, _ = pool.apply(_oracle_sample_worker, ((args.config, 1),))
        k = max(1, min(len(ctx), int(budget / max(dt1, 1e-3))))
        times, nbytes, toks = [], 0, 0
        for i in range(args.warmup + args.steps):
            dt, nb, tk, _ = pool.apply(_oracle_sample_worker, ((args.config, k),))
            if i >= args.warmup:
                times.append(dt)
                nbytes, toks = nb, tk
    total = sum(times)
    value = nbytes * len(times) / total / 1e9
    sample = (f"first {k} of {len(ctx)} sequences of the workload per step (same recipe), "
              "fp64 oracle: set-up append, step append and attention")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"cfg{args.config}: {CONFIG_NAMES[args.config]}",
                       "sample_seqs": k},
            "attended_tokens_per_s": toks * len(times) / total,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------------
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
    import paged_kv_cache_286_gb300 as pa
    from synthetic.workloads import CONFIG_NAMES, make_config

    if args.seqs:
        from synthetic.workloads import config_lengths, make_workload
        ctx, ql, kw = config_lengths(args.config)
        w = make_workload(ctx[:args.seqs], ql[:args.seqs], seed=1000 + args.config,
                          name=f"cfg{args.config}-first{args.seqs}", **kw)
    else:
        w = make_config(args.config)
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
    clocks = ClockSampler(local)
    torch.cuda.synchronize(device)
    barrier(dist, device)
    clocks.start()
    # The sampler reads the clocks every 200 ms and the timed regions below last milliseconds:
    # replay the same step for about a second first, so that the samples are taken under this
    # load, which runs on into the timed regions without a pause.
    t_end = time.monotonic() + 1.0
    while time.monotonic() < t_end:
        for _ in range(20):
            graph.replay()
        torch.cuda.synchronize(device)
    # (1) eager steps, with the main attention kernel bracketed by events for the roofline
    torch.cuda.synchronize(device)
    start.record(stream)
    for i in range(K):
        pa.set_kernel_timing_events(kb[i], ka[i])
        pa.set_prefill_timing_events(pfb[i], pfa[i])
        dw.step()
    stop.record(stream)
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
    clk = clocks.stop()
    assert pa.check_error(dw.ws) == 0
    kern_ms = statistics.mean(kb[i].elapsed_time(ka[i]) for i in range(K))
    pf_flops = prefill_flops(w) if dw.has_prefill() else 0
    pf_ms = statistics.mean(pfb[i].elapsed_time(pfa[i]) for i in range(K)) if pf_flops else None
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

    peak, peak_kind, _ = load_peaks()
    value = world * algo_step / (step_ms * 1e-3) / 1e9
    achieved = algo_decode / (kern_ms * 1e-3) / 1e9 if decode_seqs else 0.0
    result = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline:
            s = oracle_sample(args.config, args.cpu_seconds)
            cpu = {"value": s["value"], "unit": UNIT, "cores": 1, "kind": "oracle",
                   "sample": f"first {s['seqs']} of {s['of_seqs']} sequences of the workload "
                             f"(same recipe), fp64 oracle step (set-up append, step append, "
                             f"attention), {s['seconds']:.1f} s on one host core",
                   "tokens_per_s": s["tokens_per_s"]}
        result = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3" if w.cache_dtype == "fp8_e4m3" else "bf16", "data": "synthetic",
            "config": {"workload": f"cfg{args.config}: {CONFIG_NAMES[args.config]}"
                                   + (f" (first {args.seqs} sequences)" if args.seqs else ""),
                       "l2": f"no flush: each step streams {algo_attn / 1e9:.2f} GB of K/V "
                             "and q/out, far above the 129 MB L2",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "hbm_frac_of_peak": value / world / peak,
            "timing": "CUDA graph of one step, replayed K times between CUDA events",
            "eager_ms_per_step": eager_ms,
            "attended_tokens_per_s": world * w.attended_tokens() / (step_ms * 1e-3),
            "algorithmic_bytes_per_step": algo_step,
            "e2e": {"value": world * algo_step / (e2e_ms * 1e-3) / 1e9, "unit": UNIT,
                    "h2d_bytes_per_step": dw.h2d_bytes, "d2h_bytes_per_step": dw.d2h_bytes,
                    "ms_per_step": e2e_ms,
                    "copies": "one packed host-to-device copy of each step's inputs and one "
                              "device-to-host copy of its output, on a copy stream, double-"
                              "buffered against the steps' compute"},
            "gpu_launches": K * dw.launches_per_step(),
            "roofline": {"bound": "hbm", "kernel": "decode_kernel (split-KV paged attention)",
                         "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
                         "traffic": traffic_from_profiles(args.config),
                         "algorithmic_bytes_per_launch": algo_decode,
                         "kernel_ms": kern_ms},
            "cpu_baseline": cpu,
            "clocks": clk,
        }
        if pf_flops and not decode_seqs:
            # every run of the step is on the tensor-core tiles (e.g. speculative verify with
            # GQA): that kernel is the dominant one, and it streams each K/V tile once
            pf_gbs = algo_prefill / (pf_ms * 1e-3) / 1e9
            result["roofline"] = {
                "bound": "hbm", "kernel": "prefill_kernel (tcgen05 causal tiles)",
                "achieved": pf_gbs, "peak": peak, "unit": "GB/s", "frac": pf_gbs / peak,
                "peak_source": f"{peak_kind} hbm_gbs", "traffic": None,
                "algorithmic_bytes_per_launch": algo_prefill, "kernel_ms": pf_ms}
        if pf_flops:
            peaks = load_peaks()[2]
            pf_peak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
            pf_tf = pf_flops / (pf_ms * 1e-3) / 1e12
            result["prefill"] = {
                "bound": "tensor", "kernel": "prefill_kernel (tcgen05 causal tiles)",
                "achieved": pf_tf, "peak": pf_peak, "unit": "TFLOP/s", "frac": pf_tf / pf_peak,
                "peak_source": ("measured" if "bf16_tflops" in peaks else "fallback")
                               + " bf16_tflops (burst)",
                "flops_per_launch": pf_flops, "kernel_ms": pf_ms,
                "algorithmic_bytes_per_launch": algo_prefill,
                "achieved_gbs": algo_prefill / (pf_ms * 1e-3) / 1e9,
                "flops": "algorithmic: 4 * head_dim * q heads * attended keys of the chunk "
                         "queries (QK^T and PV); masked tile parts and the second (lo) half "
                         "of P's bf16 split are extra MMA work not counted"}
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
