#!/usr/bin/env python3
"""Benchmark of exact sink-aware attention, forward + backward, on GB300.

One step = one forward and one backward pass (every kernel of the path) over
one batch of the workload.  Default workload: 2 sequences x 8192 tokens,
64 query / 8 key-value heads, head_dim 64, full causal mask, bf16 inputs.

The line's value is TFLOP/s counting only unmasked (query, key, head) pairs
at 14 * 64 FLOP per pair (forward 4 * 64, backward 10 * 64).  Inputs are
resident in HBM; L2 is flushed before every timed step (a 256 MiB write, then a
256 MiB read so the written lines drain outside the timed region), and
each step is timed alone with CUDA events on the stream the kernels run on.

Decode workloads (``--workload decode_*``): one step = one decode forward
(one key-chunk kernel that also merges) of the workload's query rows against the
key/value cache of every sequence, reported in GB/s of algorithmic HBM
traffic (the visible keys and values once, the queries, O and lse).

GRPO workloads (``--workload grpo_*``): one step = the GRPO token loss and
its gradient over one update batch of rollouts, in GB/s of algorithmic HBM
traffic (three fp32 log-probabilities and the mask read, the gradient written).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
       python bench.py --impl reference ...   (times the CPU float64 oracle)
Under torchrun each rank runs its own batch (weak scaling, no collective on
the data path; the process group only carries the barrier and the max-time
reduction).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "sink-attn fwd+bwd TFLOP/s (bf16, S=4k/8k) and % of GB300 dense bf16 peak"
DEFAULT_WORKLOAD = "causal_gqa_b2_s8192"
FLOP_FWD_PER_PAIR = 4 * 64
FLOP_BWD_PER_PAIR = 10 * 64
L2_FLUSH_BYTES = 256 << 20
# Attention: the library counts its launches per step (sinkattn_kernel_launches): forward, backward
# preprocess, backward main, dK/dV conversion of split key tiles (when any), dQ convert.
DECODE_METRIC = "sink-attn decode GB/s (bf16 KV-cache stream) and % of measured HBM copy bandwidth"
DECODE_LAUNCHES_PER_STEP = 1  # key-chunk kernel (the last chunk of each sequence merges)
GRPO_METRIC = "GRPO token loss GB/s (fp32 log-probs) and % of measured HBM copy bandwidth"
GRPO_LAUNCHES_PER_STEP = 1  # one cooperative kernel: advantages, tokens, grid barrier, 1/N scaling
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_NAMES = {"fwd": "fwd_tc_kernel", "bwd_main": "bwd_tc_kernel"}
# Attention workloads the default run also measures (one entry each under "configs").
EXTRA_CONFIGS = ("causal_gqa_s4096", "window128_gqa_s4096", "window128_prefix4_gqa_b2_s8192", "varlen8_window128",
                 "varlen8_causal")


# ----------------------------------------------------------------- accounting
def visible_pairs(wl) -> int:
    """Unmasked (query, key) pairs summed over sequences and query heads."""
    total = 0
    for n in wl.seqlens:
        q = np.arange(int(n), dtype=np.int64)
        lo = np.zeros_like(q) if wl.window < 0 else np.maximum(0, q - wl.window)
        hi = q if wl.causal else np.full_like(q, int(n) - 1)
        band = np.maximum(0, hi - lo + 1)
        extra = np.minimum(wl.prefix, lo)  # prefix keys below the band
        total += int(np.sum(band + extra))
    return total * wl.num_heads_q


def algorithmic_bytes(wl):
    """Minimum HBM bytes: fwd reads Q,K,V and writes O,lse; bwd reads
    Q,K,V,O,dO,lse and writes dQ,dK,dV."""
    T, hq, hkv, d = wl.total_tokens, wl.num_heads_q, wl.num_heads_kv, wl.head_dim
    q = T * hq * d * 2
    kv = T * hkv * d * 2
    lse = T * hq * 4
    fwd = q + 2 * kv + q + lse
    bwd = q + 2 * kv + q + q + lse + q + 2 * kv
    return fwd, bwd


def decode_visible_keys(wl, n):
    """Keys that at least one of the last n query rows of a sequence sees, summed over sequences."""
    total = 0
    for L in wl.seqlens:
        L = int(L)
        lo = 0 if wl.window < 0 else max(0, L - n - wl.window)
        total += (L - lo) + min(wl.prefix, lo)
    return total


def decode_plan_tiles(wl, n):
    """Key tiles per kv head of a decode step (the planner's count: the prefix
    tiles below the window, then the window/causal band of the last n rows)."""
    total = 0
    for L in wl.seqlens:
        q0, hi = L - n, L - 1
        lo = 0 if wl.window < 0 else max(0, q0 - wl.window)
        pre_end = max(0, min(min(wl.prefix, lo), hi + 1))
        lo_t = lo // 128
        total += min((pre_end + 127) // 128, lo_t) + (hi // 128 - lo_t + 1)
    return total


def decode_kernel(wl, n):
    """(short name, kernel function) of the decode launch: the tcgen05 kernel
    above 16 rows per (sequence, kv head) and for 16 or fewer from 128 key
    tiles per kv head, the warp-MMA kernel for the smallest steps."""
    rows = (wl.num_heads_q // wl.num_heads_kv) * n
    tc = rows > 16 or decode_plan_tiles(wl, n) >= 128
    return ("decode_tc", "decode_tc_kernel") if tc else ("decode_split", "decode_split_kernel")


def decode_bytes(wl, n):
    """Algorithmic HBM bytes of one decode step: visible K and V once per kv
    head, the query rows, O and lse."""
    rows = wl.num_seqs * n
    kv = decode_visible_keys(wl, n) * wl.num_heads_kv * wl.head_dim * 2 * 2
    q = rows * wl.num_heads_q * wl.head_dim * 2
    return kv + 2 * q + rows * wl.num_heads_q * 4


def grpo_bytes(inp):
    """Algorithmic HBM bytes of one GRPO step: logp, logp_old, logp_ref and
    the mask read once, dlogp written; rewards in, advantages and stats out."""
    T = int(inp.cu_tokens[-1])
    R = len(inp.cu_tokens) - 1
    ref = 4 if inp.wl.kl_beta else 0
    return T * (4 + 4 + ref + 1 + 4) + R * (4 + 4 + 4) + 16


def grpo_oracle_seconds(inp, rounds):
    import oracle.grpo_ref as gref

    args = (inp.logp.astype(np.float64), inp.logp_old.astype(np.float64), inp.logp_ref.astype(np.float64), inp.mask,
            inp.rewards.astype(np.float64), inp.cu_tokens, inp.wl.group_size, inp.wl.clip_eps, inp.wl.adv_eps,
            inp.wl.kl_beta)
    secs = []
    for _ in range(rounds):
        t = time.perf_counter()
        gref.grpo_loss(*args)
        secs.append(time.perf_counter() - t)
    return secs


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling (every ``interval_ms``) while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 50):
        self.gpu = gpu_index
        self.interval_ms = int(interval_ms)
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.interval_ms)], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        # nvidia-smi takes a moment to start: wait (up to 3 s) for its first
        # sample so that the timed region that follows is sampled from its start.
        t0 = time.monotonic()
        while time.monotonic() - t0 < 3.0 and self.proc.poll() is None:
            self.fh.flush()
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.01)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.06)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "interval_ms": self.interval_ms,
                "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------- oracle (CPU)
def _oracle_head_job(args):
    import oracle

    q, k, v, do, sink, cu, window, prefix, causal, scale = args
    t = time.perf_counter()
    oracle.forward_backward(q, k, v, sink, do, cu, window, prefix, causal, scale)
    return time.perf_counter() - t


def _init_worker():
    import oracle  # noqa: F401  (import cost outside the timed region)


def oracle_sample_jobs(wl, n_heads):
    """One sequence (the first), ``n_heads`` query heads: float64 slices."""
    inp = W.make_inputs(wl.with_(seqlens=(wl.seqlens[0],), uniform=True))
    group = wl.num_heads_q // wl.num_heads_kv
    cu = np.array([0, wl.seqlens[0]], dtype=np.int64)
    q, k, v, do, sink = (inp.f64(n) for n in ("q", "k", "v", "do", "sink"))
    jobs = []
    for i in range(n_heads):
        h = i % wl.num_heads_q
        g = h // group
        jobs.append((np.ascontiguousarray(q[:, h:h + 1]), np.ascontiguousarray(k[:, g:g + 1]),
                     np.ascontiguousarray(v[:, g:g + 1]), np.ascontiguousarray(do[:, h:h + 1]),
                     sink[h:h + 1].copy(), cu, wl.window, wl.prefix, wl.causal, wl.scale))
    one = wl.with_(seqlens=(wl.seqlens[0],), num_heads_q=1, num_heads_kv=1)
    flops = visible_pairs(one) * (FLOP_FWD_PER_PAIR + FLOP_BWD_PER_PAIR) * n_heads
    return jobs, flops


class OraclePool:
    """A spawn pool of single-threaded oracle workers (one per host core, up to
    16; the line reports the host's core count beside the worker count)."""

    def __init__(self):
        import multiprocessing as mp

        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        self.cores = max(1, min(16, os.cpu_count() or 1))
        self.pool = mp.get_context("spawn").Pool(self.cores, initializer=_init_worker)

    def run(self, jobs):
        t = time.perf_counter()
        self.pool.map(_oracle_head_job, jobs, chunksize=1)
        return time.perf_counter() - t

    def close(self):
        self.pool.terminate()


def cpu_baseline(wl, pool=None):
    own = pool is None
    pool = pool or OraclePool()
    try:
        jobs, flops = oracle_sample_jobs(wl, pool.cores)
        rounds = 3
        sec = sum(pool.run(jobs) for _ in range(rounds))
    finally:
        if own:
            pool.close()
    return {"value": rounds * flops / sec / 1e12, "unit": "TFLOP/s", "cores": pool.cores, "kind": "oracle",
            "host_cpu_count": os.cpu_count(),
            "sample": f"{rounds} rounds of {len(jobs)} query heads x 1 sequence of {wl.seqlens[0]} tokens of "
                      f"{wl.name}, fwd+bwd, one single-threaded worker per head, {sec:.2f} s wall"}


def _oracle_decode_job(args):
    import oracle

    q, k, v, sink, cu, n, window, prefix, causal, scale = args
    t = time.perf_counter()
    oracle.decode_forward(q, k, v, sink, cu, n, window, prefix, causal, scale)
    return time.perf_counter() - t


def decode_oracle_jobs(wl, n, cores):
    """One job per sequence of a bounded sample (the first min(B, cores)
    sequences, float64), and the algorithmic bytes the sample covers."""
    nseq = max(1, min(wl.num_seqs, cores))
    sub_wl = wl.with_(seqlens=tuple(wl.seqlens[:nseq]))
    inp = W.make_decode_inputs(sub_wl, n)
    q, k, v, sink = (inp.f64(x) for x in ("q", "k", "v", "sink"))
    cu = sub_wl.cu_seqlens()
    jobs = []
    for b in range(nseq):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        jobs.append((np.ascontiguousarray(q[b * n:(b + 1) * n]), np.ascontiguousarray(k[t0:t1]),
                     np.ascontiguousarray(v[t0:t1]), sink, np.array([0, t1 - t0]), n, wl.window, wl.prefix,
                     wl.causal, wl.scale))
    return jobs, decode_bytes(sub_wl, n), nseq


def decode_cpu_baseline(wl, n, steps=3):
    pool = OraclePool()
    try:
        jobs, nbytes, nseq = decode_oracle_jobs(wl, n, pool.cores)
        t = time.perf_counter()
        for _ in range(steps):
            pool.pool.map(_oracle_decode_job, jobs, chunksize=1)
        sec = time.perf_counter() - t
    finally:
        pool.close()
    return {"value": steps * nbytes / sec / 1e9, "unit": "GB/s", "cores": pool.cores, "kind": "oracle",
            "host_cpu_count": os.cpu_count(),
            "sample": f"{steps} rounds of {nseq} sequences of {wl.name} (all heads, {n} query rows each), "
                      f"one single-threaded worker per sequence, {sec:.2f} s wall"}


def run_reference_decode(args, rank):
    if rank != 0:
        return 0
    wl, n = W.DECODE_WORKLOADS[args.workload]
    pool = OraclePool()
    try:
        jobs, nbytes, nseq = decode_oracle_jobs(wl, n, pool.cores)
        for _ in range(args.warmup):
            pool.pool.map(_oracle_decode_job, jobs[:1], chunksize=1)
        secs = []
        for _ in range(args.steps):
            t = time.perf_counter()
            pool.pool.map(_oracle_decode_job, jobs, chunksize=1)
            secs.append(time.perf_counter() - t)
    finally:
        pool.close()
    total = sum(secs)
    value = nbytes * len(secs) / total / 1e9
    line = {
        "impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "sample_per_step": f"{nseq} sequences, all heads"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": pool.cores, "kind": "oracle",
                         "sample": f"each step: {nseq} sequences of {wl.name}, {n} query rows each"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference_grpo(args, rank):
    if rank != 0:
        return 0
    inp = W.make_grpo_inputs(W.GRPO_WORKLOADS[args.workload])
    grpo_oracle_seconds(inp, max(0, args.warmup))
    secs = grpo_oracle_seconds(inp, args.steps)
    total = sum(secs)
    nbytes = grpo_bytes(inp)
    value = nbytes * len(secs) / total / 1e9
    line = {
        "impl": "reference", "metric": GRPO_METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": inp.wl.name, "tokens": int(inp.cu_tokens[-1])},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"each step: the whole {inp.wl.name} batch, one NumPy process"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args, rank):
    """The oracle as the reference arm, on the host cores of rank 0."""
    if args.workload in W.GRPO_WORKLOADS:
        return run_reference_grpo(args, rank)
    if args.workload in W.DECODE_WORKLOADS:
        return run_reference_decode(args, rank)
    if rank != 0:
        return 0
    wl = W.WORKLOADS[args.workload]
    pool = OraclePool()
    try:
        jobs, flops = oracle_sample_jobs(wl, pool.cores)
        for _ in range(args.warmup):
            pool.run(jobs[:1])
        secs = [pool.run(jobs) for _ in range(args.steps)]
    finally:
        pool.close()
    total = sum(secs)
    value = flops * len(secs) / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "sample_per_step": f"{pool.cores} query heads x 1 sequence"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": pool.cores, "kind": "oracle",
                         "sample": f"each step: {pool.cores} query heads x 1 sequence of {wl.seqlens[0]} tokens "
                                   f"of {wl.name}, fwd+bwd"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- GPU arm
class L2Flush:
    """Between timed steps: write a buffer larger than L2 (evicts every line
    a step could reuse), then read a second one, so the write's dirty lines
    go back to HBM here and not during the next timed step."""

    def __init__(self, device):
        import torch

        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.out = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self, value=1.0):
        import torch

        self.w.fill_(float(value))
        torch.sum(self.r, dim=0, out=self.out)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(values, world, device):
    """Max over ranks of a list of floats (identity for one rank)."""
    if world == 1:
        return list(values)
    import torch
    import torch.distributed as dist

    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def attention_setup(wl, dev):
    """Device inputs, outputs and workspace of one attention workload."""
    import torch

    import sink_aware_masked_gb300 as sa

    inp = W.make_inputs(wl)
    q, k, v, do = (t.to(dev) for t in (inp.q_bf16, inp.k_bf16, inp.v_bf16, inp.do_bf16))
    sink = inp.sink.to(dev)
    if wl.uniform:
        prob = dict(num_seqs=wl.num_seqs)
    else:
        cu = wl.cu_seqlens()
        prob = dict(cu_seqlens=torch.tensor(cu, dtype=torch.int32, device=dev),
                    cu_seqlens_host=[int(x) for x in cu], max_seqlen=wl.max_seqlen)
    prob.update(window=wl.window, prefix=wl.prefix, causal=wl.causal, scale=wl.scale)
    st = dict(q=q, k=k, v=v, do=do, sink=sink, prob=prob, o=torch.empty_like(q),
              lse=torch.empty((wl.num_heads_q, wl.total_tokens), dtype=torch.float32, device=dev),
              dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v), dsink=torch.empty_like(sink))
    st["ws"] = torch.empty(max(16, sa.bwd_workspace_bytes(q, k, **prob)), dtype=torch.uint8, device=dev)
    # Our kernels per step, counted by the library from its own work lists.
    st["launches_per_step"] = (sa.kernel_launches(q, k, "fwd", **prob) + sa.kernel_launches(q, k, "bwd", **prob))
    return st


def attention_step(st):
    import sink_aware_masked_gb300 as sa

    sa.sinkattn_fwd(st["q"], st["k"], st["v"], st["sink"], o=st["o"], lse=st["lse"], **st["prob"])
    sa.sinkattn_bwd(st["q"], st["k"], st["v"], st["o"], st["lse"], st["do"], st["sink"], dq=st["dq"], dk=st["dk"],
                    dv=st["dv"], dsink=st["dsink"], workspace=st["ws"], **st["prob"])


def time_attention(st, K, warmup, dev, flush, world, sample_ms=50):
    """K timed steps (L2 flushed before each, outside its events), then K
    more with the library's per-kernel events installed.  The first pass
    replays the step captured once as a CUDA graph (the same kernels with
    the same arguments, no host work between them, as a training loop
    replays its step) and gives the step times and the clocks.  The second
    runs the calls eagerly with events around the forward and backward-main
    kernels and gives their times.  Returns (step ms, forward ms,
    backward-main ms, step ms of the second pass, clocks)."""
    import torch

    import sink_aware_masked_gb300 as sa

    for _ in range(max(warmup, 0)):
        flush(1.0)
        attention_step(st)
    torch.cuda.synchronize()
    if sa.sinkattn_get_device_status() != 0:
        raise RuntimeError("device status reported a timed-out wait during warm-up")
    graph = capture_step(lambda: attention_step(st))
    for _ in range(max(warmup, 1)):
        flush(1.0)
        graph.replay()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(K)]
    for e in ev:  # torch creates the CUDA event on first record(); the hook needs the handle
        for x in e:
            x.record()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index if dev.index is not None else 0, sample_ms)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    for i in range(K):
        flush(float(i))
        ev[i][0].record()
        graph.replay()
        ev[i][1].record()
    torch.cuda.synchronize()
    barrier(world)
    clock_info = clocks.stop()
    del graph
    for i in range(K):
        flush(float(i))
        e = ev[i]
        sa.sinkattn_set_profile_events(sa.PROFILE_FWD, e[2], e[3])
        sa.sinkattn_set_profile_events(sa.PROFILE_BWD_MAIN, e[4], e[5])
        e[6].record()
        attention_step(st)
        e[7].record()
    torch.cuda.synchronize()
    sa.sinkattn_set_profile_events(sa.PROFILE_FWD)
    sa.sinkattn_set_profile_events(sa.PROFILE_BWD_MAIN)
    if sa.sinkattn_get_device_status() != 0:
        raise RuntimeError("device status reported a timed-out wait")
    return ([e[0].elapsed_time(e[1]) for e in ev], [e[2].elapsed_time(e[3]) for e in ev],
            [e[4].elapsed_time(e[5]) for e in ev], [e[6].elapsed_time(e[7]) for e in ev], clock_info)


def roofline_of(wl, fwd_ms, bwd_main_ms, peaks, peak_src, workload_name):
    """Roofline of the dominant kernel (the larger mean CUDA-event time): its
    algorithmic FLOP per byte against the ridge point of the measured peaks
    (278 FLOP/B on GB300) decides whether tensor or HBM bounds it."""
    pairs = visible_pairs(wl)
    fwd_b, bwd_b = algorithmic_bytes(wl)
    avg_bwd, avg_fwd = statistics.mean(bwd_main_ms), statistics.mean(fwd_ms)
    dom = "bwd_main" if avg_bwd >= avg_fwd else "fwd"
    dom_ms = avg_bwd if dom == "bwd_main" else avg_fwd
    dom_flop = pairs * (FLOP_BWD_PER_PAIR if dom == "bwd_main" else FLOP_FWD_PER_PAIR)
    dom_bytes = bwd_b if dom == "bwd_main" else fwd_b
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if dom_flop / dom_bytes >= ridge:
        roof = {"bound": "tensor", "achieved": dom_flop / (dom_ms / 1e3) / 1e12, "peak": peaks["bf16_tflops"],
                "peak_source": f"{peak_src} bf16 burst", "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": dom_bytes / (dom_ms / 1e3) / 1e9, "peak": peaks["hbm_gbs"],
                "peak_source": f"{peak_src} HBM copy", "unit": "GB/s"}
    return {"bound": roof["bound"], "kernel": dom, "kernel_name": KERNEL_NAMES[dom], "achieved": roof["achieved"],
            "peak": roof["peak"], "peak_source": roof["peak_source"], "unit": roof["unit"],
            "frac": roof["achieved"] / roof["peak"], "traffic": _committed_traffic(workload_name, dom),
            "flop_per_byte": dom_flop / dom_bytes, "ridge_flop_per_byte": ridge, "algorithmic_bytes": dom_bytes,
            "kernel_ms": dom_ms, "tflops": dom_flop / (dom_ms / 1e3) / 1e12,
            "hbm_gbs_equiv": dom_bytes / (dom_ms / 1e3) / 1e9}


def measure_config(name, dev, flush, peaks, peak_src, target_s=0.3):
    """One extra workload at N = 1: enough timed steps to span about
    ``target_s`` seconds (so the 20 ms clock sampler sees the load), with its
    TFLOP/s, the dominant kernel against its roof, and the clocks."""
    import torch

    wl = W.WORKLOADS[name]
    st = attention_setup(wl, dev)
    probe = time_attention(st, 3, 3, dev, flush, 1)[0]
    K = int(min(2000, max(20, math.ceil(target_s * 1e3 / (statistics.median(probe) + 0.1)))))
    step_ms, fwd_ms, bwd_ms, step2_ms, clocks = time_attention(st, K, 3, dev, flush, 1, sample_ms=20)
    flop = visible_pairs(wl) * (FLOP_FWD_PER_PAIR + FLOP_BWD_PER_PAIR)
    tot = sum(step_ms)
    value = flop * K / (tot / 1e3) / 1e12
    roof = roofline_of(wl, fwd_ms, bwd_ms, peaks, peak_src, name)
    out = {"tflops": value, "pct_of_peak": 100.0 * value / peaks["bf16_tflops"], "ms_per_step": tot / K, "steps": K,
           "dominant_kernel": roof["kernel_name"], "dominant_ms": roof["kernel_ms"],
           "breakdown_ms": {"fwd_kernel": statistics.mean(fwd_ms), "bwd_main_kernel": statistics.mean(bwd_ms),
                            "rest": statistics.mean(step2_ms) - statistics.mean(fwd_ms) - statistics.mean(bwd_ms),
                            "step_with_kernel_events": statistics.mean(step2_ms)},
           "roofline": roof, "gpu_launches": K * st["launches_per_step"], "clocks": clocks,
           "flop_per_step": flop, "algorithmic_bytes_per_step": sum(algorithmic_bytes(wl))}
    del st
    torch.cuda.empty_cache()
    return out


def _time_graph(step, K, dev, flush, sample_ms=20):
    """K CUDA-graph replays of ``step`` (L2 flushed before each, outside its
    events), with the clocks sampled meanwhile."""
    import torch

    graph = capture_step(step)
    for _ in range(3):
        flush(1.0)
        graph.replay()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index if dev.index is not None else 0, sample_ms)
    clocks.start()
    for i in range(K):
        flush(float(i))
        ev[i][0].record()
        graph.replay()
        ev[i][1].record()
    torch.cuda.synchronize()
    info = clocks.stop()
    return [a.elapsed_time(b) for a, b in ev], info


def measure_decode_config(name, dev, flush, peaks, peak_src, target_s=0.3):
    """One decode workload at N = 1: graph replays of the one-kernel step for
    about ``target_s`` seconds, GB/s of algorithmic bytes against HBM."""
    import torch

    import sink_aware_masked_gb300 as sa

    wl, n = W.DECODE_WORKLOADS[name]
    inp = W.make_decode_inputs(wl, n)
    q, k, v, sink = (t.to(dev) for t in (inp.q_bf16, inp.k_bf16, inp.v_bf16, inp.sink))
    if wl.uniform:
        prob = dict(num_seqs=wl.num_seqs)
    else:
        cu = wl.cu_seqlens()
        prob = dict(cu_seqlens=torch.tensor(cu, dtype=torch.int32, device=dev),
                    cu_seqlens_host=[int(x) for x in cu], max_seqlen=wl.max_seqlen)
    prob.update(window=wl.window, prefix=wl.prefix, causal=wl.causal, scale=wl.scale)
    o = torch.empty_like(q)
    lse = torch.empty((wl.num_heads_q, q.shape[0]), dtype=torch.float32, device=dev)
    ws = torch.zeros(max(16, sa.decode_workspace_bytes(q, k, q_per_seq=n, **prob)), dtype=torch.uint8, device=dev)

    def step():
        sa.sinkattn_decode_fwd(q, k, v, sink, q_per_seq=n, o=o, lse=lse, workspace=ws, **prob)

    for _ in range(3):
        flush(1.0)
        step()
    torch.cuda.synchronize()
    probe, _ = _time_graph(step, 5, dev, flush)
    K = int(min(3000, max(20, math.ceil(target_s * 1e3 / (statistics.median(probe) + 0.1)))))
    ms, clocks = _time_graph(step, K, dev, flush)
    if sa.sinkattn_get_device_status() != 0:
        raise RuntimeError("device status reported a timed-out wait")
    nbytes = decode_bytes(wl, n)
    gbs = nbytes * K / (sum(ms) / 1e3) / 1e9
    short, kname = decode_kernel(wl, n)
    out = {"gbs": gbs, "ms_per_step": sum(ms) / K, "steps": K, "dominant_kernel": kname,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "peak_source": f"{peak_src} HBM copy",
                        "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes": nbytes,
                        "traffic": _committed_traffic(name, short)},
           "gpu_launches": K * DECODE_LAUNCHES_PER_STEP, "clocks": clocks,
           "timing": "CUDA-graph replay of the one-kernel step"}
    del q, k, v, o, lse, ws
    torch.cuda.empty_cache()
    return out


def measure_grpo_config(name, dev, flush, peaks, peak_src, target_s=0.3):
    """The GRPO loss workload at N = 1: graph replays of the one-kernel step."""
    import torch

    import sink_aware_masked_gb300 as sa

    inp = W.make_grpo_inputs(W.GRPO_WORKLOADS[name])
    wl = inp.wl
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    logp, old, lref, mask, rew, cu = (t(a) for a in (inp.logp, inp.logp_old, inp.logp_ref, inp.mask, inp.rewards,
                                                      inp.cu_tokens))
    cu_host = [int(x) for x in inp.cu_tokens]
    dlogp = torch.empty_like(logp)
    ws = torch.zeros(sa.grpo_workspace_bytes(cu, cu_host, group_size=wl.group_size), dtype=torch.uint8, device=dev)
    kw = dict(group_size=wl.group_size, clip_eps=wl.clip_eps, adv_eps=wl.adv_eps, kl_beta=wl.kl_beta,
              logp_ref=lref if wl.kl_beta else None, dlogp=dlogp, workspace=ws)

    def step():
        sa.grpo_loss(logp, old, mask, rew, cu, cu_host, **kw)

    for _ in range(3):
        flush(1.0)
        step()
    torch.cuda.synchronize()
    probe, _ = _time_graph(step, 5, dev, flush)
    K = int(min(3000, max(20, math.ceil(target_s * 1e3 / (statistics.median(probe) + 0.1)))))
    ms, clocks = _time_graph(step, K, dev, flush)
    if sa.sinkattn_get_device_status() != 0:
        raise RuntimeError("device status reported a timed-out wait")
    nbytes = grpo_bytes(inp)
    gbs = nbytes * K / (sum(ms) / 1e3) / 1e9
    return {"gbs": gbs, "ms_per_step": sum(ms) / K, "steps": K, "dominant_kernel": "grpo_kernel",
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "peak_source": f"{peak_src} HBM copy",
                         "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes": nbytes,
                         "traffic": _committed_traffic(name, "grpo")},
            "gpu_launches": K * GRPO_LAUNCHES_PER_STEP, "clocks": clocks,
            "timing": "CUDA-graph replay of the one-kernel step"}


def run_gpu(args, world, rank, local):
    import torch

    import sink_aware_masked_gb300 as sa
    from sink_aware_masked_gb300 import build as sa_build

    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    sa_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    base = W.WORKLOADS[args.workload]
    wl = base.with_(seed=base.seed + 1000 * rank)  # each rank: its own batch
    st = attention_setup(wl, dev)
    q, k, v, do, sink, o, lse, ws, prob = (st[n] for n in ("q", "k", "v", "do", "sink", "o", "lse", "ws", "prob"))
    flush = L2Flush(dev)
    K = args.steps
    step_ms, fwd_ms, bwd_main_ms, step2_ms, clock_info = time_attention(st, K, args.warmup, dev, flush, world,
                                                                          sample_ms=20)

    # ---- end to end through host buffers (pinned), copies inside the timed
    # region.  Double-buffered, as a training loop feeding the library would
    # run it: step i+1's inputs go up on one stream and step i-1's results
    # come back on another while step i computes; every step copies its own
    # inputs in and all of its outputs out.
    host_in = [t.cpu().pin_memory() for t in (q, k, v, do, sink)]
    sets = []
    for _ in range(2):
        din = [torch.empty_like(t) for t in (q, k, v, do, sink)]
        dout = [torch.empty_like(t) for t in (o, lse, st["dq"], st["dk"], st["dv"], st["dsink"])]
        sets.append((din, dout, [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dout]))
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in sets[0][2])
    s_comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    Ke = max(2, min(K, 10))
    ev_in, ev_comp, ev_out = ([torch.cuda.Event() for _ in range(Ke)] for _ in range(3))
    e2e_start, e2e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e2e_start.record(s_comp)
    s_in.wait_stream(s_comp)
    for i in range(Ke):
        din, dout, hout = sets[i % 2]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_comp[i - 2])  # step i - 2 has finished with this input set
            for d_, h_ in zip(din, host_in):
                d_.copy_(h_, non_blocking=True)
            ev_in[i].record(s_in)
        s_comp.wait_event(ev_in[i])
        if i >= 2:
            s_comp.wait_event(ev_out[i - 2])  # step i - 2's results have left this output set
        sa.sinkattn_fwd(din[0], din[1], din[2], din[4], o=dout[0], lse=dout[1], **prob)
        sa.sinkattn_bwd(din[0], din[1], din[2], dout[0], dout[1], din[3], din[4], dq=dout[2], dk=dout[3],
                        dv=dout[4], dsink=dout[5], workspace=ws, **prob)
        ev_comp[i].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[i])
            for h_, d_ in zip(hout, dout):
                h_.copy_(d_, non_blocking=True)
            ev_out[i].record(s_out)
    s_comp.wait_stream(s_out)
    s_comp.wait_stream(s_in)
    e2e_end.record(s_comp)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = [e2e_start.elapsed_time(e2e_end)]
    if sa.sinkattn_get_device_status() != 0:
        raise RuntimeError("device status reported a timed-out wait")
    del sets, host_in

    # ---- reduce over ranks (max) and report
    tot, e2e_tot = reduce_max([sum(step_ms), sum(e2e_ms)], world, dev)
    pairs = visible_pairs(wl)
    flop_step = pairs * (FLOP_FWD_PER_PAIR + FLOP_BWD_PER_PAIR)
    value = world * flop_step * K / (tot / 1e3) / 1e12
    e2e_value = world * flop_step * Ke / (e2e_tot / 1e3) / 1e12
    peaks, peak_src = load_peaks()
    roof = roofline_of(wl, fwd_ms, bwd_main_ms, peaks, peak_src, args.workload)
    avg_fwd, avg_bwd = statistics.mean(fwd_ms), statistics.mean(bwd_main_ms)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": tot / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": wl.name, "global_batch": wl.num_seqs * world, "seq_len": wl.max_seqlen,
                   "heads_q": wl.num_heads_q, "heads_kv": wl.num_heads_kv, "head_dim": wl.head_dim,
                   "window": wl.window, "prefix": wl.prefix, "causal": wl.causal,
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "l2": "flushed before every step (256 MiB write, then 256 MiB read so the written lines drain; outside the step events)",
                   "timing": "each step one CUDA-graph replay of the forward and backward calls (every kernel of the "
                             "path, captured once); e2e = eager calls with host copies",
                   "flop_per_step": flop_step, "unmasked_pairs": pairs},
        "pct_of_peak": 100.0 * value / world / peaks["bf16_tflops"],
        "breakdown_ms": {"fwd_kernel": avg_fwd, "bwd_main_kernel": avg_bwd,
                         "rest": statistics.mean(step2_ms) - avg_fwd - avg_bwd,
                         "step_with_kernel_events": statistics.mean(step2_ms),
                         "note": "ms_per_step: CUDA-graph replays of the whole step; kernel times from a second, "
                                 "eager pass of the same steps with events around the two main kernels"},
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": Ke, "mode": "pinned host buffers, double-buffered: step i+1's inputs up and step i-1's "
                                     "outputs down on two copy streams while step i computes; one timed region"},
        "gpu_launches": K * st["launches_per_step"],
        "clocks": clock_info,
    }
    del st, q, k, v, do, sink, o, lse, ws
    torch.cuda.empty_cache()
    if world == 1 and not args.no_configs:
        # The other attention workloads at N = 1, each timed the same way
        # (not part of the line's value): causal and windowed, uniform and packed.
        line["configs"] = {name: measure_config(name, dev, flush, peaks, peak_src)
                           for name in EXTRA_CONFIGS if name != args.workload}
        # The rollout-side decode forward and the GRPO loss of the same
        # training loop, each one kernel, in GB/s of algorithmic bytes.
        for name in sorted(W.DECODE_WORKLOADS):
            line["configs"][name] = measure_decode_config(name, dev, flush, peaks, peak_src)
        for name in sorted(W.GRPO_WORKLOADS):
            line["configs"][name] = measure_grpo_config(name, dev, flush, peaks, peak_src)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def run_gpu_decode(args, world, rank, local):
    """Decode steps of a DECODE_WORKLOADS entry; the key/value cache stays
    resident (it is the decoder's state), the query rows are the step's input."""
    import torch

    import sink_aware_masked_gb300 as sa
    from sink_aware_masked_gb300 import build as sa_build

    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    sa_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    base, n = W.DECODE_WORKLOADS[args.workload]
    wl = base.with_(seed=base.seed + 1000 * rank)
    inp = W.make_decode_inputs(wl, n)
    q, k, v, sink = (t.to(dev) for t in (inp.q_bf16, inp.k_bf16, inp.v_bf16, inp.sink))
    if wl.uniform:
        prob = dict(num_seqs=wl.num_seqs)
    else:
        cu = wl.cu_seqlens()
        prob = dict(cu_seqlens=torch.tensor(cu, dtype=torch.int32, device=dev),
                    cu_seqlens_host=[int(x) for x in cu], max_seqlen=wl.max_seqlen)
    prob.update(window=wl.window, prefix=wl.prefix, causal=wl.causal, scale=wl.scale)
    o = torch.empty_like(q)
    lse = torch.empty((wl.num_heads_q, q.shape[0]), dtype=torch.float32, device=dev)
    ws = torch.zeros(max(16, sa.decode_workspace_bytes(q, k, q_per_seq=n, **prob)), dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)

    def step():
        sa.sinkattn_decode_fwd(q, k, v, sink, q_per_seq=n, o=o, lse=lse, workspace=ws, **prob)

    for _ in range(max(args.warmup, 0)):
        flush(1.0)
        step()
    torch.cuda.synchronize()
    if sa.sinkattn_get_device_status() != 0:
        raise RuntimeError("device status reported a timed-out wait during warm-up")
    # The step is one kernel; a graph replay of it is timed, so the events
    # measure the kernel without the Python-side argument marshalling.
    graph = capture_step(step)
    for _ in range(max(args.warmup, 0)):
        flush(1.0)
        graph.replay()
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    for i in range(K):
        flush(float(i))
        e = ev[i]
        e[0].record()
        graph.replay()
        e[1].record()
    torch.cuda.synchronize()
    barrier(world)
    clock_info = clocks.stop()
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    split_ms = step_ms
    if sa.sinkattn_get_device_status() != 0:
        raise RuntimeError("device status reported a timed-out wait")

    # end to end: the step's query rows from pinned host memory, O and lse back
    host_q = q.cpu().pin_memory()
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse)]
    h2d = host_q.numel() * host_q.element_size()
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    Ke = max(1, min(K, 20))
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Ke)]
    barrier(world)
    for i in range(Ke):
        flush(float(i))
        e2e_ev[i][0].record()
        q.copy_(host_q, non_blocking=True)
        step()
        for h_, d_ in zip(host_out, (o, lse)):
            h_.copy_(d_, non_blocking=True)
        e2e_ev[i][1].record()
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = [a.elapsed_time(b) for a, b in e2e_ev]

    tot, e2e_tot = reduce_max([sum(step_ms), sum(e2e_ms)], world, dev)
    nbytes = decode_bytes(wl, n)
    value = world * nbytes * K / (tot / 1e3) / 1e9
    e2e_value = world * nbytes * Ke / (e2e_tot / 1e3) / 1e9
    peaks, peak_src = load_peaks()
    avg_split = statistics.mean(split_ms)
    achieved = nbytes / (avg_split / 1e3) / 1e9
    line = {
        "metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": tot / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": wl.name, "sequences": wl.num_seqs * world, "cached_tokens": wl.total_tokens,
                   "query_rows_per_seq": n, "heads_q": wl.num_heads_q, "heads_kv": wl.num_heads_kv,
                   "head_dim": wl.head_dim, "window": wl.window, "prefix": wl.prefix, "causal": wl.causal,
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "l2": "flushed before every step (256 MiB write, then 256 MiB read so the written lines drain; outside the step events)",
                   "timing": "CUDA graph replay of one step (one kernel); e2e = eager calls with host copies",
                   "algorithmic_bytes_per_step": nbytes,
                   "decode_rows_per_s": world * wl.num_seqs * n * K / (tot / 1e3)},
        "pct_of_peak": 100.0 * value / world / peaks["hbm_gbs"],
        "breakdown_ms": {"split_kernel": avg_split, "rest": statistics.mean(step_ms) - avg_split},
        "roofline": {"bound": "hbm", "kernel": decode_kernel(wl, n)[0], "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "peak_source": f"{peak_src} HBM copy", "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "traffic": _committed_traffic(args.workload, decode_kernel(wl, n)[0]),
                     "algorithmic_bytes": nbytes},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "the key/value cache is the decoder's resident state; the step's query rows cross PCIe"},
        "gpu_launches": K * DECODE_LAUNCHES_PER_STEP,
        "clocks": clock_info,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = decode_cpu_baseline(wl, n)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def run_gpu_grpo(args, world, rank, local):
    """GRPO loss steps; each rank its own batch (weak scaling)."""
    import dataclasses

    import torch

    import sink_aware_masked_gb300 as sa
    from sink_aware_masked_gb300 import build as sa_build

    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    sa_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    base = W.GRPO_WORKLOADS[args.workload]
    inp = W.make_grpo_inputs(dataclasses.replace(base, seed=base.seed + 1000 * rank))
    wl = inp.wl
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    logp, old, lref, mask, rew, cu = (t(a) for a in (inp.logp, inp.logp_old, inp.logp_ref, inp.mask, inp.rewards,
                                                      inp.cu_tokens))
    cu_host = [int(x) for x in inp.cu_tokens]
    dlogp = torch.empty_like(logp)
    # Zero-filled once; every completed call leaves it reusable.
    ws = torch.zeros(sa.grpo_workspace_bytes(cu, cu_host, group_size=wl.group_size), dtype=torch.uint8, device=dev)
    kw = dict(group_size=wl.group_size, clip_eps=wl.clip_eps, adv_eps=wl.adv_eps, kl_beta=wl.kl_beta,
              logp_ref=lref if wl.kl_beta else None, dlogp=dlogp, workspace=ws)
    flush = L2Flush(dev)
    out = {}

    def step():
        out["stats"], _, out["adv"] = sa.grpo_loss(logp, old, mask, rew, cu, cu_host, **kw)

    for _ in range(max(args.warmup, 0)):
        flush(1.0)
        step()
    torch.cuda.synchronize()
    graph = capture_step(step)
    for _ in range(max(args.warmup, 0)):
        flush(1.0)
        graph.replay()
    torch.cuda.synchronize()
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    for i in range(K):
        flush(float(i))
        ev[i][0].record()
        graph.replay()
        ev[i][1].record()
    torch.cuda.synchronize()
    barrier(world)
    clock_info = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]

    host_in = [torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
               for a in (inp.logp, inp.logp_old, inp.logp_ref, inp.mask, inp.rewards)]
    dev_in = (logp, old, lref, mask, rew)
    host_out = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in (dlogp, out["stats"])]
    h2d = sum(x.numel() * x.element_size() for x in host_in)
    d2h = sum(x.numel() * x.element_size() for x in host_out)
    Ke = max(1, min(K, 20))
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Ke)]
    barrier(world)
    for i in range(Ke):
        flush(float(i))
        e2e_ev[i][0].record()
        for d_, h_ in zip(dev_in, host_in):
            d_.copy_(h_, non_blocking=True)
        step()
        for h_, d_ in zip(host_out, (dlogp, out["stats"])):
            h_.copy_(d_, non_blocking=True)
        e2e_ev[i][1].record()
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = [a.elapsed_time(b) for a, b in e2e_ev]

    tot, e2e_tot = reduce_max([sum(step_ms), sum(e2e_ms)], world, dev)
    nbytes = grpo_bytes(inp)
    value = world * nbytes * K / (tot / 1e3) / 1e9
    peaks, peak_src = load_peaks()
    achieved = nbytes / (statistics.mean(step_ms) / 1e3) / 1e9
    line = {
        "metric": GRPO_METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": tot / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": wl.name, "prompts": wl.prompts * world, "group_size": wl.group_size,
                   "tokens": int(inp.cu_tokens[-1]), "optimised_tokens": int(np.count_nonzero(inp.mask)),
                   "clip_eps": wl.clip_eps, "kl_beta": wl.kl_beta,
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "l2": "flushed before every step (256 MiB write, then 256 MiB read so the written lines drain; outside the step events)",
                   "timing": "CUDA graph replay of one step (one kernel); e2e = eager calls with host copies",
                   "algorithmic_bytes_per_step": nbytes},
        "pct_of_peak": 100.0 * value / world / peaks["hbm_gbs"],
        "roofline": {"bound": "hbm", "kernel": "grpo_kernel (the whole step: one launch)", "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "peak_source": f"{peak_src} HBM copy", "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": _committed_traffic(args.workload, "grpo"),
                     "algorithmic_bytes": nbytes},
        "e2e": {"value": world * nbytes * Ke / (e2e_tot / 1e3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": K * GRPO_LAUNCHES_PER_STEP,
        "clocks": clock_info,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        secs = grpo_oracle_seconds(inp, 3)
        line["cpu_baseline"] = {"value": 3 * nbytes / sum(secs) / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": f"3 rounds of the whole {wl.name} batch, one NumPy process, "
                                          f"{sum(secs):.2f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def capture_step(step):
    """One step captured as a CUDA graph (for microsecond-scale steps whose
    Python-side argument marshalling would otherwise be timed as GPU idle)."""
    import torch

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    return graph


def _committed_traffic(workload, kernel):
    """DRAM bytes per launch from the committed ncu summary, if one matches."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(workload, {}).get(kernel)
    if not rec:
        return None
    import hashlib

    src = os.path.join(ROOT, rec["source"])
    if not os.path.exists(src):
        return None
    with open(src, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != rec["sha256"]:
            return None  # the kernel changed since the counters were taken
    return rec["bytes"]


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(W.WORKLOADS) + sorted(W.DECODE_WORKLOADS) + sorted(W.GRPO_WORKLOADS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle CPU baseline leg")
    ap.add_argument("--no-configs", action="store_true", help="skip the extra attention workloads (configs)")
    args = ap.parse_args(argv)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, rank)
    if args.workload in W.DECODE_WORKLOADS:
        return run_gpu_decode(args, world, rank, local)
    if args.workload in W.GRPO_WORKLOADS:
        return run_gpu_grpo(args, world, rank, local)
    return run_gpu(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
