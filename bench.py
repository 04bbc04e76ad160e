"""Benchmark of the GB300 gated delta-rule block (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload batched_decode_64|single_seq_decode_1000|
                                serving_pool_256_of_512|prefill_scan_4x4096|
                                prefill_chunked_4x4096|prefill_block_4x4096|
                                spec_verify_64x4]

Default workload: batched decode, 64 independent sequences, one token each per
step (Hk=16, H=32, S=128, conv 4), through the fused gdn_block_decode kernel.
A step is one fused launch over the 64 sequences; the state (128 MiB) is carried
from step to step. L2 is flushed before every timed step (a 256 MiB write, then a
256 MiB read, so no dirty lines are left to write back), and each step is timed
with CUDA events on the launching stream.

With N > 1 (torchrun, one process per GPU) every rank serves its own 64
sequences (weak scaling, no collective on the data path); rank 0 prints the
line, timed as the max over ranks.

--impl reference times the CPU oracle (the plain C reference, float build,
single-threaded) on a bounded sample of the same workload.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gated_deltanet_linear_scan_gb300 import inputs as I  # noqa: E402

METRIC = "GDN decode tokens/s and state HBM GB/s (fraction of GB300 peak), 1 GPU"
WORKLOADS = {"batched_decode_64": 3, "single_seq_decode_1000": 1,
             "serving_pool_256_of_512": 4, "prefill_scan_4x4096": 2,
             "prefill_chunked_4x4096": 2, "prefill_block_4x4096": 2,
             "spec_verify_64x4": 3, "prefill_varlen_16k": 2}
# Ragged prefill: a seeded mix of lengths (log-uniform in [1, 4096]) adding up to the
# 4 x 4096 workload's 16384 tokens, through the chunked prefill block in one call.
VARLEN_TOKENS = 16384
# Workloads that take a configuration with fields replaced: speculative-decoding
# verification scores 4 draft tokens of each of the 64 batched-decode sequences.
OVERRIDES = {"spec_verify_64x4": {"n_tokens": 4}}
SPEC_TOKENS = 4


def chunked_tensor_flops(n_seqs, n_tokens, n_v_heads):
    """Tensor-core flops the chunked scan issues (S = 128, chunks of 32, bf16 operand
    parts): per (sequence, v-head, chunk) the S products hi(S) [hi W | hi Gam q | lo W |
    lo Gam q] (N = 128, K = 128) and lo(S) [hi W | hi Gam q] (N = 64), then the state
    update with the U part of y, U^T [w K | M]^T in 3 passes (N = 160, K = 32)."""
    per = 2 * 128 * 128 * 128 + 2 * 128 * 64 * 128 + 3 * (2 * 128 * 160 * 32)
    return per * n_seqs * n_v_heads * ((n_tokens + 31) // 32)


def chunked_method_flops(n_chunks_total, n_v_heads):
    """The chunked scan's own contraction flops, without the 3xBF16 passes: per (sequence,
    v-head, chunk) the S products S^T [Gam q | W] (M = 128, N = 64, K = 128) and the state
    update with the U part of y, U^T [w K | M]^T (M = 128, N = 160, K = 32)."""
    per = 2 * 128 * 64 * 128 + 2 * 128 * 160 * 32
    return per * n_chunks_total * n_v_heads


def chunk_prepare_flops(n_seqs, n_tokens, n_k_heads, n_v_heads):
    """FP32 flops of the chunk-preparation phase (S = 128, chunks of 32): per (sequence,
    k-head, chunk) the Gram products k_t.k_s (s < t) and q_t.k_s (s <= t) over dk; per
    v-head the right-hand sides, A and M, and the two forward substitutions (W and Ut,
    128 columns each, 496 multiply-adds per column)."""
    gram = (496 + 528) * 128 * 2
    per_vhead = 2 * 128 * 496 * 2 + 32 * 128 * 3 + (496 + 528) * 3
    n_chunks = (n_tokens + 31) // 32
    return n_seqs * n_k_heads * n_chunks * (gram + (n_v_heads // n_k_heads) * per_vhead)
FLUSH_BYTES = 256 << 20
L2_NOTE = "flushed before every timed step (256 MiB write, then 256 MiB read: cold, clean L2)"
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ small helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": FALLBACK_HBM_GBS, "sm_max_mhz": 2070.0}, "fallback"


def source_sha(files):
    h = hashlib.sha256()
    for rel in files:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "block_decode_kernel": ["gated_deltanet_linear_scan_gb300/csrc/gdn_block.cu",
                            "gated_deltanet_linear_scan_gb300/csrc/gdn_device.cuh",
                            "gated_deltanet_linear_scan_gb300/csrc/gdn_internal.h"],
    "recurrence_scan_kernel": ["gated_deltanet_linear_scan_gb300/csrc/gdn_recurrence.cu",
                               "gated_deltanet_linear_scan_gb300/csrc/gdn_device.cuh",
                               "gated_deltanet_linear_scan_gb300/csrc/gdn_internal.h"],
    "chunked_scan_kernel": ["gated_deltanet_linear_scan_gb300/csrc/gdn_chunked.cu",
                            "gated_deltanet_linear_scan_gb300/csrc/gdn_chunk_common.cuh",
                            "gated_deltanet_linear_scan_gb300/csrc/gdn_device.cuh",
                            "gated_deltanet_linear_scan_gb300/csrc/gdn_tc.cuh",
                            "gated_deltanet_linear_scan_gb300/csrc/gdn_internal.h"],
    "chunk_state_kernel": ["gated_deltanet_linear_scan_gb300/csrc/gdn_chunked_ws.cu",
                           "gated_deltanet_linear_scan_gb300/csrc/gdn_chunk_common.cuh",
                           "gated_deltanet_linear_scan_gb300/csrc/gdn_device.cuh",
                           "gated_deltanet_linear_scan_gb300/csrc/gdn_tc.cuh",
                           "gated_deltanet_linear_scan_gb300/csrc/gdn_internal.h"],
}


def time_chunked_phases(gdn, torch, stream, state, state0, x, y, dims, scale, ws, steps, flush):
    """Per-step seconds of the two phases of the chunked scan (gdn_chunked_prepare,
    gdn_chunked_advance over all chunks), each timed with CUDA events on `stream`, L2
    flushed before every step."""
    N, T, Hk, H, S = dims
    nc = (T + 31) // 32
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    gpu_head_start(torch)
    for i in range(steps):
        state.copy_(state0)
        flush()
        ev[i][0].record(stream)
        gdn.gdn_chunked_prepare(x["q"], x["k"], x["v"], x["g"], x["beta"], ws, N, T, Hk, H, S,
                                0, nc)
        ev[i][1].record(stream)
        gdn.gdn_chunked_advance(state, x["q"], x["k"], x["g"], ws, y, N, T, Hk, H, S, scale, 0,
                                nc)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    prep = sum(e[0].elapsed_time(e[1]) for e in ev) / 1e3 / steps
    adv = sum(e[1].elapsed_time(e[2]) for e in ev) / 1e3 / steps
    return prep, adv


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch of this kernel and workload from the machine-readable ncu
    record (profiles/ncu_traffic.json, one entry per committed summary), if the
    kernel's source is unchanged since the counters were taken; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(f"{kernel}_{workload}")
    if not rec or rec.get("source_sha256_16") != source_sha(KERNEL_SOURCES[kernel]):
        return None
    return float(rec["dram_bytes_per_launch"])


def gpu_head_start(torch):
    """Give the device about a millisecond of work before the first timed step, so the
    host enqueues the timed steps ahead of the device: no host latency lands between a
    step's two events."""
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is not None:
        sleep(4_000_000)


def host_cpu():
    """The host's logical CPU count and model name (lscpu, else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None and os.path.exists("/proc/cpuinfo"):
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                model = line.split(":", 1)[1].strip()
                break
    return {"nproc": os.cpu_count(), "cpu_model": model}


def cpu_record(value, sample, cores=1):
    """The cpu_baseline object: the oracle's rate with the host it ran on and its build."""
    from oracle import build as oracle_build
    return {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": sample, **host_cpu(),
            "oracle_build": "gcc " + " ".join(oracle_build.CFLAGS) + " (float build)"}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_mark = None

    def mark(self):
        """The timed region starts now: the summary keeps only later samples."""
        self.t_mark = time.monotonic()

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = [ln for t, ln in self.lines if self.t_mark is None or t >= self.t_mark]
        if not lines and self.lines:  # a timed region shorter than one sampling period
            lines = [self.lines[-1][1]]
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def timed_steps(torch, stream, gpu, dist, warmup, steps, before, launch):
    """`warmup` untimed steps, then exactly `steps` timed ones, each bracketed by CUDA
    events on `stream` around launch(i) (before(i) -- the L2 flush, a state reset -- runs
    outside the events), between a barrier and a synchronize on both sides. The clock
    sampler starts before the warm-up, so no idle gap precedes the timed steps, and its
    summary covers the timed steps only. Returns (per-step ms, clock summary, wall s)."""
    with ClockSampler(gpu) as clocks:
        for w in range(warmup):
            before(w)
            launch(w)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        clocks.mark()
        t_wall = time.perf_counter()
        gpu_head_start(torch)
        for i in range(steps):
            before(i)
            ev[i][0].record(stream)
            launch(i)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in ev], clocks.summary(), t_wall


PIPELINE_NOTE = ("pipelined: step i + 1's inputs cross to the device on one copy stream and "
                 "step i - 1's result back on another while step i computes (inputs and "
                 "outputs double-buffered); every step's copies are inside the timed region; "
                 "no L2 flush (the step's working set exceeds L2)")
PIPELINE_NOTE_ONE = ("pipelined on one copy stream: once step i has computed, its result "
                     "and step i + 2's inputs cross while step i + 1 computes (inputs and "
                     "outputs double-buffered); every step's copies are inside the timed "
                     "region; no L2 flush (the step's working set exceeds L2)")


def pipelined_e2e(torch, dist, steps, h2d, compute, d2h, warmup=2, graph=False,
                  one_copy_stream=False):
    """End-to-end steps as a server runs them: h2d(i, b) copies step i's inputs from pinned
    host memory into device buffer set b = i % 2 on a copy stream, compute(i, b) runs the
    step on the current stream once they have landed, d2h(i, b) copies its result back on
    a second copy stream. A buffer set is refilled only after the step that used it has
    finished computing and its result has been copied out. Returns the seconds from the
    first input copy to the last result copy of the `steps` timed steps (max over ranks),
    after `warmup` untimed ones. With graph=True the same `steps` steps (the copies and the
    library calls, in their stream order) are captured once in a CUDA graph and the graph
    is replayed, once untimed and once timed: the device time without the host's per-call
    overhead. one_copy_stream: both directions on one copy stream (for steps whose copies
    take well under a step, where the host's event and stream calls are the cost): the
    result of step i and the inputs of step i + 2 cross once step i has computed."""
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    s_last = s_in if one_copy_stream else s_out  # the stream of the last result copy

    def enqueue_one(n, cur):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_done = [torch.cuda.Event() for _ in range(n)]
        torch.cuda.set_stream(s_in)
        for i in range(min(2, n)):
            h2d(i, i % 2)
            ev_in[i].record(s_in)
        torch.cuda.set_stream(cur)
        for i in range(n):
            b = i % 2
            cur.wait_event(ev_in[i])      # its inputs have landed; step i - 2's result has
            compute(i, b)                 # left buffer b (copied before those inputs)
            ev_done[i].record(cur)
            s_in.wait_event(ev_done[i])
            torch.cuda.set_stream(s_in)
            d2h(i, b)
            if i + 2 < n:                 # buffer b is free for step i + 2's inputs
                h2d(i + 2, b)
                ev_in[i + 2].record(s_in)
            torch.cuda.set_stream(cur)

    def enqueue(n, cur):
        if one_copy_stream:
            return enqueue_one(n, cur)
        # streams switched with set_stream (a stream context costs the host several times
        # more, and at decode rates the host's enqueue cost is what a step is waiting for)
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_done = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        for i in range(n):
            b = i % 2
            if i >= 2:
                s_in.wait_event(ev_done[i - 2])  # step i - 2 no longer reads buffer b
            torch.cuda.set_stream(s_in)
            h2d(i, b)
            torch.cuda.set_stream(cur)
            ev_in[i].record(s_in)
            cur.wait_event(ev_in[i])
            if i >= 2:
                cur.wait_event(ev_out[i - 2])  # step i - 2's result has left buffer b
            compute(i, b)
            ev_done[i].record(cur)
            s_out.wait_event(ev_done[i])
            torch.cuda.set_stream(s_out)
            d2h(i, b)
            torch.cuda.set_stream(cur)
            ev_out[i].record(s_out)

    cur = torch.cuda.current_stream()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if graph:
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            cap = torch.cuda.current_stream()
            s_in.wait_stream(cap)
            s_out.wait_stream(cap)
            enqueue(steps, cap)
            cap.wait_stream(s_in)
            cap.wait_stream(s_out)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        start.record(cur)
        g.replay()
        end.record(cur)
        torch.cuda.synchronize()
        return reduce_max(start.elapsed_time(end) / 1e3, dist, "cuda")

    def run(n, timed):
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        with torch.cuda.stream(s_in):
            if timed:
                gpu_head_start(torch)
            start.record(s_in)
        enqueue(n, cur)
        with torch.cuda.stream(s_last):
            end.record(s_last)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / 1e3

    run(warmup, False)
    return reduce_max(run(steps, True), dist, "cuda")


# ------------------------------------------------------------------ ranks (weak scaling)

def rank_work(cfg, rank):
    """The sequences and pool slots rank `rank` serves: every rank its own n_seqs
    sequences (own seeded streams) and its own pool; nothing is shared."""
    n, pool = cfg.n_seqs, cfg.pool_size
    return {"seqs": list(range(rank * n, (rank + 1) * n)),
            "pool_ids": list(range(rank * pool, (rank + 1) * pool))}


def reduce_max(value, dist, device):
    """Max of a float over all ranks (the timing rule); the value itself at one rank."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ the workload

def algorithmic_bytes_block(cfg, n):
    """Bytes a fused block decode launch over n sequences must move at minimum."""
    H, S, C, K = cfg.n_v_heads, cfg.state_size, cfg.conv_dim, cfg.conv_kernel
    state = 2 * n * H * S * S * 4
    other = (2 * n * C * (K - 1) * 4      # conv_state read + write
             + n * C * 4                  # qkv
             + 2 * n * H * S * 4          # z in, out
             + 2 * n * H * 4              # alpha, b
             + C * K * 4 + S * 4 + 2 * H * 4)  # conv weight, norm weight, dt, a
    return state, state + other


def cpu_sample_block(cfg, seqs, max_steps, budget_s):
    """Time the oracle (float build) on `seqs` sequences of the workload for up to
    max_steps steps or budget_s seconds. Returns (tokens/s, steps, seconds)."""
    import oracle
    st = I.block_static(cfg)
    state = I.state_pool(cfg, which=[int(s) for s in seqs]).astype(np.float32)
    conv = I.conv_state_pool(cfg, which=[int(s) for s in seqs]).astype(np.float32)
    steps_in = [I.block_step(cfg, s, seqs=seqs) for s in range(min(max_steps, 8))]
    oracle.sigmoid(np.zeros(1, np.float32), "f32")  # load the library outside the timing
    t0 = time.perf_counter()
    done = 0
    while done < max_steps:
        a = steps_in[done % len(steps_in)]
        oracle.block_decode(a["qkv"], st["conv_w"], conv, a["alpha"], a["b"], st["dt"], st["a"],
                            a["z"], st["norm_w"], state, cfg.n_k_heads, cfg.scale, cfg.eps,
                            cfg.eps, prec="f32")
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return len(seqs) * done / dt, done, dt


def cpu_sample_block_all_cores(cfg, budget_s):
    """The oracle's block on every host core at once: one thread per core, each stepping
    its own sequence (the oracle is C called through ctypes, which releases the GIL; the
    oracle itself is unchanged). Returns (tokens/s over all threads, threads, seconds)."""
    from concurrent.futures import ThreadPoolExecutor
    threads = max(1, min(os.cpu_count() or 1, cfg.n_seqs))
    with ThreadPoolExecutor(max_workers=threads) as ex:
        t0 = time.perf_counter()
        runs = list(ex.map(lambda n: cpu_sample_block(cfg, [n], 10 ** 6, budget_s),
                           range(threads)))
        dt = time.perf_counter() - t0
    return sum(r[0] for r in runs), threads, dt


def cpu_sample_scan(cfg, tokens, budget_s):
    """Time the oracle scan on one (sequence, v-head) unit for `tokens` tokens and
    scale to all units: returns tokens/s of the whole workload on one core."""
    import oracle
    x = I.recurrence_seq(cfg, 0, n_tokens=tokens)
    st = I.state_slot(cfg, 0)[:1][None].astype(np.float32)
    unit = {"q": x["q"][None, :, :1], "k": x["k"][None, :, :1], "v": x["v"][None, :, :1],
            "g": x["g"][None, :, :1], "beta": x["beta"][None, :, :1]}
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.recurrence(st, scale=cfg.scale, prec="f32", **unit)
        reps += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    # A token of the workload is one position of one sequence, which the oracle
    # advances through all n_v_heads units of that sequence: one core runs the
    # workload at (unit tokens per second) / n_v_heads tokens per second, for any
    # number of sequences.
    return reps * tokens / dt / cfg.n_v_heads, reps, dt


# ------------------------------------------------------------------ reference arm

def run_reference(args, cfg, rank, world):
    if rank != 0:
        return 0
    if args.workload == "spec_verify_64x4":
        vals = []
        for _ in range(args.warmup):
            cpu_sample_scan(cfg, SPEC_TOKENS, 0.0)
        for _ in range(args.steps):
            v, _, _ = cpu_sample_scan(cfg, SPEC_TOKENS, 0.2)
            vals.append(v)
        value = statistics.mean(vals)
        sample = (f"one (sequence, v-head) unit's {SPEC_TOKENS} tokens, repeated for 0.2 s per "
                  f"step, scaled to the {cfg.n_v_heads} v-heads of a token (the oracle's scan; "
                  "it keeps no snapshots)")
        ms = 1e3 * cfg.n_seqs * SPEC_TOKENS / value
        unit = "tokens/s"
    elif args.workload in ("prefill_scan_4x4096", "prefill_chunked_4x4096"):
        tokens = 256
        vals = []
        t_all = time.perf_counter()
        for _ in range(args.warmup):
            cpu_sample_scan(cfg, tokens, 0.0)
        for _ in range(args.steps):
            v, _, _ = cpu_sample_scan(cfg, tokens, 0.0)
            vals.append(v)
        value = statistics.mean(vals)
        sample = (f"one (sequence, v-head) unit of the 4x4096 scan, {tokens} tokens per step, "
                  f"scaled to the {cfg.n_v_heads} v-heads of a token")
        ms = 1e3 * cfg.n_seqs * cfg.n_tokens / value
        unit = "tokens/s"
    else:
        seqs = list(range(min(4, cfg.n_seqs)))
        cpu_sample_block(cfg, seqs, args.warmup, 1e9)
        t0 = time.perf_counter()
        value, done, dt = cpu_sample_block(cfg, seqs, args.steps, 1e9)
        sample = (f"{len(seqs)} of {cfg.n_seqs} sequences per step, {done} chained steps of the "
                  "fused block" + (" (one token of each sequence per step)" if cfg.cid == 2 else ""))
        ms = 1e3 * dt / done
        unit = "tokens/s"
    line = {
        "metric": METRIC, "value": value, "unit": unit, "impl": "reference", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "oracle": "plain C, float build, 1 thread"},
        "cpu_baseline": cpu_record(value, sample),
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm

def run_ours(args, cfg, rank, world, local_rank):
    import torch
    import gated_deltanet_linear_scan_gb300 as gdn

    dist = None
    if world > 1:
        import torch.distributed as dist
    gdn.build_if_needed()
    torch.cuda.set_device(local_rank)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
    stream = torch.cuda.current_stream()
    flush_w = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    flush_r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    pk, pk_kind = peaks()
    N = cfg.n_seqs

    def flush():
        # Evict the previous step's lines with a write larger than L2, then read
        # another buffer larger than L2 so the write-backs of that write happen here,
        # outside the timed region: the timed kernel starts with a cold, clean L2.
        flush_w.fill_(1.0)
        flush_r.sum()

    if args.workload == "prefill_block_4x4096":
        return run_ours_prefill(args, cfg, rank, world, dev, flush, pk, pk_kind, dist)
    if args.workload == "spec_verify_64x4":
        return run_ours_spec(args, cfg, rank, world, dev, flush, pk, pk_kind, dist)
    if args.workload == "prefill_varlen_16k":
        return run_ours_varlen(args, cfg, rank, world, dev, flush, pk, pk_kind, dist)
    if cfg.cid == 2:
        return run_ours_scan(args, cfg, rank, world, dev, flush, pk, pk_kind, dist)

    # This rank's sequences (its own seeded streams) and pool slots.
    work = rank_work(cfg, rank)
    seqs = work["seqs"]
    slots = I.slots(cfg)
    pool = cfg.pool_size
    st = I.block_static(cfg)
    d_st = {k: dev(v) for k, v in st.items()}
    state = dev(I.state_pool(cfg, which=work["pool_ids"]))
    conv = dev(I.conv_state_pool(cfg, which=work["pool_ids"]))
    d_slots = dev(slots) if slots is not None else None
    n_distinct = 8
    steps_in = [I.block_step(cfg, s, seqs=seqs) for s in range(n_distinct)]
    d_steps = [{k: dev(v) for k, v in a.items()} for a in steps_in]
    H, S = cfg.n_v_heads, cfg.state_size
    out = torch.empty(N, H, S, device="cuda")

    def launch(a, o):
        gdn.gdn_block_decode(a["qkv"], d_st["conv_w"], conv, a["alpha"], a["b"], d_st["dt"],
                             d_st["a"], a["z"], d_st["norm_w"], state, o, N, cfg.n_k_heads, H, S,
                             cfg.conv_kernel, cfg.scale, cfg.eps, cfg.eps, slots=d_slots,
                             pool=pool)

    kernel_ms, clk, t_wall = timed_steps(
        torch, stream, local_rank, dist, args.warmup, args.steps, lambda i: flush(),
        lambda i: launch(d_steps[i % n_distinct], out))
    gdn.gdn_device_error()
    total_s = reduce_max(sum(kernel_ms) / 1e3, dist, "cuda")
    step_us = sorted(1e3 * t for t in kernel_ms)
    tokens = world * N * args.steps
    value = tokens / total_s
    per_launch_s = total_s / args.steps
    state_b, alg_b = algorithmic_bytes_block(cfg, N)
    achieved = alg_b / per_launch_s / 1e9

    # ---- the same steps back to back, nothing between them (how a server runs them):
    # each step also writes back what the previous one left dirty in L2, and reads what
    # it left there; one span over all the steps
    b2b = [torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
    torch.cuda.synchronize()
    gpu_head_start(torch)
    b2b[0].record(stream)
    for i in range(args.steps):
        launch(d_steps[i % n_distinct], out)
    b2b[1].record(stream)
    torch.cuda.synchronize()
    gdn.gdn_device_error()
    b2b_s = reduce_max(b2b[0].elapsed_time(b2b[1]) / 1e3, dist, "cuda") / args.steps
    back_to_back = {"us_per_step": 1e6 * b2b_s, "tokens_per_s": world * N / b2b_s,
                    "hbm_gbs": alg_b / b2b_s / 1e9,
                    "hbm_frac_of_peak": alg_b / b2b_s / 1e9 / pk["hbm_gbs"],
                    "timing": "the steps with no flush between them, one event pair around "
                              "all of them"}

    # ---- the recurrence alone (gdn_recurrence_decode on precomputed q^, k^, v, g, beta),
    # on the same state and slots, timed the same way; reported beside the fused block.
    xr = I.recurrence_batch(cfg, seqs=seqs, n_tokens=n_distinct)
    r_steps = [{key: dev(xr[key][:, t]) for key in xr} for t in range(n_distinct)]
    y_rec = torch.empty(N, H, S, device="cuda")

    def launch_rec(a):
        gdn.gdn_recurrence_decode(state, a["q"], a["k"], a["v"], a["g"], a["beta"], y_rec, N,
                                  cfg.n_k_heads, H, S, cfg.scale, slots=d_slots, pool=pool)

    for w in range(args.warmup):
        flush()
        launch_rec(r_steps[w % n_distinct])
    rec_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    gpu_head_start(torch)
    for i in range(args.steps):
        flush()
        rec_ev[i][0].record(stream)
        launch_rec(r_steps[i % n_distinct])
        rec_ev[i][1].record(stream)
    torch.cuda.synchronize()
    rec_s = reduce_max(sum(e0.elapsed_time(e1) for e0, e1 in rec_ev) / 1e3, dist,
                       "cuda") / args.steps
    rec_bytes = state_b + N * (2 * cfg.n_k_heads * S + 2 * H * S + 2 * H) * 4
    rb = [torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
    torch.cuda.synchronize()
    gpu_head_start(torch)
    rb[0].record(stream)
    for i in range(args.steps):
        launch_rec(r_steps[i % n_distinct])
    rb[1].record(stream)
    torch.cuda.synchronize()
    rec_b2b_s = reduce_max(rb[0].elapsed_time(rb[1]) / 1e3, dist, "cuda") / args.steps
    recurrence_only = {"kernel": "gdn_recurrence_decode", "us_per_step": 1e6 * rec_s,
                       "state_gbs": state_b / rec_s / 1e9,
                       "hbm_gbs": rec_bytes / rec_s / 1e9,
                       "hbm_frac_of_peak": rec_bytes / rec_s / 1e9 / pk["hbm_gbs"],
                       "back_to_back_us_per_step": 1e6 * rec_b2b_s}

    # ---- the same with the factorised readout (gdn_recurrence_decode_2pass)
    tp_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps)]
    gpu_head_start(torch)
    for i in range(args.steps):
        flush()
        a = r_steps[i % n_distinct]
        tp_ev[i][0].record(stream)
        gdn.gdn_recurrence_decode_2pass(state, a["q"], a["k"], a["v"], a["g"], a["beta"], y_rec,
                                        N, cfg.n_k_heads, H, S, cfg.scale, slots=d_slots,
                                        pool=pool)
        tp_ev[i][1].record(stream)
    torch.cuda.synchronize()
    tp_s = reduce_max(sum(e0.elapsed_time(e1) for e0, e1 in tp_ev) / 1e3, dist,
                      "cuda") / args.steps
    recurrence_only["two_pass"] = {"kernel": "gdn_recurrence_decode_2pass",
                                   "us_per_step": 1e6 * tp_s,
                                   "hbm_gbs": rec_bytes / tp_s / 1e9,
                                   "hbm_frac_of_peak": rec_bytes / tp_s / 1e9 / pk["hbm_gbs"]}

    # ---- end to end: pinned host inputs -> device, the C-ABI call, output -> host.
    # A step's inputs (qkv, alpha, b, z) are packed in one pinned host buffer and
    # cross in one copy; the output comes back in one copy.
    keys = ["qkv", "alpha", "b", "z"]
    sizes = [steps_in[0][key].size for key in keys]
    h_packed = [torch.from_numpy(np.concatenate([np.ascontiguousarray(a[key]).ravel()
                                                 for key in keys])).pin_memory()
                for a in steps_in]
    d_packed = torch.empty(sum(sizes), device="cuda")
    views, off = {}, 0
    for key, sz in zip(keys, sizes):
        views[key] = d_packed[off:off + sz].view(d_steps[0][key].shape)
        off += sz
    h_out = torch.empty(N, H, S).pin_memory()
    h2d = sum(sizes) * 4
    d2h = h_out.numel() * 4
    e2e_note, e2e_graph_s = None, None
    if cfg.cid == 1:
        # one sequence: its 2 MiB state fits in L2, so every step is flushed and its copies
        # and launch run one after the other
        e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
        gpu_head_start(torch)
        for i in range(args.steps):
            flush()
            e2e_ev[i][0].record(stream)
            d_packed.copy_(h_packed[i % n_distinct], non_blocking=True)
            launch(views, out)
            h_out.copy_(out, non_blocking=True)
            e2e_ev[i][1].record(stream)
        torch.cuda.synchronize()
        e2e_s = reduce_max(sum(e0.elapsed_time(e1) for e0, e1 in e2e_ev) / 1e3, dist, "cuda")
        e2e_note = ("serial: each step's input copy, launch and result copy in turn on one "
                    "stream, L2 flushed before every step")
    else:
        packed = [d_packed, torch.empty_like(d_packed)]
        views2 = [views, {}]
        off = 0
        for key, sz in zip(keys, sizes):
            views2[1][key] = packed[1][off:off + sz].view(d_steps[0][key].shape)
            off += sz
        outs = [out, torch.empty_like(out)]
        h_outs = [h_out, torch.empty(N, H, S).pin_memory()]
        e2e_fns = (lambda i, b: packed[b].copy_(h_packed[i % n_distinct], non_blocking=True),
                   lambda i, b: launch(views2[b], outs[b]),
                   lambda i, b: h_outs[b].copy_(outs[b], non_blocking=True))
        e2e_s = pipelined_e2e(torch, dist, args.steps, *e2e_fns, one_copy_stream=True)
        e2e_note = PIPELINE_NOTE_ONE
        # the same pipelined steps captured once in a CUDA graph and replayed (how a server
        # runs decode steps without the host's per-call cost, ~60 us of Python a step here)
        e2e_graph_s = pipelined_e2e(torch, dist, args.steps, *e2e_fns, graph=True,
                                    one_copy_stream=True)

    # ---- one sequence: the serving form of the chain, a CUDA graph of 1000 consecutive
    # decode steps replayed as one unit (state and conv history carried, L2 warm: the
    # 2 MiB state stays resident from step to step). Reported beside the flushed value.
    chain = None
    if cfg.cid == 1:
        n_chain = 1000
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(n_chain):
                launch(d_steps[i % n_distinct], out)
        torch.cuda.synchronize()
        reps = []
        for _ in range(5):
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            graph.replay()
            g1.record(stream)
            torch.cuda.synchronize()
            reps.append(g0.elapsed_time(g1) / 1e3)
        reps.sort()
        chain_s = reduce_max(reps[len(reps) // 2], dist, "cuda")
        chain = {"steps": n_chain, "us_per_step": 1e6 * chain_s / n_chain,
                 "tokens_per_s": world * N * n_chain / chain_s, "replays": len(reps),
                 "l2": "warm (no flush inside the chain; the state stays L2-resident)"}
        del graph

    if rank != 0:
        return 0
    cpu = None
    if world == 1:
        sample_seqs = list(range(min(4, N)))
        v_cpu, done, dt = cpu_sample_block(cfg, sample_seqs, 10 ** 6, args.cpu_budget)
        cpu = cpu_record(v_cpu, f"{len(sample_seqs)} of {N} sequences, {done} chained steps "
                                f"of the block ({dt:.1f} s), plain C float build, 1 thread")
        v_all, threads, dt_all = cpu_sample_block_all_cores(cfg, min(3.0, args.cpu_budget))
        cpu["all_cores"] = {"value": v_all, "unit": "tokens/s", "cores": threads,
                            "sample": f"{threads} sequences, one thread each, stepping for "
                                      f"{dt_all:.1f} s (the same oracle)"}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded PCG64; N(0,1) qkv/z, state N(0,0.1^2), g~U(-2,-0.01))",
        "config": {"workload": args.workload, "n_seqs_per_gpu": N, "n_k_heads": cfg.n_k_heads,
                   "n_v_heads": H, "state_size": S, "conv_kernel": cfg.conv_kernel,
                   "pool_slots": pool, "kernel": "gdn_block_decode (fused, 1 launch/step)",
                   "l2": L2_NOTE,
                   "state_gbs": state_b / per_launch_s / 1e9,
                   "state_frac_of_peak": state_b / per_launch_s / 1e9 / pk["hbm_gbs"],
                   "step_us": {"mean": statistics.fmean(step_us), "min": step_us[0],
                               "median": statistics.median(step_us),
                               "p90": step_us[int(0.9 * (len(step_us) - 1))],
                               "max": step_us[-1]},
                   "wall_s_timed_loop": t_wall,
                   "back_to_back": back_to_back,
                   "recurrence_only": recurrence_only,
                   **({"graph_chain": chain} if chain else {})},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / pk["hbm_gbs"],
                     "traffic": ncu_traffic("block_decode_kernel", args.workload),
                     "algorithmic_bytes_per_launch": alg_b,
                     "peak_source": f"hbm_gbs ({pk_kind})"},
        "cpu_baseline": cpu,
        "e2e": {"value": tokens / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "timing": e2e_note,
                "graph_replay": None if e2e_graph_s is None else {
                    "value": tokens / e2e_graph_s, "unit": "tokens/s",
                    "timing": "the same pipelined steps captured once in a CUDA graph and "
                              "replayed (first input copy to last result copy)"}},
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours_scan(args, cfg, rank, world, dev, flush, pk, pk_kind, dist):
    import torch
    import gated_deltanet_linear_scan_gb300 as gdn
    stream = torch.cuda.current_stream()
    N, T, H, Hk, S = cfg.n_seqs, cfg.n_tokens, cfg.n_v_heads, cfg.n_k_heads, cfg.state_size
    seqs = rank_work(cfg, rank)["seqs"]
    x = I.recurrence_batch(cfg, seqs=seqs)
    d = {k: dev(v) for k, v in x.items()}
    state0 = dev(I.state_pool(cfg, which=seqs))
    state = state0.clone()
    y = torch.empty(N, T, H, S, device="cuda")

    chunked = args.workload == "prefill_chunked_4x4096"
    ws = None
    if chunked:
        ws = torch.empty(gdn.gdn_recurrence_scan_chunked_ws_size(N, T, H, S) // 4, device="cuda")

    def launch(dd=None, yy=None):
        dd = d if dd is None else dd
        yy = y if yy is None else yy
        if chunked:
            gdn.gdn_recurrence_scan_chunked_ws(state, dd["q"], dd["k"], dd["v"], dd["g"],
                                               dd["beta"], yy, N, T, Hk, H, S, cfg.scale, ws)
        else:
            gdn.gdn_recurrence_scan(state, dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], yy,
                                    N, T, Hk, H, S, cfg.scale)

    def before(i):
        state.copy_(state0)
        flush()

    step_ms, clk, _ = timed_steps(torch, stream, torch.cuda.current_device(), dist,
                                  args.warmup, args.steps, before, lambda i: launch())
    gdn.gdn_device_error()
    total_s = reduce_max(sum(step_ms) / 1e3, dist, "cuda")
    per = total_s / args.steps
    tokens = world * N * T * args.steps

    # ---- end to end: q, k, v, g, beta from pinned host memory, the call (the state reset
    # first), y back; pipelined over double buffers
    keys = ["q", "k", "v", "g", "beta"]
    h_in = {key: torch.from_numpy(np.ascontiguousarray(x[key])).pin_memory() for key in keys}
    h_y = [torch.empty(N, T, H, S).pin_memory() for _ in range(2)]
    h2d = sum(h_in[key].numel() for key in keys) * 4
    d2h = h_y[0].numel() * 4
    d_in = [{key: d[key] for key in keys}, {key: torch.empty_like(d[key]) for key in keys}]
    ys = [y, torch.empty_like(y)]

    def e2e_in(i, b):
        for key in keys:
            d_in[b][key].copy_(h_in[key], non_blocking=True)

    def e2e_step(i, b):
        state.copy_(state0)
        launch(d_in[b], ys[b])

    e2e_s = pipelined_e2e(torch, dist, args.steps, e2e_in, e2e_step,
                          lambda i, b: h_y[b].copy_(ys[b], non_blocking=True))
    flops = 7.0 * N * T * H * S * S
    props = torch.cuda.get_device_properties(0)
    mhz = clk["sm_mhz"] or pk.get("sm_max_mhz", 2070.0)
    fp32_peak = props.multi_processor_count * 128 * 2 * mhz * 1e6 / 1e12
    achieved = flops / per / 1e12
    extra = {}
    if chunked:
        # the two phases timed apart (the dominant, tensor-core one for the roofline), and
        # the one-kernel form on the same inputs for comparison
        prep_s, adv_s = time_chunked_phases(gdn, torch, stream, state, state0, d, y,
                                            (N, T, Hk, H, S), cfg.scale, ws, args.steps, flush)
        one_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
        gpu_head_start(torch)
        for i in range(args.steps):
            state.copy_(state0)
            flush()
            one_ev[i][0].record(stream)
            gdn.gdn_recurrence_scan_chunked(state, d["q"], d["k"], d["v"], d["g"], d["beta"], y,
                                            N, T, Hk, H, S, cfg.scale)
            one_ev[i][1].record(stream)
        torch.cuda.synchronize()
        one_s = sum(e0.elapsed_time(e1) for e0, e1 in one_ev) / 1e3 / args.steps
        # the snapshot form (prefix caching): the state every 16 chunks (512 positions)
        every = 16
        n_snaps = gdn.gdn_chunked_snapshot_count(T, every)
        snaps = torch.empty(N, n_snaps, H, S, S, device="cuda")
        snap_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
        gpu_head_start(torch)
        for i in range(args.steps):
            state.copy_(state0)
            flush()
            snap_ev[i][0].record(stream)
            gdn.gdn_recurrence_scan_chunked_snapshots(state, d["q"], d["k"], d["v"], d["g"],
                                                      d["beta"], y, snaps, every, N, T, Hk, H, S,
                                                      cfg.scale, ws)
            snap_ev[i][1].record(stream)
        torch.cuda.synchronize()
        gdn.gdn_device_error()
        snap_s = sum(e0.elapsed_time(e1) for e0, e1 in snap_ev) / 1e3 / args.steps
        snap_bytes = snaps.numel() * 4
        del snaps
        tf = chunked_tensor_flops(N, T, H)
        pf = chunk_prepare_flops(N, T, Hk, H)
        bf16_peak = pk.get("bf16_tflops", 1900.0)
        mf = chunked_method_flops(N * ((T + 31) // 32), H)
        roofline = {"bound": "tensor", "kernel": "chunk_state_kernel (gdn_chunked_advance)",
                    "achieved": mf / adv_s / 1e12, "peak": bf16_peak,
                    "unit": "TFLOP/s", "frac": mf / adv_s / 1e12 / bf16_peak,
                    "traffic": ncu_traffic("chunk_state_kernel", args.workload),
                    "flops_per_launch": mf,
                    "flops_note": "the method's own contraction flops (each product once); "
                                  "the kernel issues 3 bf16 passes per product (3xBF16)",
                    "peak_source": f"bf16_tflops ({pk_kind})"}
        extra = {"advance_ms": 1e3 * adv_s, "prepare_ms": 1e3 * prep_s,
                 "advance_tensor_issued_tflops": tf / adv_s / 1e12,
                 "prepare_fp32_tflops": pf / prep_s / 1e12,
                 "prepare_frac_of_fp32_pipes": pf / prep_s / 1e12 / fp32_peak,
                 "one_kernel_form_ms": 1e3 * one_s,
                 "snapshot_form": {"call": "gdn_recurrence_scan_chunked_snapshots",
                                   "snap_every_chunks": every, "snapshots_per_seq": n_snaps,
                                   "snapshot_bytes": snap_bytes, "ms": 1e3 * snap_s,
                                   "over_plain_ms": 1e3 * (snap_s - per)},
                 "workspace_bytes": ws.numel() * 4}
    else:
        roofline = {"bound": "alu", "achieved": achieved, "peak": fp32_peak, "unit": "TFLOP/s",
                    "frac": achieved / fp32_peak,
                    "traffic": ncu_traffic("recurrence_scan_kernel", args.workload),
                    "peak_source": "FP32 FMA pipes: SMs x 128 lanes x 2 flop x median SM clock"}
    if rank != 0:
        return 0
    cpu = None
    if world == 1:
        v_cpu, reps, dt = cpu_sample_scan(cfg, 256, args.cpu_budget)
        cpu = cpu_record(v_cpu, f"one (sequence, v-head) unit, 256 tokens x {reps} reps "
                                f"({dt:.1f} s), scaled to the {H} v-heads of a token; plain C "
                                "float build, 1 thread")
    line = {
        "metric": METRIC, "value": tokens / total_s, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * per,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded PCG64; unit q/k, g~U(-0.5,-0.001))",
        "config": {"workload": args.workload, "n_seqs": N, "n_tokens": T, "n_k_heads": Hk,
                   "n_v_heads": H, "state_size": S,
                   "kernel": ("gdn_recurrence_scan_chunked_ws (2 launches: chunk preparation, "
                              "tensor-core state advance)") if chunked else "gdn_recurrence_scan",
                   "l2": L2_NOTE,
                   "method_fp32_tflops": achieved,
                   "method_fp32_frac_of_fp32_pipe_peak": achieved / fp32_peak, **extra},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": tokens / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "timing": PIPELINE_NOTE},
        "gpu_launches": (2 if chunked else 1) * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours_spec(args, cfg, rank, world, dev, flush, pk, pk_kind, dist):
    """Speculative-decoding verification: the delta-rule scan over 4 draft tokens of each
    of 64 sequences, keeping the state after every token (gdn_recurrence_scan_snapshots),
    so the caller can roll back to the last accepted token. HBM-bound: the state is read
    and written once and written again as a snapshot after every token."""
    import torch
    import gated_deltanet_linear_scan_gb300 as gdn
    stream = torch.cuda.current_stream()
    N, T, H, Hk, S = cfg.n_seqs, cfg.n_tokens, cfg.n_v_heads, cfg.n_k_heads, cfg.state_size
    seqs = rank_work(cfg, rank)["seqs"]
    x = I.recurrence_batch(cfg, seqs=seqs)
    d = {k: dev(v) for k, v in x.items()}
    state0 = dev(I.state_pool(cfg, which=seqs))
    state = state0.clone()
    y = torch.empty(N, T, H, S, device="cuda")
    snaps = torch.empty(N, T, H, S, S, device="cuda")

    def launch(dd=None, yy=None):
        dd = d if dd is None else dd
        yy = y if yy is None else yy
        gdn.gdn_recurrence_scan_snapshots(state, dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"],
                                          yy, snaps, N, T, Hk, H, S, cfg.scale)

    def before(i):
        state.copy_(state0)
        flush()

    step_ms, clk, _ = timed_steps(torch, stream, torch.cuda.current_device(), dist,
                                  args.warmup, args.steps, before, lambda i: launch())
    gdn.gdn_device_error()
    total_s = reduce_max(sum(step_ms) / 1e3, dist, "cuda")
    per = total_s / args.steps
    tokens = world * N * T * args.steps
    # algorithmic bytes of one launch: the state read and written once, a snapshot per
    # token, and the per-token activations (q, k per k-head; v, y per v-head; g, beta)
    state_bytes = N * H * (2 + T) * S * S * 4
    alg_bytes = state_bytes + N * T * (2 * Hk * S + 2 * H * S + 2 * H) * 4
    achieved = alg_bytes / per / 1e9

    # ---- the rollback that follows a verification (gdn_snapshot_restore), timed the same
    # way: every sequence back to a seeded accepted count in [1, T]
    acc = torch.from_numpy(np.random.default_rng(cfg.seed).integers(1, T + 1, N)
                           .astype(np.int32)).cuda()
    rs_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps)]
    gpu_head_start(torch)
    for i in range(args.steps):
        flush()
        rs_ev[i][0].record(stream)
        gdn.gdn_snapshot_restore(state, snaps, acc, N, T, H, S)
        rs_ev[i][1].record(stream)
    torch.cuda.synchronize()
    gdn.gdn_device_error()
    rs_s = reduce_max(sum(e0.elapsed_time(e1) for e0, e1 in rs_ev) / 1e3, dist, "cuda") / args.steps
    rs_bytes = 2 * N * H * S * S * 4
    restore = {"kernel": "gdn_snapshot_restore", "us_per_call": 1e6 * rs_s,
               "hbm_gbs": rs_bytes / rs_s / 1e9, "hbm_frac_of_peak": rs_bytes / rs_s / 1e9 / pk["hbm_gbs"]}

    # ---- end to end, a serving step: q, k, v, g, beta and the accepted counts from pinned
    # host memory, the verification, the rollback to the accepted counts (the seeded ones
    # above stand in for the verifier's), y back (the snapshots stay on the device, where
    # the rollback reads them); pipelined over double buffers
    keys = ["q", "k", "v", "g", "beta"]
    h_in = {key: torch.from_numpy(np.ascontiguousarray(x[key])).pin_memory() for key in keys}
    h_acc = acc.cpu().pin_memory()
    h_y = [torch.empty(N, T, H, S).pin_memory() for _ in range(2)]
    h2d = sum(h_in[key].numel() for key in keys) * 4 + h_acc.numel() * 4
    d2h = h_y[0].numel() * 4
    d_in = [{key: d[key] for key in keys}, {key: torch.empty_like(d[key]) for key in keys}]
    d_acc = [acc, torch.empty_like(acc)]
    ys = [y, torch.empty_like(y)]

    def e2e_in(i, b):
        for key in keys:
            d_in[b][key].copy_(h_in[key], non_blocking=True)
        d_acc[b].copy_(h_acc, non_blocking=True)

    def e2e_step(i, b):
        launch(d_in[b], ys[b])
        gdn.gdn_snapshot_restore(state, snaps, d_acc[b], N, T, H, S)

    e2e_s = pipelined_e2e(torch, dist, args.steps, e2e_in, e2e_step,
                          lambda i, b: h_y[b].copy_(ys[b], non_blocking=True))
    if rank != 0:
        return 0
    cpu = None
    if world == 1:
        v_cpu, reps, dt = cpu_sample_scan(cfg, T, args.cpu_budget)
        cpu = cpu_record(v_cpu, f"one (sequence, v-head) unit's {T} tokens x {reps} reps "
                                f"({dt:.1f} s), scaled to the {H} v-heads of a token; the "
                                "oracle's scan keeps no snapshots; plain C float build, 1 thread")
    line = {
        "metric": METRIC, "value": tokens / total_s, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * per,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded PCG64; unit q/k, g~U(-2,-0.01))",
        "config": {"workload": args.workload, "n_seqs": N, "n_tokens": T, "n_k_heads": Hk,
                   "n_v_heads": H, "state_size": S,
                   "kernel": "gdn_recurrence_scan_snapshots (state after every token)",
                   "l2": L2_NOTE, "snapshot_bytes": snaps.numel() * 4,
                   "algorithmic_bytes_per_step": alg_bytes,
                   "state_gbs": state_bytes / per / 1e9, "restore": restore},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                     "traffic": ncu_traffic("recurrence_scan_kernel", args.workload),
                     "kernel": "recurrence_scan_kernel<4, true>",
                     "peak_source": f"hbm_gbs ({pk_kind})"},
        "cpu_baseline": cpu,
        "e2e": {"value": tokens / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "timing": PIPELINE_NOTE + "; a step is the verification and the rollback to "
                          "its accepted counts (gdn_snapshot_restore)"},
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours_prefill(args, cfg, rank, world, dev, flush, pk, pk_kind, dist):
    """The whole block over 4 sequences x 4096 tokens (gdn_block_prefill)."""
    import torch
    import gated_deltanet_linear_scan_gb300 as gdn
    stream = torch.cuda.current_stream()
    N, T, H, Hk, S = cfg.n_seqs, cfg.n_tokens, cfg.n_v_heads, cfg.n_k_heads, cfg.state_size
    seqs = rank_work(cfg, rank)["seqs"]
    per = [I.prefill_seq(cfg, n) for n in seqs]
    d = {key: dev(np.stack([p_[key] for p_ in per])) for key in per[0]}
    st = {k_: dev(v_) for k_, v_ in I.block_static(cfg).items()}
    state0 = dev(I.state_pool(cfg, which=seqs))
    conv0 = dev(I.conv_state_pool(cfg, which=seqs))
    state, conv = state0.clone(), conv0.clone()
    out = torch.empty(N, T, H, S, device="cuda")
    ws = torch.empty(gdn.gdn_block_prefill_chunked_workspace_size(N, T, Hk, H, S) // 4 + 64,
                     device="cuda")

    def launch(dd=None, oo=None):
        dd = d if dd is None else dd
        oo = out if oo is None else oo
        gdn.gdn_block_prefill_chunked(dd["qkv"], st["conv_w"], conv, dd["alpha"], dd["b"],
                                      st["dt"], st["a"], dd["z"], st["norm_w"], state, oo, N, T,
                                      Hk, H, S, cfg.conv_kernel, cfg.scale, cfg.eps, cfg.eps, ws)

    def reset():
        state.copy_(state0)
        conv.copy_(conv0)

    def before(i):
        reset()
        flush()

    step_ms, clk, _ = timed_steps(torch, stream, torch.cuda.current_device(), dist,
                                  args.warmup, args.steps, before, lambda i: launch())
    gdn.gdn_device_error()
    total_s = reduce_max(sum(step_ms) / 1e3, dist, "cuda")
    per_s = total_s / args.steps
    tokens = world * N * T * args.steps

    # ---- the dominant kernel alone: the tensor-core state advance of the chunked scan
    # over the same intermediates (made once by the stand-alone step entry points),
    # timed on the same stream.
    C = (2 * Hk + H) * S
    conv_out = torch.empty(N, T, C, device="cuda")
    q = torch.empty(N, T, Hk, S, device="cuda")
    k = torch.empty_like(q)
    v = torch.empty(N, T, H, S, device="cuda")
    g = torch.empty(N, T, H, device="cuda")
    beta = torch.empty_like(g)
    y = torch.empty_like(out)
    reset()
    gdn.gdn_conv1d_silu_seq(d["qkv"], st["conv_w"], conv, conv_out, N, T, C, cfg.conv_kernel)
    gdn.gdn_qkv_split_norm(conv_out, q, k, v, N * T, Hk, H, S, cfg.eps)
    gdn.gdn_decay_gate(d["alpha"], st["dt"], st["a"], g, H, N * T)
    gdn.gdn_beta_sigmoid(d["b"], beta, N * T * H)
    scan_ws = torch.empty(gdn.gdn_recurrence_scan_chunked_ws_size(N, T, H, S) // 4,
                          device="cuda")
    prep_s, adv_s = time_chunked_phases(gdn, torch, stream, state, state0,
                                        {"q": q, "k": k, "v": v, "g": g, "beta": beta}, y,
                                        (N, T, Hk, H, S), cfg.scale, scan_ws, args.steps, flush)
    adv_s = reduce_max(adv_s, dist, "cuda")
    del scan_ws

    # ---- end to end: qkv, alpha, b, z from pinned host memory, the call (state and conv
    # history reset first), out back; pipelined over double buffers
    keys = ["qkv", "alpha", "b", "z"]
    h_in = {key: d[key].cpu().pin_memory() for key in keys}
    h_out = [torch.empty(N, T, H, S).pin_memory() for _ in range(2)]
    h2d = sum(h_in[key].numel() for key in keys) * 4
    d2h = h_out[0].numel() * 4
    d_in = [{key: d[key] for key in keys}, {key: torch.empty_like(d[key]) for key in keys}]
    outs = [out, torch.empty_like(out)]

    def e2e_in(i, b):
        for key in keys:
            d_in[b][key].copy_(h_in[key], non_blocking=True)

    def e2e_step(i, b):
        reset()
        launch(d_in[b], outs[b])

    e2e_s = pipelined_e2e(torch, dist, args.steps, e2e_in, e2e_step,
                          lambda i, b: h_out[b].copy_(outs[b], non_blocking=True))

    flops = 7.0 * N * T * H * S * S
    mf = chunked_method_flops(N * ((T + 31) // 32), H)
    bf16_peak = pk.get("bf16_tflops", 1900.0)
    props = torch.cuda.get_device_properties(0)
    mhz = clk["sm_mhz"] or pk.get("sm_max_mhz", 2070.0)
    fp32_peak = props.multi_processor_count * 128 * 2 * mhz * 1e6 / 1e12
    if rank != 0:
        return 0
    cpu = None
    if world == 1:
        v_cpu, done, dt = cpu_sample_block(cfg, [int(seqs[0])], 10 ** 6, args.cpu_budget)
        cpu = cpu_record(v_cpu, f"1 of {N} sequences, {done} consecutive tokens through the "
                                f"block ({dt:.1f} s; per-token work is the same in every "
                                "sequence), plain C float build, 1 thread")
    line = {
        "metric": METRIC, "value": tokens / total_s, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * per_s,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded PCG64; N(0,1) qkv/z, g~U(-0.5,-0.001))",
        "config": {"workload": args.workload, "n_seqs": N, "n_tokens": T, "n_k_heads": Hk,
                   "n_v_heads": H, "state_size": S, "conv_kernel": cfg.conv_kernel,
                   "kernel": "gdn_block_prefill_chunked (5 launches: conv scan with the q/k "
                             "split-norm, gate and beta, chunk preparation, tensor-core state "
                             "advance, gated norm)", "l2": L2_NOTE,
                   "workspace_bytes": ws.numel() * 4,
                   "scan_prepare_ms": 1e3 * prep_s, "scan_advance_ms": 1e3 * adv_s,
                   "method_fp32_tflops_of_scan": flops / (prep_s + adv_s) / 1e12,
                   "fp32_pipe_peak_tflops": fp32_peak},
        "roofline": {"bound": "tensor", "kernel": "chunk_state_kernel (gdn_chunked_advance)",
                     "achieved": mf / adv_s / 1e12, "peak": bf16_peak, "unit": "TFLOP/s",
                     "frac": mf / adv_s / 1e12 / bf16_peak,
                     "traffic": ncu_traffic("chunk_state_kernel", "prefill_chunked_4x4096"),
                     "flops_per_launch": mf,
                     "flops_note": "the method's own contraction flops (each product once); "
                                   "the kernel issues 3 bf16 passes per product (3xBF16)",
                     "peak_source": f"bf16_tflops ({pk_kind})"},
        "cpu_baseline": cpu,
        "e2e": {"value": tokens / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "timing": PIPELINE_NOTE},
        "gpu_launches": 5 * args.steps, "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours_varlen(args, cfg, rank, world, dev, flush, pk, pk_kind, dist):
    """A ragged prefill batch: sequences of mixed lengths (seeded, log-uniform in [1, 4096],
    16384 tokens in all) packed token-major through gdn_block_prefill_chunked_varlen in one
    call per step (conv + q/k split-norm, gate, beta, the two-phase chunked scan, gated
    norm). The state and conv history of every sequence start fresh each step."""
    import torch
    import gated_deltanet_linear_scan_gb300 as gdn
    stream = torch.cuda.current_stream()
    H, Hk, S, K = cfg.n_v_heads, cfg.n_k_heads, cfg.state_size, cfg.conv_kernel
    lengths = I.ragged_lengths(cfg, VARLEN_TOKENS)
    N, total, maxt = len(lengths), sum(lengths), max(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    vcfg = I.get_config(2, n_seqs=N)
    first = rank * N  # this rank's sequences: their own seeded streams
    per = [I.prefill_seq(vcfg, first + n, n_tokens=L) for n, L in enumerate(lengths)]
    d = {key: dev(np.concatenate([p_[key] for p_ in per])) for key in per[0]}
    d_cu = dev(cu)
    st = {k_: dev(v_) for k_, v_ in I.block_static(vcfg).items()}
    state0 = dev(I.state_pool(vcfg, which=range(first, first + N)))
    conv0 = dev(I.conv_state_pool(vcfg, which=range(first, first + N)))
    state, conv = state0.clone(), conv0.clone()
    out = torch.empty(total, H, S, device="cuda")
    ws = torch.empty(gdn.gdn_block_prefill_chunked_varlen_workspace_size(N, total, Hk, H, S) // 4
                     + 64, device="cuda")

    def launch(dd=None, oo=None, cu_d=None):
        dd = d if dd is None else dd
        oo = out if oo is None else oo
        cu_d = d_cu if cu_d is None else cu_d
        gdn.gdn_block_prefill_chunked_varlen(dd["qkv"], st["conv_w"], conv, dd["alpha"],
                                             dd["b"], st["dt"], st["a"], dd["z"], st["norm_w"],
                                             state, oo, cu_d, N, total, maxt, Hk, H, S, K,
                                             cfg.scale, cfg.eps, cfg.eps, ws)

    def before(i):
        state.copy_(state0)
        conv.copy_(conv0)
        flush()

    step_ms, clk, _ = timed_steps(torch, stream, torch.cuda.current_device(), dist,
                                  args.warmup, args.steps, before, lambda i: launch())
    gdn.gdn_device_error()
    total_s = reduce_max(sum(step_ms) / 1e3, dist, "cuda")
    per_s = total_s / args.steps
    tokens = world * total * args.steps

    # ---- the chunked scan alone (both phases, the dominant part of the step) over the
    # same lengths, on the recurrence inputs of the scan workloads (unit q, k): method
    # flops per time
    rx = [I.recurrence_seq(vcfg, first + n, n_tokens=L) for n, L in enumerate(lengths)]
    rd = {key: dev(np.concatenate([p_[key] for p_ in rx])) for key in rx[0]}
    q, k, v, g, beta = rd["q"], rd["k"], rd["v"], rd["g"], rd["beta"]
    y = torch.empty_like(out)
    scan_ws = torch.empty(gdn.gdn_recurrence_scan_chunked_varlen_ws_size(N, total, H, S) // 4,
                          device="cuda")
    scan_ms, _, _ = timed_steps(
        torch, stream, torch.cuda.current_device(), dist, 3, args.steps, lambda i: before(i),
        lambda i: gdn.gdn_recurrence_scan_chunked_varlen(state, q, k, v, g, beta, y, d_cu, N,
                                                         total, maxt, Hk, H, S, cfg.scale,
                                                         workspace=scan_ws))
    scan_s = reduce_max(sum(scan_ms) / 1e3, dist, "cuda") / args.steps
    del scan_ws
    n_chunks = sum((L + 31) // 32 for L in lengths)
    mflops = chunked_method_flops(n_chunks, H)
    bf16_peak = pk.get("bf16_tflops", 1900.0)

    # ---- end to end: qkv, alpha, b, z and cu_seqlens from pinned host memory, the call
    # (state and conv history reset first), out back; pipelined over double buffers
    keys = ["qkv", "alpha", "b", "z"]
    h_in = {key: d[key].cpu().pin_memory() for key in keys}
    h_cu = torch.from_numpy(cu).pin_memory()
    h_out = [torch.empty(total, H, S).pin_memory() for _ in range(2)]
    h2d = sum(h_in[key].numel() for key in keys) * 4 + h_cu.numel() * 4
    d2h = h_out[0].numel() * 4
    d_in = [{key: d[key] for key in keys}, {key: torch.empty_like(d[key]) for key in keys}]
    cus = [d_cu, torch.empty_like(d_cu)]
    outs = [out, torch.empty_like(out)]

    def e2e_in(i, b):
        for key in keys:
            d_in[b][key].copy_(h_in[key], non_blocking=True)
        cus[b].copy_(h_cu, non_blocking=True)

    def e2e_step(i, b):
        state.copy_(state0)
        conv.copy_(conv0)
        launch(d_in[b], outs[b], cus[b])

    e2e_s = pipelined_e2e(torch, dist, args.steps, e2e_in, e2e_step,
                          lambda i, b: h_out[b].copy_(outs[b], non_blocking=True))
    if rank != 0:
        return 0
    cpu = None
    if world == 1:
        v_cpu, done, dt = cpu_sample_block(vcfg, [0], 10 ** 6, args.cpu_budget)
        cpu = cpu_record(v_cpu, f"1 sequence, {done} consecutive tokens through the block "
                                f"({dt:.1f} s; per-token work does not depend on the length), "
                                "plain C float build, 1 thread")
    line = {
        "metric": METRIC, "value": tokens / total_s, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * per_s,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded PCG64; N(0,1) qkv/z, g~U(-0.5,-0.001); lengths "
                "log-uniform in [1, 4096])",
        "config": {"workload": args.workload, "n_seqs": N, "total_tokens": total,
                   "max_tokens": maxt, "lengths": lengths, "n_k_heads": Hk, "n_v_heads": H,
                   "state_size": S, "conv_kernel": K,
                   "kernel": "gdn_block_prefill_chunked_varlen (5 launches: conv scan with the "
                             "q/k split-norm, gate and beta, chunk preparation, tensor-core "
                             "state advance, gated norm)", "l2": L2_NOTE,
                   "workspace_bytes": ws.numel() * 4, "scan_ms": 1e3 * scan_s,
                   "chunks": n_chunks},
        "roofline": {"bound": "tensor",
                     "kernel": "chunk_prepare_kernel + chunk_state_kernel "
                               "(gdn_recurrence_scan_chunked_varlen, timed together)",
                     "achieved": mflops / scan_s / 1e12, "peak": bf16_peak, "unit": "TFLOP/s",
                     "frac": mflops / scan_s / 1e12 / bf16_peak,
                     "traffic": ncu_traffic("chunk_state_kernel", args.workload),
                     "traffic_note": "both kernels of the ragged chunked scan, per call",
                     "flops_per_launch": mflops,
                     "flops_note": "the method's own contraction flops (each product once); "
                                   "the kernels issue 3 bf16 passes per product (3xBF16)",
                     "peak_source": f"bf16_tflops ({pk_kind})"},
        "cpu_baseline": cpu,
        "e2e": {"value": tokens / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "timing": PIPELINE_NOTE},
        "gpu_launches": 5 * args.steps, "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="batched_decode_64")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle time for the cpu_baseline sample")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != world:
        # one process per GPU: N > 1 needs a launcher that starts N ranks (torchrun)
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; run N > 1 as "
              f"python -m torch.distributed.run --nproc-per-node {args.gpus} bench.py "
              f"--gpus {args.gpus} ...", file=sys.stderr)
        return 2
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    cfg = I.get_config(WORKLOADS[args.workload], **OVERRIDES.get(args.workload, {}))
    if args.impl == "reference":
        return run_reference(args, cfg, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        return run_ours(args, cfg, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
