#!/usr/bin/env python
"""Benchmark of usp_attention, the whole context-parallel attention path, on synthetic inputs.

One step = one usp_attention call on the workload: Q, K, V read in place through each virtual
rank's tensor maps (the reorder and the seq->head all-to-all are addressing), the attention launch
over every chunk pair or ring chain, the LSE merge of ring partials when the ring steps run
separately, and O and LSE written in the global layout (the head->seq all-to-all as store
addressing).  Inputs are resident in HBM when the timed region starts; the
L2 cache is flushed between steps (outside the step's events) because the inputs of the default
workload fit in L2.  The flush READS a 256 MiB buffer: a flush that writes would leave up to the
whole L2 dirty, and writing those lines back would then be charged to the timed kernels.  Each
step is bracketed by one pair of events; a short spin kernel after the flush lets the host enqueue
the step before the GPU reaches the start event, so the step's time is device execution (host
planning and launch latency are in the e2e figure).  The per-phase breakdown comes from a second
loop whose events sit between the phases.  Times come from CUDA events on the launching stream.

  value     attention TFLOP/s of the whole step: algorithmic FLOPs 4 B H D x (visible query/key
            pairs) over the step's device time (all phases), summed over ranks.
  e2e       the same metric through the C ABI with the inputs in pinned host memory: each step
            copies Q, K, V host->device, runs usp_attention and copies O and LSE back.  `value` is
            pipelined as a caller serving a stream of requests runs it (two device buffer sets;
            step i's copy-in overlaps step i-1's attention and copy-out); `serial_value` runs one
            step at a time on one stream.  `host_link` = the copies' rates in this run (each
            direction alone and both at once), `pipelined_estimate` = the pipelined figure they
            predict (the host link is shared with other jobs, so it varies from run to run), and
            `serial_stage_ms` / `pipelined_stage_ms` = each stage's median and maximum time.
  roofline  the partial-attention phase alone against the measured dense bf16 tensor peak: the
            sustained figure when the timed steps add up to a long run (>= 0.25 s of device time,
            as for the 64K ring), the burst figure otherwise; both fractions are in the line.
  relayout_merge  GB/s of the step's bandwidth-bound phases, plus separately timed standalone
            measurements of the re-layout entry points on the workload's tensors and of the LSE
            merge entry point on two ring partials of the workload's size.

Multi-GPU: the method is partitioned onto virtual ranks of one GPU, so N GPUs run N independent
replicas (weak scaling); the only cross-rank traffic is the timing reduction.

``--impl reference`` times the fp64 CPU oracle (the reference arm: a deliberately slow program)
on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention TFLOP/s & % bf16 tensor peak; re-layout+merge GB/s & % HBM BW"
DEFAULT_WORKLOAD = "llm_64k_ring8_zigzag"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_HBM_GBS = 8000.0
# A timed region at least this long (device time of all timed steps) is a kernel timed inside a
# long run: the roofline then divides by the sustained bf16 peak instead of the burst one.
SUSTAINED_MS = 250.0

# DRAM bytes (read + write) per launch of the attention kernel, dram__bytes_read.sum +
# dram__bytes_write.sum from one ncu capture of that workload's launch, with the hash of the kernel
# code they were taken on (kernel_hash); reported as null once that code changes.
ATTN_TRAFFIC = {
    # one full-size launch: dram__bytes_read.sum 1697439744 + dram__bytes_write.sum 574841344
    "llm_64k_ring8_zigzag": {"bytes": 1697439744 + 574841344, "kernel_hash": "75f1b74594938e16"},
}
L2_BYTES = 129e6


def code_of(src: str) -> str:
    """C/C++ source without its comments and whitespace (the code the compiler sees)."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return re.sub(r"\s+", "", src)


def kernel_hash() -> str:
    """Hash of the attention kernel's code (attn.cu and ptx.cuh without comments or whitespace):
    the recorded DRAM traffic stays attached to the code it was measured on."""
    h = hashlib.sha256()
    for f in ("attn.cu", "ptx.cuh"):
        with open(os.path.join(ROOT, "sequence_attention_tcgen05_gb300", "csrc", f)) as fh:
            h.update(code_of(fh.read()).encode())
    return h.hexdigest()[:16]


def roofline_peak(peaks: dict, timed_ms: float):
    """(bf16 peak, sustained?) for a timed region of `timed_ms` ms of device time: the burst peak
    for a kernel timed alone, the sustained one (cuBLAS over a seconds-long loop under the power
    cap) for a kernel timed inside a long run of steps."""
    sustained = timed_ms >= SUSTAINED_MS
    return (peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]), sustained


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ------------------------------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def reduce_max(x: float, device=None) -> float:
    """Max over ranks of a host scalar (identity on one process)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index] if device is not None else None)
        else:
            dist.barrier()


def aggregate(units_per_rank: float, seconds_this_rank: float, world: int, device=None):
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    t = reduce_max(seconds_this_rank, device)
    return world * units_per_rank / t, t


# ------------------------------------------------------------------------------------------------
# clocks
# ------------------------------------------------------------------------------------------------

CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(prefix="usp_clocks_", suffix=".csv")
        self.proc = None
        self.gpu = gpu_index
        self.marks = []

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
                except Exception:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        t0, t1 = (self.marks[0], self.marks[-1]) if len(self.marks) >= 2 else (0, 1e30)
        inside = [r for r in rows if t0 - 1 <= r[0] <= t1 + 1]
        window = "timed region"
        if len(inside) < 3:
            inside, window = rows, "warm-up and timed region"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


# ------------------------------------------------------------------------------------------------
# workload helpers
# ------------------------------------------------------------------------------------------------

def workload(name: str):
    from sequence_attention_tcgen05_gb300 import synth
    return synth.WORKLOADS[name]


def phase_bytes(w, out_elem: int, ring_mode: str):
    """Algorithmic HBM bytes of the bandwidth-bound phases (each element read once + written once).

    Q/K/V are never re-laid by a pass: the attention's tensor maps address each virtual rank's
    head-sharded view in place for every ordering.  O and LSE are always written in the global
    layout by the attention (one ring rank, or fused ring steps) or by the merge (separate ring
    steps)."""
    elems = w.B * w.S * w.H * w.D
    rows_h = w.B * w.S * w.H
    b = {"qkv_relayout": 0}
    if ring_mode == "separate":
        # every partial's LSE is read; only partials whose rows saw a key are read in full (a
        # fully masked chunk pair leaves lse = -inf and the merge skips its O)
        seen = w.B * visible_partial_vectors(w)
        b["merge"] = w.ring_degree * rows_h * 4 + seen * w.D * 4 + elems * out_elem + rows_h * 4
    else:
        b["merge"] = 0
    return b


def visible_partial_vectors(w) -> int:
    """(row, head) vectors of one batch whose ring-step partial saw at least one key, from the
    library's host-side chunk-pair planner (usp_plan_pairs: q rows, visible kv rows and the
    diagonal of every run)."""
    from sequence_attention_tcgen05_gb300 import usp
    U = w.ulysses_degree
    heads = [w.H // U + (1 if u < w.H % U else 0) for u in range(U)]
    total = 0
    for (u, _r, _k, _r2, _row0, q_rows, kv_rows, diag) in usp.usp_plan_pairs(
            w.S, U, w.ring_degree, w.causal, w.order):
        if kv_rows <= 0:
            continue
        rows = q_rows if diag == 2**31 - 1 else max(0, q_rows - max(0, -diag))
        total += rows * heads[u]
    return total


def gpu_head_start(us: float = 60.0):
    """Keeps the GPU busy for about ``us`` microseconds (a spin kernel) so that the host can enqueue
    the next timed region before the GPU reaches its start event: the region then measures device
    execution, not host launch latency (which the e2e figure includes)."""
    import torch
    torch.cuda._sleep(int(us * 2000))


class L2Flush:
    """Evicts the L2 cache (129 MB) by reading a 256 MiB buffer; the lines it leaves are clean, so
    no write-back of earlier data falls into the next timed region."""

    def __init__(self, device):
        import torch
        self.buf = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=device)
        self.acc = torch.zeros((), dtype=torch.float32, device=device)

    def __call__(self):
        import torch
        torch.sum(self.buf, 0, out=self.acc)


def back_to_back_us(launch, n_sets: int, reps: int, flush, stream):
    """Mean device time (us) of one launch, from ``reps`` launches issued back to back between one
    pair of events on ``stream``.  Launch i uses buffer set i mod n_sets; the sets together span
    several times the L2, so no launch finds its inputs in L2.  A GPU spin before the first event,
    sized from the measured host enqueue time, lets the host enqueue every launch first, so that
    host launch latency is not timed."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(n_sets):
        launch(i)
    torch.cuda.synchronize()
    head_us = 100.0 + 40.0 * reps
    for _attempt in range(3):
        flush()
        gpu_head_start(head_us)
        e0.record(stream)
        t0 = time.perf_counter()
        for i in range(reps):
            launch(i % n_sets)
        host_us = (time.perf_counter() - t0) * 1e6
        e1.record(stream)
        e1.synchronize()
        if host_us < head_us:
            break
        head_us = 2.0 * host_us + 100.0  # the host fell behind the GPU: repeat with a longer spin
    return e0.elapsed_time(e1) * 1e3 / reps


def host_link_rates(dev_in, host_in, dev_out, host_out, stream, reps: int = 3):
    """Median ms and GB/s of one step's host->device copies alone, its device->host copies alone,
    and both on two streams at once (the host link is shared by the two directions)."""
    import torch
    n_in = sum(t.numel() * t.element_size() for t in dev_in)
    n_out = sum(t.numel() * t.element_size() for t in dev_out)
    s2 = torch.cuda.Stream(stream.device)

    def copy_in(s):
        with torch.cuda.stream(s):
            for d, h in zip(dev_in, host_in):
                d.copy_(h, non_blocking=True)

    def copy_out(s):
        with torch.cuda.stream(s):
            for h, d in zip(host_out, dev_out):
                h.copy_(d, non_blocking=True)

    def both(s):
        start = torch.cuda.Event()
        start.record(s)
        s2.wait_event(start)
        copy_in(s)
        copy_out(s2)
        done = torch.cuda.Event()
        done.record(s2)
        s.wait_event(done)

    def median_ms(fn):
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn(stream)
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    t_in, t_out, t_both = median_ms(copy_in), median_ms(copy_out), median_ms(both)
    return {"h2d_ms": t_in, "h2d_GB/s": n_in / t_in / 1e6, "d2h_ms": t_out,
            "d2h_GB/s": n_out / t_out / 1e6, "both_ms": t_both,
            "both_GB/s": (n_in + n_out) / t_both / 1e6}


def rotation(bytes_per_set: float) -> int:
    """Buffer sets so that a full rotation streams at least three times the L2 (129 MB)."""
    return max(1, math.ceil(3 * L2_BYTES / bytes_per_set))


def standalone_relayout(w, q, k, v, o, flush, stream, reps: int = 30):
    """GB/s of the standalone Ulysses re-layout entry points on this workload's tensors: seq->head
    of Q, K, V (one usp_relayout_seq2head_multi launch) and head->seq of O over the Ulysses split (a
    separately timed measurement, since the end-to-end step addresses these layouts in place).
    Back-to-back launches over rotating buffer sets; bytes = every element read once and written
    once."""
    import torch

    from sequence_attention_tcgen05_gb300 import usp
    U = max(2, w.ulysses_degree)
    lens = [w.S // U + (1 if p < w.S % U else 0) for p in range(U)]
    elems = w.B * w.S * w.H * w.D
    bin_, bout = 2 * 3 * elems * 2, 2 * elems * o.element_size()
    n_in = rotation(bin_)
    sets_in = [((q, k, v) if i == 0 else tuple(torch.empty_like(x) for x in (q, k, v)),
                tuple(torch.empty_like(x) for x in (q, k, v))) for i in range(n_in)]

    def seq2head(i):  # Q, K and V in one launch
        src, dst = sets_in[i]
        usp.usp_relayout_seq2head_multi(src, dst, w.B, w.H, w.D, lens, stream=stream)

    us_in = back_to_back_us(seq2head, n_in, reps, flush, stream)
    del sets_in
    n_out = rotation(bout)
    sets_out = [(o if i == 0 else torch.empty_like(o), torch.empty_like(o)) for i in range(n_out)]

    def head2seq(i):
        src, dst = sets_out[i]
        usp.usp_relayout_head2seq(src, dst, w.B, w.H, w.D, lens, stream=stream)

    us_out = back_to_back_us(head2seq, n_out, reps, flush, stream)
    del sets_out
    return {"ulysses_split": lens, "timing": f"{reps} back-to-back launches per figure",
            "seq2head_qkv": {"GB/s": bin_ / (us_in * 1e-6) / 1e9, "bytes": bin_, "us": us_in,
                             "buffer_sets": n_in, "launches": 1},
            "head2seq_o": {"GB/s": bout / (us_out * 1e-6) / 1e9, "bytes": bout, "us": us_out,
                           "buffer_sets": n_out, "launches": 1}}


def torch_copy_GBs(nbytes: int, flush, stream, reps: int = 30) -> float:
    """GB/s (bytes read + written) of torch's device-to-device copy of a tensor of nbytes / 2
    bytes, timed like the standalone legs: the practical ceiling for a transfer of that size."""
    import torch
    n = max(1, nbytes // 4)  # bf16 elements of half the traffic
    sets = [(torch.empty(n, dtype=torch.bfloat16, device="cuda"),
             torch.empty(n, dtype=torch.bfloat16, device="cuda")) for _ in range(rotation(nbytes))]

    def launch(i):
        a, b = sets[i]
        b.copy_(a)

    us = back_to_back_us(launch, len(sets), reps, flush, stream)
    del sets
    return 2 * n * 2 / (us * 1e-6) / 1e9


def standalone_merge(w, out_dt, flush, stream, reps: int = 30):
    """GB/s of the standalone usp_lse_merge entry point on two fp32 ring partials of this
    workload's size (a separately timed measurement: the step itself may have no merge).  Bytes:
    both partials and their LSE read, O (out_dt) and LSE written.  Back-to-back launches over
    rotating buffer sets."""
    import torch

    from sequence_attention_tcgen05_gb300 import usp
    rows, H, D = w.B * w.S, w.H, w.D
    elems, rows_h = rows * H * D, rows * H
    esz = torch.empty((), dtype=out_dt).element_size()
    nbytes = 2 * (elems * 4 + rows_h * 4) + elems * esz + rows_h * 4
    g = torch.Generator(device="cuda").manual_seed(1)
    sets = []
    for _ in range(rotation(nbytes)):
        sets.append((torch.randn((2, rows, H, D), dtype=torch.float32, device="cuda", generator=g),
                     torch.randn((2, rows, H), dtype=torch.float32, device="cuda", generator=g),
                     torch.empty((rows, H, D), dtype=out_dt, device="cuda"),
                     torch.empty((rows, H), dtype=torch.float32, device="cuda")))

    def call(i):
        o_parts, l_parts, o_out, l_out = sets[i]
        usp.usp_lse_merge(2, o_parts, rows * H * D, l_parts, rows * H, rows, H, D, o_out, l_out,
                          stream=stream)

    us = back_to_back_us(call, len(sets), reps, flush, stream)
    n_sets = len(sets)
    del sets
    return {"partials": 2, "bytes": nbytes, "us": us, "GB/s": nbytes / (us * 1e-6) / 1e9,
            "buffer_sets": n_sets, "timing": f"{reps} back-to-back launches"}


def cpu_oracle_sample(w, target_s: float, rng_seed: int = 0, max_scores: int = 1 << 26):
    """Time the fp64 oracle on a sample of the workload: heads in a seeded random order; per head
    every query row when the head's score matrix has at most ``max_scores`` entries, else that
    many scores' worth of random query rows, each against the head's full key set, until about
    ``target_s`` seconds have passed (at least one draw).  The FLOP count is the algorithmic one
    of the sampled rows (4 D per visible query/key pair), so the rate is comparable with the GPU
    figure.  Returns (TFLOP/s, seconds, description of the sample)."""
    import numpy as np

    import oracle
    from sequence_attention_tcgen05_gb300 import synth
    scale = 1.0 / math.sqrt(w.D)
    rng = np.random.default_rng(rng_seed)
    heads = [int(h) for h in rng.permutation(w.H)]
    n_rows = min(w.S, max(1, max_scores // max(1, w.S)))
    done_flops, spent, rows_done, draws = 0.0, 0.0, 0, 0
    heads_seen = set()
    for h in heads:
        k, v = (oracle.widen_bf16(synth.qkv_rows_bits(w.seed, st, w.B, w.S, w.H, w.D, 0,
                                                      np.arange(w.S), h, w.text_rows,
                                                      w.text_scale))
                for st in (synth.STREAM_K, synth.STREAM_V))
        heads_seen.add(h)
        while True:  # whole head once, or random row draws of this head until the time is up
            rows = (np.arange(w.S) if n_rows == w.S else
                    np.sort(rng.choice(w.S, size=n_rows, replace=False)))
            q = oracle.widen_bf16(synth.qkv_rows_bits(w.seed, synth.STREAM_Q, w.B, w.S, w.H, w.D,
                                                      0, rows, h, w.text_rows, w.text_scale))
            t0 = time.perf_counter()
            oracle.attention_rows(q, k, v, scale, w.causal, rows)
            spent += time.perf_counter() - t0
            visible = float((rows + 1).sum()) if w.causal else float(len(rows)) * w.S
            done_flops += 4.0 * w.D * visible
            rows_done += len(rows)
            draws += 1
            if n_rows == w.S or spent >= target_s:
                break
        if spent >= target_s:
            break
    if n_rows == w.S:
        desc = (f"{draws} whole heads of {w.H} (batch 0): every query row against the full key "
                f"set")
    else:
        desc = (f"sampled: {rows_done} random query rows ({draws} draws of {n_rows}) of "
                f"{len(heads_seen)} heads of {w.H} (batch 0), each against the full key set; "
                f"FLOPs of the visible pairs only")
    return done_flops / spent / 1e12, spent, desc


def nvtx_ranges(torch):
    """torch.cuda.nvtx, or do-nothing stand-ins if NVTX is unavailable (it never stops a run)."""
    try:
        torch.cuda.nvtx.range_push("bench")
        torch.cuda.nvtx.range_pop()
        return torch.cuda.nvtx
    except Exception:  # noqa: BLE001
        class _Off:
            @staticmethod
            def range_push(_name):
                return 0

            @staticmethod
            def range_pop():
                return 0
        return _Off()


def cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (model name; on Arm, implementer and part)."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if ":" in line:
                    key, val = (x.strip() for x in line.split(":", 1))
                    fields.setdefault(key, val)
    except OSError:
        pass
    if fields.get("model name"):
        return fields["model name"]
    if "CPU part" in fields:
        return (f"{platform.machine()} implementer {fields.get('CPU implementer', '?')} "
                f"part {fields['CPU part']}")
    return platform.machine()


# ------------------------------------------------------------------------------------------------
# arms
# ------------------------------------------------------------------------------------------------

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = workload(args.workload)
    # each step a bounded sample, sized so the whole run stays within about two minutes
    per_step = max(0.2, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    vals, secs = [], []
    for i in range(args.warmup + args.steps):
        v, dt, desc = cpu_oracle_sample(w, per_step, rng_seed=i)
        if i >= args.warmup:
            vals.append(v)
            secs.append(dt)
    value = sum(v * s for v, s in zip(vals, secs)) / sum(secs)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000 * statistics.mean(secs), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, args.out_dtype),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores(), "kind": "oracle",
                             "sample": desc, "cpu": cpu_model()},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_of(w, out_dtype: str):
    """The workload, as both arms name it: shapes, grid, ordering and the requested output dtype
    (how an implementation runs it goes into other keys of its line)."""
    return {"workload": w.name, "B": w.B, "S": w.S, "H": w.H, "D": w.D,
            "ulysses_degree": w.ulysses_degree, "ring_degree": w.ring_degree,
            "causal": w.causal, "order": w.order, "text_rows": w.text_rows,
            "seq_lens": list(w.seq_lens) or "default split", "out_dtype": out_dtype}


L2_NOTE = "flushed between timed steps (256 MiB read outside the step events)"


def run_ours(args):
    import numpy as np
    import torch

    from sequence_attention_tcgen05_gb300 import build, synth, usp

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    build.build_library()
    usp.lib()
    w = workload(args.workload)
    out_dt = torch.bfloat16 if args.out_dtype == "bf16" else torch.float32
    o_code = usp.USP_BF16 if out_dt == torch.bfloat16 else usp.USP_FP32
    out_elem = 2 if out_dt == torch.bfloat16 else 4
    B, S, H, D = w.B, w.S, w.H, w.D
    scale = 1.0 / math.sqrt(D)
    flops = w.attention_flops()

    qb, kb, vb = synth.make_qkv_bits(B, S, H, D, w.seed, w.text_rows, w.text_scale)
    host = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in (qb, kb, vb)]
    q, k, v = (x.to(device) for x in host)
    o = torch.empty((B, S, H, D), dtype=out_dt, device=device)
    lse = torch.empty((B, S, H), dtype=torch.float32, device=device)
    nbytes = usp.usp_attention_workspace_size(B, S, H, D, w.ulysses_degree, w.ring_degree,
                                              w.order, o_code, w.causal)
    ring_mode = usp.usp_attention_ring_mode(B, S, H, D, w.causal, w.ulysses_degree, w.ring_degree,
                                            w.order, o_code)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=device)
    flush = L2Flush(device)  # 256 MiB > L2
    stream = torch.cuda.current_stream()
    seq = list(w.seq_lens) or None

    def make_events():
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        for e in evs:
            e.record(stream)  # materialise the handle
        return evs

    events = make_events()
    handles = [e.cuda_event for e in events]

    def step(evs):
        return usp.usp_attention_events(q, k, v, B, S, H, D, scale, w.causal, w.ulysses_degree,
                                        w.ring_degree, o, lse, ws, nbytes, evs, seq, None,
                                        w.order, o_code, stream)

    no_events = [None] * 5
    nvtx = nvtx_ranges(torch)  # section ranges for profiler timelines (no-ops without a profiler)
    # clocks are sampled from before the warm-up, so that the GPU goes straight from the warm-up
    # steps into the timed ones (no idle gap that would let it cool and change clocks)
    clocks = ClockSampler(local)
    clocks.start()
    nvtx.range_push("bench: warm-up")
    for _ in range(args.warmup):
        flush()
        step(handles)
    torch.cuda.synchronize()
    nvtx.range_pop()
    if usp.usp_check_status(ws) != usp.USP_OK:
        raise RuntimeError("device status after warm-up: " + usp.lib().usp_last_error().decode())

    # headline: one event pair around each step; the flush and a short GPU spin before the start
    # event let the host enqueue the whole step before the GPU reaches it
    e_begin, e_finish = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    total_ms = 0.0
    step_ms = []
    launches = 0
    barrier(device)
    torch.cuda.synchronize()
    clocks.mark()
    nvtx.range_push("bench: timed steps")
    for _ in range(args.steps):
        flush()
        gpu_head_start()
        e_begin.record(stream)
        launches += sum(step(no_events))
        e_finish.record(stream)
        e_finish.synchronize()
        step_ms.append(e_begin.elapsed_time(e_finish))
        total_ms += step_ms[-1]
    torch.cuda.synchronize()
    nvtx.range_pop()
    barrier(device)
    clocks.mark()
    clk = clocks.stop()

    # per-phase breakdown (separate loop: the phase events themselves cost about 2 us each)
    phases = {"qkv_relayout": 0.0, "attention": 0.0, "merge": 0.0, "out_relayout": 0.0}
    phase_launches = [0, 0, 0, 0]
    breakdown_steps = min(args.steps, 200)
    nvtx.range_push("bench: phase breakdown")
    for _ in range(breakdown_steps):
        flush()
        gpu_head_start()
        phase_launches = step(handles)
        events[4].synchronize()
        t = [events[i].elapsed_time(events[i + 1]) for i in range(4)]
        for name, dt in zip(phases, t):
            phases[name] += dt
    nvtx.range_pop()
    status = usp.usp_check_status(ws)
    if status != usp.USP_OK:
        raise RuntimeError("device status after timing: " + usp.lib().usp_last_error().decode())
    value, t_max = aggregate(args.steps * flops, total_ms / 1000.0, world, device)
    value /= 1e12

    # the same step on a QKV-packed input [B][S][3][H][D] (usp_attention_qkvpacked), timed the
    # same way over a shorter loop
    nvtx.range_push("bench: packed QKV")
    qkv = torch.stack([q, k, v], dim=2).contiguous()
    packed_steps = min(args.steps, 50)
    packed_ms = 0.0
    for i in range(packed_steps + 3):
        flush()
        gpu_head_start()
        e_begin.record(stream)
        usp.usp_attention_qkvpacked(qkv, B, S, H, D, scale, w.causal, w.ulysses_degree,
                                    w.ring_degree, o, lse, ws, nbytes, seq, None, w.order, o_code,
                                    stream)
        e_finish.record(stream)
        e_finish.synchronize()
        if i >= 3:
            packed_ms += e_begin.elapsed_time(e_finish)
    del qkv
    nvtx.range_pop()
    packed_value, _ = aggregate(packed_steps * flops, packed_ms / 1000.0, world, device)

    # end to end through the C ABI with host buffers
    nvtx.range_push("bench: end to end")
    e2e_steps = max(3, min(args.steps, 50))
    o_host = torch.empty(o.shape, dtype=out_dt).pin_memory()
    l_host = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    # (a) serial: one step at a time on one stream (copy in, usp_attention, copy out), with an
    # event between the stages
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    e2e_ms = 0.0
    serial_stages = {"h2d": [], "attention": [], "d2h": []}
    for i in range(e2e_steps + 1):
        flush()
        ev_s[0].record(stream)
        for dst, src in zip((q, k, v), host):
            dst.copy_(src, non_blocking=True)
        ev_s[1].record(stream)
        usp.usp_attention(q, k, v, B, S, H, D, scale, w.causal, w.ulysses_degree, w.ring_degree,
                          o, lse, ws, nbytes, seq, None, w.order, o_code, stream)
        ev_s[2].record(stream)
        o_host.copy_(o, non_blocking=True)
        l_host.copy_(lse, non_blocking=True)
        ev_s[3].record(stream)
        ev_s[3].synchronize()
        if i > 0:
            e2e_ms += ev_s[0].elapsed_time(ev_s[3])
            for n, a, b_ in (("h2d", 0, 1), ("attention", 1, 2), ("d2h", 2, 3)):
                serial_stages[n].append(ev_s[a].elapsed_time(ev_s[b_]))
    e2e_serial, _ = aggregate(e2e_steps * flops, e2e_ms / 1000.0, world, device)
    # the host link's rates in this run (the e2e figure's ceiling): each direction alone, then both
    # at once, as the pipelined loop runs them
    link = host_link_rates((q, k, v), host, (o, lse), (o_host, l_host), stream)
    # (b) pipelined, as a caller serving a stream of requests runs it: two sets of device buffers,
    # one stream per direction of the host link (the two directions overlap) and one for compute.
    # Every step still copies its Q, K, V in and its O, LSE out inside the timed region; step i's
    # copy-in overlaps step i-1's attention and copy-out.
    sets = [(q, k, v, o, lse, o_host, l_host),
            (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(o),
             torch.empty_like(lse), torch.empty(o.shape, dtype=out_dt).pin_memory(),
             torch.empty(lse.shape, dtype=torch.float32).pin_memory())]
    s_in, s_cmp, s_out = (torch.cuda.Stream(device) for _ in range(3))
    ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("in", "cmp", "out")}
    for b_ in range(2):
        ev["cmp"][b_].record(s_cmp)
        ev["out"][b_].record(s_out)

    def pipelined(n_steps, timed=False):
        marks = []
        for i in range(n_steps):
            b_ = i & 1
            qd, kd, vd, od, ld, oh, lh = sets[b_]
            te = [torch.cuda.Event(enable_timing=True) for _ in range(6)] if timed else None
            s_in.wait_event(ev["cmp"][b_])  # step i-2's attention has read this input set
            if timed:
                te[0].record(s_in)
            with torch.cuda.stream(s_in):
                for dst, src in zip((qd, kd, vd), host):
                    dst.copy_(src, non_blocking=True)
            if timed:
                te[1].record(s_in)
            ev["in"][b_].record(s_in)
            s_cmp.wait_event(ev["in"][b_])
            s_cmp.wait_event(ev["out"][b_])  # step i-2's copy-out has read this output set
            if timed:
                te[2].record(s_cmp)
            usp.usp_attention(qd, kd, vd, B, S, H, D, scale, w.causal, w.ulysses_degree,
                              w.ring_degree, od, ld, ws, nbytes, seq, None, w.order, o_code, s_cmp)
            if timed:
                te[3].record(s_cmp)
            ev["cmp"][b_].record(s_cmp)
            s_out.wait_event(ev["cmp"][b_])
            if timed:
                te[4].record(s_out)
            with torch.cuda.stream(s_out):
                oh.copy_(od, non_blocking=True)
                lh.copy_(ld, non_blocking=True)
            if timed:
                te[5].record(s_out)
            ev["out"][b_].record(s_out)
            if timed:
                marks.append(te)
        return marks

    pipelined(4)
    torch.cuda.synchronize()
    p_start, p_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p_start.record(s_in)
    marks = pipelined(e2e_steps, timed=True)
    p_end.record(s_out)  # after the last copy-out, which depends on every earlier operation
    p_end.synchronize()
    # per-stage durations inside the pipeline, and the attention's start-to-start period
    pipe_stages = {"h2d": [m[0].elapsed_time(m[1]) for m in marks],
                   "attention": [m[2].elapsed_time(m[3]) for m in marks],
                   "d2h": [m[4].elapsed_time(m[5]) for m in marks],
                   "attention_period": [a[2].elapsed_time(b_[2]) for a, b_ in zip(marks, marks[1:])]}
    e2e_value, _ = aggregate(e2e_steps * flops, p_start.elapsed_time(p_end) / 1000.0, world, device)
    nvtx.range_pop()
    if usp.usp_check_status(ws, s_cmp) != usp.USP_OK:
        raise RuntimeError("device status after the end-to-end loops: " +
                           usp.lib().usp_last_error().decode())
    h2d = 3 * B * S * H * D * 2
    d2h = B * S * H * D * out_elem + B * S * H * 4

    peaks, peak_kind = load_peaks()
    att_s = phases["attention"] / 1000.0 / breakdown_steps
    achieved = flops / att_s / 1e12
    peak, sustained = roofline_peak(peaks, total_ms)
    traffic = ATTN_TRAFFIC.get(w.name)
    traffic_bytes = traffic["bytes"] if traffic and traffic["kernel_hash"] == kernel_hash() else None
    pb = phase_bytes(w, out_elem, ring_mode)
    ran = dict(zip(phases, (n > 0 for n in phase_launches)))
    bw = {}
    for name in ("qkv_relayout", "merge"):
        if pb[name] and ran[name]:
            s = phases[name] / 1000.0 / breakdown_steps
            gbs = pb[name] / s / 1e9
            bw[name] = {"GB/s": gbs, "bytes": pb[name], "us": s * 1e6,
                        "frac_measured_hbm": gbs / peaks["hbm_gbs"], "frac_8TBs": gbs / NOMINAL_HBM_GBS}
    bw_bytes = sum(pb[n] for n in ("qkv_relayout", "merge") if ran[n])
    nvtx.range_push("bench: standalone re-layout and merge")
    standalone = standalone_relayout(w, q, k, v, o, flush, stream)
    standalone_m = standalone_merge(w, out_dt, flush, stream)
    # the same legs on the FLUX 1024^2 shape (57 MB tensors) when the workload is another one
    flux_legs = None
    if w.name != "flux_1024_u2":
        wf = workload("flux_1024_u2")
        shape = (wf.B, wf.S, wf.H, wf.D)
        qf, kf, vf = (torch.zeros(shape, dtype=torch.bfloat16, device=device) for _ in range(3))
        of = torch.zeros(shape, dtype=out_dt, device=device)
        flux_legs = {"workload": wf.name, "relayout": standalone_relayout(wf, qf, kf, vf, of, flush, stream),
                     "merge": standalone_merge(wf, out_dt, flush, stream)}
        del qf, kf, vf, of
    nvtx.range_pop()
    legs = [standalone["seq2head_qkv"], standalone["head2seq_o"], standalone_m]
    if flux_legs:
        legs += [flux_legs["relayout"]["seq2head_qkv"], flux_legs["relayout"]["head2seq_o"], flux_legs["merge"]]
    for part in legs:
        part["frac_measured_hbm"] = part["GB/s"] / peaks["hbm_gbs"]
        part["frac_8TBs"] = part["GB/s"] / NOMINAL_HBM_GBS
        part["torch_copy_same_bytes_GB/s"] = torch_copy_GBs(part["bytes"], flush, stream)
    bw_s = sum(phases[n] for n in ("qkv_relayout", "merge") if ran[n]) / 1000.0 / breakdown_steps
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t_max * 1000.0 / args.steps, "higher_is_better": True,
        "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms),
                    "max": max(step_ms)},
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_of(w, args.out_dtype),
        "ring_steps": ring_mode, "l2": L2_NOTE,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic_bytes,
                     "kernel": "attn_fwd_kernel (all chunk pairs and ring steps, one launch)",
                     "peak_kind": f"{peak_kind} bf16 {'sustained' if sustained else 'burst'} "
                                  f"(timed region {total_ms:.0f} ms of device time; sustained "
                                  f"from {SUSTAINED_MS:.0f} ms)",
                     "frac_burst_peak": achieved / peaks["bf16_tflops"],
                     "frac_sustained_peak": achieved / peaks["bf16_tflops_sustained"]},
        "relayout_merge": {"GB/s": bw_bytes / bw_s / 1e9 if bw_s > 0 else None,
                           "frac_measured_hbm": (bw_bytes / bw_s / 1e9 / peaks["hbm_gbs"]) if bw_s > 0 else None,
                           "frac_8TBs": (bw_bytes / bw_s / 1e9 / NOMINAL_HBM_GBS) if bw_s > 0 else None,
                           "phases": bw, "standalone_relayout": standalone,
                           "standalone_merge": standalone_m, "standalone_flux_1024_shape": flux_legs},
        "phases_ms_per_step": {k: (v / breakdown_steps if ran[k] else None)
                               for k, v in phases.items()},
        "phase_launches": dict(zip(phases, phase_launches)),
        "phases_steps": breakdown_steps,
        "e2e": {"value": e2e_value / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "mode": "pipelined: step i's copy-in overlaps step i-1's attention and copy-out "
                        "(two device buffer sets, one stream per link direction)",
                "serial_value": e2e_serial / 1e12, "host_link": link,
                # median and maximum ms of each stage (and of the attention's start-to-start
                # period when pipelined), from events between the stages: a maximum far above the
                # median is a stall of the shared host link, not of the kernels
                "serial_stage_ms": {n: {"median": statistics.median(x), "max": max(x)}
                                    for n, x in serial_stages.items()},
                "pipelined_stage_ms": {n: {"median": statistics.median(x), "max": max(x)}
                                       for n, x in pipe_stages.items() if x},
                # the pipelined figure this run's link rates predict: the FLOPs of a step over the
                # larger of its device time and its copies in both directions at once (a short
                # burst; back-to-back steps keep the link busier, so the figure can exceed it a
                # little)
                "pipelined_estimate": flops / max(t_max * 1000.0 / args.steps,
                                                  link["both_ms"]) / 1e9},
        "qkvpacked": {"value": packed_value / 1e12, "unit": "TFLOP/s",
                      "ms_per_step": packed_ms / packed_steps, "steps": packed_steps,
                      "input": "bf16 [B][S][3][H][D] through usp_attention_qkvpacked"},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cv, cdt, desc = cpu_oracle_sample(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": cv, "unit": "TFLOP/s", "cores": cores(), "kind": "oracle",
                                "sample": desc, "seconds": cdt, "cpu": cpu_model()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--out-dtype", choices=["bf16", "fp32"], default="bf16")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
