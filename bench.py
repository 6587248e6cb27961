#!/usr/bin/env python
"""Benchmark of the paged-KV attention hot path on GB300.

Headline step (workload "llama8b_decode": batch 64, 32 q / 8 kv heads, head_dim 128, bf16, KV
lengths U[512, 4096], page size 16, pages randomly permuted in a pool 1.25x the need): one pass of
the path for one batch = plan (host work + metadata copy) + KV write of the 64 new tokens + paged
decode (+ split-KV merge).  Metric: KV-read GB/s = algorithmic K/V bytes the decode must read
(every visible key row, K and V, every KV head) / step time.

Also measured (same JSON line, "prefill" object): the prefix-cached extend workload (batch 8, new
U[128, 2048], prefix U[0, 4096], page size 1) as TFLOP/s over the causally visible (query, key)
pairs, when the prefill kernel is built.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1: launched by torch.distributed.run, one rank per GPU; every rank runs its own independent
batch (weak scaling, no data-path collective); the step time is the max over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e nominal, reported beside the measured-copy fraction
DEFAULT_BF16_TFLOPS = 1900.0


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return DEFAULT_HBM_GBS, DEFAULT_BF16_TFLOPS, 1700.0, "fallback"


def _src_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "paged_kv_attention_slot_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


DECODE_SOURCES = ["decode.cu", "ptx.cuh", "pkv_internal.h"]
# the workload both arms name in `config` (the oracle arm times the step's attention on a bounded sample
# of its requests, stated in its `cpu_baseline.sample`)
DECODE_WORKLOAD = ("llama8b_decode: batch 64, 32 q / 8 kv heads, head_dim 128, bf16 KV, KV length U[512,4096], "
                   "page 16, pool 1.25x, step = kv_store + plan + decode")
PREFILL_SOURCES = ["prefill.cu", "ptx.cuh", "tc.cuh", "pkv_internal.h"]


def _traffic(kernel: str, source_files):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d or d.get("source_hash") != _src_hash(*source_files):
        return None
    return d.get("bytes_per_launch")


# ------------------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.lines = []
        self.proc = None
        self.device_index = device_index

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}", "--format=csv,noheader,nounits", "-lms", "200"]
        uuid = None
        try:
            import torch

            uuid = str(torch.cuda.get_device_properties(self.device_index).uuid)
        except Exception:
            pass
        if uuid:
            cmd += ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------------------------------------
# CPU oracle baseline (spawned process pool; one task = one request)
# ------------------------------------------------------------------------------------------------
_WORKER_BATCHES = None


def _oracle_worker_init(workload_ns, seed_offset):
    """Each worker regenerates the seeded batches once (untimed), so tasks carry only row ids."""
    global _WORKER_BATCHES
    import numpy as np
    import torch

    import workloads as W

    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    from oracle import attention as OA

    _WORKER_BATCHES = {}
    for n in workload_ns:
        b = W.workload(n, seed_offset=seed_offset)
        kb, vb = bits(b.k_pool), bits(b.v_pool)
        if b.q_len.max() > 1:  # the prefill workload reads this step's new rows: the pool after its KV write
            kb, vb = kb.copy(), vb.copy()
            OA.kv_store(kb, vb, bits(b.k_new), bits(b.v_new), b.slot_mapping, b.page_size)
        _WORKER_BATCHES[n] = (b, bits(b.q), kb, vb)


def _noop(_):
    return _WORKER_BATCHES is not None


def _oracle_rows_task(task):
    """Worker: the oracle, as it stands, on the given token rows of workload n (one request's rows)."""
    import numpy as np

    from oracle import attention as OA

    n, rows = task
    b, qb, kb, vb = _WORKER_BATCHES[n]
    o, _ = OA.paged_attention(qb, kb, vb, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.page_size,
                              sm_scale=b.sm_scale if b.sm_scale > 0 else None, window_left=b.window_left,
                              q_format="bf16_bits", kv_format="bf16_bits", rows=list(rows))
    return float(np.nansum(o))


class OraclePool:
    def __init__(self, workload_ns=(2,), seed_offset=0):
        import multiprocessing as mp

        self.cores = max(1, os.cpu_count() or 1)
        env = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"}
        old = {k: os.environ.get(k) for k in env}
        os.environ.update(env)
        try:
            self.pool = mp.get_context("spawn").Pool(self.cores, initializer=_oracle_worker_init,
                                                     initargs=(tuple(workload_ns), seed_offset))
        finally:
            for k, v in old.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def wait_ready(self):
        """Block until every worker has finished its (CPU-heavy) initialisation, so no worker competes
        with the GPU timing for host cores."""
        self.pool.map(_noop, range(4 * self.cores), chunksize=1)

    def run(self, b, req_ids, n=2):
        """Wall time of the oracle over these decode requests (workload n), one request per task."""
        return self.run_rows(n, [[int(b.qo_indptr[i])] for i in req_ids])

    def run_rows(self, n, row_groups):
        """Wall time of the oracle over these groups of token rows of workload n, one group per task."""
        t0 = time.perf_counter()
        self.pool.map(_oracle_rows_task, [(n, list(g)) for g in row_groups], chunksize=1)
        return time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


def _kv_bytes(b, req_ids):
    import numpy as np

    L = b.kv_len[np.asarray(req_ids)]
    if b.window_left >= 0:
        L = np.minimum(L, b.window_left + 1)
    elem = 1 if b.kv_dtype == "e4m3" else 2
    return int(L.sum()) * b.num_kv_heads * b.head_dim * elem * 2


def cpu_baseline(b, pool, target_s=12.0):
    """The oracle, as it stands, on the host cores: whole batches repeated until ~target_s of work."""
    ids = list(range(b.batch_size))
    pool.run(b, ids[: min(4, len(ids))])  # warm the workers
    reps, total_t = 0, 0.0
    while total_t < target_s and reps < 50:
        total_t += pool.run(b, ids)
        reps += 1
    gbs = _kv_bytes(b, ids) * reps / total_t / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": pool.cores, "kind": "oracle",
            "sample": f"{reps} x the full {b.batch_size}-request batch ({_kv_bytes(b, ids) / 1e6:.1f} MB of KV each), "
                      f"one request per task on a spawn pool of {pool.cores} single-threaded processes, "
                      f"fp64 numpy oracle as it stands, wall clock"}


def prefill_sample_rows(b, per_request=128, chunk=32, seed=3):
    """A bounded, seeded sample of the prefill workload's token rows: up to `per_request` rows of
    every request (its first and last row included), grouped by request in chunks of `chunk` rows."""
    import numpy as np

    rng = np.random.default_rng(seed)
    groups = []
    for i in range(b.batch_size):
        q0, q1 = int(b.qo_indptr[i]), int(b.qo_indptr[i + 1])
        if q1 == q0:
            continue
        rows = np.arange(q0, q1) if q1 - q0 <= per_request else np.unique(np.concatenate(
            [[q0, q1 - 1], rng.choice(np.arange(q0 + 1, q1 - 1), per_request - 2, replace=False)]))
        groups += [rows[k:k + chunk].tolist() for k in range(0, len(rows), chunk)]
    return groups


def _rows_flops(b, row_groups):
    """Algorithmic FLOPs of the sampled rows: 4 * D * Hq * visible keys of each row (causal)."""
    import numpy as np

    req = np.searchsorted(b.qo_indptr, np.arange(int(b.qo_indptr[-1])), side="right") - 1
    total = 0.0
    for g in row_groups:
        for r in g:
            i = int(req[r])
            pos = int(b.kv_len[i]) - int(b.q_len[i]) + (r - int(b.qo_indptr[i]))
            lo = 0 if b.window_left < 0 else max(0, pos - b.window_left)
            total += 4.0 * b.head_dim * b.num_qo_heads * (pos - lo + 1)
    return total


def cpu_baseline_prefill(pool, target_s=10.0):
    """The oracle, as it stands, on a bounded sample of the prefill workload's rows, TFLOP/s."""
    import workloads as W

    b = W.workload(3)
    groups = prefill_sample_rows(b)
    pool.run_rows(3, groups[:2])  # warm the workers
    reps, total_t = 0, 0.0
    while total_t < target_s and reps < 50:
        total_t += pool.run_rows(3, groups)
        reps += 1
    flops = _rows_flops(b, groups)
    nrows = sum(len(g) for g in groups)
    return {"value": round(flops * reps / total_t / 1e12, 6), "unit": "TFLOP/s", "cores": pool.cores,
            "kind": "oracle",
            "sample": f"{reps} x {nrows} token rows of the prefix_extend batch (up to 128 seeded rows per request, "
                      f"first and last included, all 32 heads; {flops / 1e9:.1f} GFLOP of visible pairs per pass), "
                      f"{len(groups)} tasks of one request's rows on a spawn pool of {pool.cores} single-threaded "
                      f"processes, fp64 numpy oracle as it stands, wall clock"}


# ------------------------------------------------------------------------------------------------
# multi-rank bookkeeping (one rank per GPU; each rank runs its own independent batch)
# ------------------------------------------------------------------------------------------------
def rank_batch(n: int, rank: int, scale_batch: float = 1.0):
    """Rank `rank`'s batch of workload n: same shape, its own seed (weak scaling, no shared requests)."""
    import workloads as W

    return W.workload(n, seed_offset=rank, scale_batch=scale_batch)


def max_over_ranks(value: float, device=None) -> float:
    """The slowest rank's time (all ranks must call it); identity without a process group."""
    import torch

    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_rank_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: the bytes every rank processed over the slowest rank's time."""
    return bytes_per_rank_step * steps * world / (max_ms * 1e-3) / 1e9


# ------------------------------------------------------------------------------------------------
# the GPU arm
# ------------------------------------------------------------------------------------------------
def _device_state(b, device):
    import torch

    import paged_kv_attention_slot_gb300 as pk

    st = {}
    if b.kv_dtype == "bf16":
        st["k_pool"] = b.k_pool.to(device)
        st["v_pool"] = b.v_pool.to(device)
        st["cache"] = pk.KVCache(st["k_pool"], st["v_pool"])
    else:  # FP8 pools written by the library's own quantising kv_store
        P, ps, H, D = b.k_pool.shape
        st["k_pool"] = torch.zeros((P, ps, H, D), dtype=torch.uint8, device=device)
        st["v_pool"] = torch.zeros((P, ps, H, D), dtype=torch.uint8, device=device)
        st["cache"] = pk.KVCache(st["k_pool"], st["v_pool"], b.k_scale, b.v_scale)
        slots = torch.arange(P * ps, dtype=torch.int64, device=device)
        pk.kv_store(b.k_pool.to(device).view(P * ps, H, D), b.v_pool.to(device).view(P * ps, H, D), slots,
                    st["cache"])
        torch.cuda.synchronize()
    st["q"] = b.q.to(device)
    st["k_new"] = b.k_new.to(device)
    st["v_new"] = b.v_new.to(device)
    st["slots"] = torch.from_numpy(b.slot_mapping).to(device)
    st["out"] = torch.empty_like(st["q"])
    return st


def _plan_kw(b):
    return dict(num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads, head_dim=b.head_dim,
                page_size=b.page_size, mode=b.mode, window_left=b.window_left, sm_scale=b.sm_scale,
                kv_dtype=b.kv_dtype)


def run_steps(b, st, plan, steps, warmup, dist_on, record_run_events=False):
    """Warm up, then time exactly `steps` steps on the device (CUDA events), inputs resident.

    record_run_events: also bracket each run with CUDA events (a diagnostic pass only: an event
    between the KV write and the run breaks their launch overlap, so the timed pass records none)."""
    import torch

    import paged_kv_attention_slot_gb300 as pk

    kw = _plan_kw(b)
    stream = torch.cuda.current_stream()
    run_ev = []

    def step(i, timed):
        # the KV write needs no plan, so it goes first: the metadata copy's reads of the pinned staging
        # (issued before its programmatic-launch wait) then overlap the KV write
        pk.kv_store(st["k_new"], st["v_new"], st["slots"], st["cache"])
        plan.plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, **kw)
        if timed and record_run_events:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            plan.run(st["q"], st["cache"], out=st["out"])
            e1.record(stream)
            run_ev.append((e0, e1))
        else:
            plan.run(st["q"], st["cache"], out=st["out"])

    for i in range(warmup):
        step(i, False)
    if dist_on:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        step(i, True)
    t1.record(stream)
    torch.cuda.synchronize()
    if dist_on:
        torch.distributed.barrier()
    total_ms = t0.elapsed_time(t1)
    run_ms = [a.elapsed_time(c) for a, c in run_ev]
    return total_ms, run_ms


def plan_host_us(b, plan, reps=30):
    """Median host time of one plan() call through the public API (the planner, the binding and the
    enqueue of the metadata copy), each call after a synchronise so no GPU wait is counted."""
    import torch

    kw = _plan_kw(b)
    ts = []
    for _ in range(reps):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        plan.plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, **kw)
        ts.append(time.perf_counter() - t0)
    torch.cuda.synchronize()
    return round(statistics.median(ts) * 1e6, 1)


def kernel_ms(run_once, reps=20, iters=7):
    """Average device time of one run launch: `reps` launches captured in one CUDA graph and replayed
    between two CUDA events on the launching stream (no host launch gaps between the kernels).  Falls
    back to eager back-to-back launches if capture fails."""
    import torch

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            run_once()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    mode = f"CUDA graph of {reps} launches, replayed"
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(reps):
                run_once()

        def replay():
            graph.replay()
    except Exception as e:  # capture unsupported here: time eager launches instead
        torch.cuda.synchronize()
        mode = f"{reps} eager back-to-back launches (graph capture failed: {type(e).__name__})"

        def replay():
            for _ in range(reps):
                run_once()
    stream = torch.cuda.current_stream()
    replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    per = []
    for _ in range(iters):
        e0.record(stream)
        replay()
        e1.record(stream)
        torch.cuda.synchronize()
        per.append(e0.elapsed_time(e1) / reps)
    return statistics.median(per), mode


def run_e2e(b, st, plan, steps, warmup, reps=5):
    """Same step through the public API from pinned HOST buffers: every step copies its inputs (Q,
    the new K/V rows, slot_mapping) host -> device, re-plans, writes the KV, runs, and copies O back
    to the host.  Steps are pipelined as a serving loop would run them: the copies go on two copy
    streams (H2D and D2H) so that step i's input copy overlaps step i - 1's kernels and step i's
    output copy overlaps step i + 1's; the host plans and enqueues step i while the device still runs
    step i - 1, then waits for step i - 1's output.  Pinned inputs, device inputs, device outputs and
    pinned outputs are double-buffered, and events order every reuse of a buffer (stream order keeps
    each plan's metadata copy behind the previous run).  The `steps`-step loop is timed `reps` times
    (a wall-clock measurement of a few milliseconds: the median resists host hiccups).  Returns the
    wall times, the H2D and D2H bytes per step, and the largest difference between the last step's
    output on the host and the same step timed on the device."""
    import torch

    import paged_kv_attention_slot_gb300 as pk

    kw = _plan_kw(b)
    # a step's inputs packed in one pinned host buffer and copied to one device buffer with a single
    # H2D copy; the device tensors are views of it
    parts = [b.q.contiguous().view(torch.uint8).reshape(-1), b.k_new.contiguous().view(torch.uint8).reshape(-1),
             b.v_new.contiguous().view(torch.uint8).reshape(-1),
             torch.from_numpy(b.slot_mapping).contiguous().view(torch.uint8).reshape(-1)]
    offs = [0]
    for t in parts:
        offs.append(offs[-1] + (t.numel() + 255) // 256 * 256)
    dev = st["q"].device
    bufs = []
    for _ in range(2):
        h_in = torch.empty(offs[-1], dtype=torch.uint8).pin_memory()
        for t, o in zip(parts, offs):
            h_in[o:o + t.numel()] = t
        d_in = torch.empty(offs[-1], dtype=torch.uint8, device=dev)
        views = (d_in[offs[0]:offs[0] + parts[0].numel()].view(torch.bfloat16).view(b.q.shape),
                 d_in[offs[1]:offs[1] + parts[1].numel()].view(torch.bfloat16).view(b.k_new.shape),
                 d_in[offs[2]:offs[2] + parts[2].numel()].view(torch.bfloat16).view(b.v_new.shape),
                 d_in[offs[3]:offs[3] + parts[3].numel()].view(torch.int64))
        bufs.append({"h_in": h_in, "d_in": d_in, "views": views, "d_out": torch.empty_like(st["out"]),
                     "h_out": torch.empty_like(b.q).pin_memory(), "in_ready": torch.cuda.Event(),
                     "run_done": torch.cuda.Event(), "out_copied": torch.cuda.Event()})
    compute = torch.cuda.current_stream()
    h2d_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)

    def enqueue(i):
        B = bufs[i & 1]
        q, k_new, v_new, slots = B["views"]
        if i >= 2:  # step i - 2's kernels have read this input buffer
            h2d_stream.wait_event(B["run_done"])
        with torch.cuda.stream(h2d_stream):
            B["d_in"].copy_(B["h_in"], non_blocking=True)
        B["in_ready"].record(h2d_stream)
        compute.wait_event(B["in_ready"])
        # the KV write needs no plan: the GPU stores this step's rows while the host plans
        pk.kv_store(k_new, v_new, slots, st["cache"], stream=compute)
        plan.plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, stream=compute, **kw)
        if i >= 2:  # step i - 2's output has left this device buffer
            compute.wait_event(B["out_copied"])
        plan.run(q, st["cache"], out=B["d_out"], stream=compute)
        B["run_done"].record(compute)
        d2h_stream.wait_event(B["run_done"])
        with torch.cuda.stream(d2h_stream):
            B["h_out"].copy_(B["d_out"], non_blocking=True)
        B["out_copied"].record(d2h_stream)

    def run(n):
        for i in range(n):
            enqueue(i)
            if i > 0:
                bufs[(i - 1) & 1]["out_copied"].synchronize()  # step i - 1's output is on the host
        bufs[(n - 1) & 1]["out_copied"].synchronize()

    run(warmup)
    torch.cuda.synchronize()
    dts = []
    for _ in range(reps):
        t0 = time.perf_counter()
        run(steps)
        dts.append(time.perf_counter() - t0)
        torch.cuda.synchronize()
    h2d = sum(t.numel() for t in parts)  # bytes of Q, K/V rows and slots (padding excluded)
    h2d += sum(a.nbytes for a in (b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len))
    d2h = bufs[0]["h_out"].numel() * bufs[0]["h_out"].element_size()
    # the host copy of the last step against the device-timed path's output on the same inputs
    diff = float((bufs[(steps - 1) & 1]["h_out"].float() - st["out"].cpu().float()).abs().max())
    return dts, h2d, d2h, diff


def decode_other_configs(device, hbm):
    """Decode kernel time on the other decode workloads (same kernel, CUDA-graph replay timing)."""
    import torch

    import paged_kv_attention_slot_gb300 as pk
    import workloads as W

    res = []
    for n, window, key, name in (
            (4, -1, "decode_llama70b_ragged", "llama70b_ragged_decode: batch 256, 64 q / 8 kv, log-normal KV (median 1024), page 64, bf16"),
            (5, -1, "decode_fp8_long", "fp8_long_decode: batch 2, KV 131072, 32 q / 8 kv, page 128, FP8 E4M3 KV"),
            (5, 4096, "decode_fp8_long_window", "fp8_long_decode_window: as above, sliding window 4096")):
        b = W.workload(n, window_left=window)
        st = _device_state(b, device)
        plan = pk.Plan()
        plan.plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, **_plan_kw(b))
        info = plan.info()
        k_ms, mode = kernel_ms(lambda: plan.run(st["q"], st["cache"], out=st["out"]))
        gbs = b.kv_bytes_read() / (k_ms * 1e-3) / 1e9
        res.append({"workload": name, "kv_bytes": b.kv_bytes_read(), "kernel_ms": round(k_ms, 4),
                    "achieved": round(gbs, 2), "unit": "GB/s", "frac": round(gbs / hbm, 4),
                    "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4), "timing": mode,
                    "traffic": _traffic(key, DECODE_SOURCES),
                    "plan": {"ctas": info["num_work"], "merge_units": info["num_merge"], "kv_chunk": info["kv_chunk"]}})
        del st, plan
        torch.cuda.empty_cache()
    return res


def prefill_measure(device, steps, warmup, peak_tflops):
    """Prefix-cached extend (page size 1): plan + KV write + prefill per step, TFLOP/s."""
    import numpy as np
    import torch

    import paged_kv_attention_slot_gb300 as pk
    import workloads as W

    b = W.workload(3)
    st = _device_state(b, device)
    plan = pk.Plan()
    try:
        plan.plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, **_plan_kw(b))
    except pk.PkvError as e:
        return {"unavailable": e.message}
    # algorithmic FLOPs: 4 * D * Hq * sum over requests of the causally visible (query, key) pairs
    n = b.q_len.astype(np.float64)
    p = (b.kv_len - b.q_len).astype(np.float64)
    pairs = float(np.sum(n * p + n * (n + 1) / 2))
    flops = 4.0 * b.head_dim * b.num_qo_heads * pairs
    total_ms, _ = run_steps(b, st, plan, steps, warmup, False)
    _, run_ms = run_steps(b, st, plan, min(steps, 5), 1, False, record_run_events=True)  # diagnostic
    run_avg = statistics.mean(run_ms)
    plan_us = plan_host_us(b, plan)
    k_ms, k_mode = kernel_ms(lambda: plan.run(st["q"], st["cache"], out=st["out"]), reps=10, iters=5)
    achieved = flops / (k_ms * 1e-3) / 1e12
    return {
        "workload": "prefix_extend: batch 8, new U[128,2048], prefix U[0,4096], page 1, 32q/8kv, D 128, bf16",
        "metric": "prefill TFLOP/s (causally visible pairs)",
        "value": round(flops * steps / (total_ms * 1e-3) / 1e12, 2),
        "unit": "TFLOP/s",
        "ms_per_step": round(total_ms / steps, 4),
        "flops_per_step": flops,
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak_tflops, "unit": "TFLOP/s",
                     "frac": round(achieved / peak_tflops, 4), "kernel_ms": round(k_ms, 4), "timing": k_mode,
                     "traffic": _traffic("prefill", PREFILL_SOURCES)},
        "run_ms_mean_in_steps": round(run_avg, 4),
        "gpu_launches_per_step": 3,  # plan metadata copy + kv_store + prefill (no split items here)
        "plan_host_us": plan_us,
    }


def _visible_pairs(kv_len, q_len):
    import numpy as np

    n = q_len.astype(np.float64)
    p = (kv_len - q_len).astype(np.float64)
    return float(np.sum(n * p + n * (n + 1) / 2))


def next_rows_measure(device, peak_tflops, hbm):
    """The widened paths, each timed as a replayed CUDA graph of its launches on resident inputs."""
    import numpy as np
    import torch

    import paged_kv_attention_slot_gb300 as pk
    import workloads as W

    out = {}
    # (1) prefix-cached extend in the paged + merge form: ragged pass over the new tokens' own K/V,
    #     paged pass over the cached prefix (every prefix key visible), LSE merge in place
    b = W.workload(3)
    st = _device_state(b, device)
    pk.kv_store(st["k_new"], st["v_new"], st["slots"], st["cache"])
    kw = dict(num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, sm_scale=b.sm_scale)
    rag = pk.Plan().plan(b.qo_indptr, b.qo_indptr, None, None, mode="ragged", **kw)
    ps = b.page_size
    pre_len = (b.kv_len - b.q_len).astype(np.int64)
    npg = (pre_len + ps - 1) // ps
    pi = np.concatenate([[0], np.cumsum(npg)]).astype(np.int32)
    px = np.concatenate([b.kv_indices[b.kv_indptr[i]:b.kv_indptr[i] + npg[i]] for i in range(b.batch_size)])
    pl = np.where(npg > 0, pre_len - (npg - 1) * ps, 0).astype(np.int32)
    pre = pk.Plan().plan(b.qo_indptr, pi, px.astype(np.int32), pl, page_size=ps, mode="prefill", causal=False, **kw)
    o1, s1 = torch.empty_like(st["q"]), torch.empty(st["q"].shape[:2], dtype=torch.float32, device=device)
    o2, s2 = torch.empty_like(o1), torch.empty_like(s1)

    def extend_by_merge():
        rag.run_ragged(st["q"], st["k_new"], st["v_new"], out=o1, lse=s1)
        pre.run(st["q"], st["cache"], out=o2, lse=s2)
        pk.merge_state(o1, s1, o2, s2, out=o1, lse_out=s1)

    def extend_by_fused_merge():  # the prefix pass merges into the ragged pass's state in its epilogue
        rag.run_ragged(st["q"], st["k_new"], st["v_new"], out=o1, lse=s1)
        pre.run(st["q"], st["cache"], out=o1, lse=s1, merge_into=True)

    # one launch over both sources: prefix pages + the new tokens' contiguous rows, one online softmax
    one = pk.Plan().plan(b.qo_indptr, pi, px.astype(np.int32), pl, page_size=ps, mode="paged_ragged", **kw)

    def extend_one_pass():
        one.run_paged_ragged(st["q"], st["cache"], st["k_new"], st["v_new"], out=o1)

    flops = 4.0 * b.head_dim * b.num_qo_heads * _visible_pairs(b.kv_len, b.q_len)
    ms_one, mode = kernel_ms(extend_one_pass, reps=10, iters=5)
    ms, _ = kernel_ms(extend_by_merge, reps=10, iters=5)
    ms_fused, _ = kernel_ms(extend_by_fused_merge, reps=10, iters=5)
    tf = lambda t: flops / (t * 1e-3) / 1e12  # noqa: E731
    out["extend_by_merge"] = {
        "workload": "prefix_extend (as the prefill line) with the new tokens' K/V as contiguous (ragged) rows "
                    "and the cached prefix through the page table",
        "launches": 1, "ms": round(ms_one, 4), "tflops": round(tf(ms_one), 2),
        "frac": round(tf(ms_one) / peak_tflops, 4), "timing": mode,
        "how": "one prefill launch over both sources (PKV_MODE_PAGED_RAGGED), one online softmax, no merge",
        "plans": {"one_pass_ctas": one.info()["num_work"], "ragged_ctas": rag.info()["num_work"],
                  "prefix_ctas": pre.info()["num_work"]},
        "three_calls": {"launches": 3 + (1 if pre.info()["num_merge"] else 0), "ms": round(ms, 4),
                        "tflops": round(tf(ms), 2), "frac": round(tf(ms) / peak_tflops, 4),
                        "how": "ragged pass + paged prefix pass + LSE merge"},
        "fused": {"launches": 2, "ms": round(ms_fused, 4), "tflops": round(tf(ms_fused), 2),
                  "frac": round(tf(ms_fused) / peak_tflops, 4),
                  "how": "the paged prefix pass merges into the ragged pass's (o, lse) in its epilogue"}}
    del st, rag, pre, o1, o2, s1, s2
    torch.cuda.empty_cache()

    # (2) cascade: batch-64 decode sharing a 4096-token system prompt, against the flat decode plan
    b = W.shared_prefix_workload()
    st = _device_state(b, device)
    pk.kv_store(st["k_new"], st["v_new"], st["slots"], st["cache"])
    flat = pk.Plan().plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, **_plan_kw(b))
    ns = len(b.meta["shared_pages"])
    rows = [r[ns:] for r in b.block_rows]
    suf = (b.kv_len - b.meta["shared_prefix"]).astype(np.int64)
    si = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    sx = np.concatenate(rows).astype(np.int32)
    sl = np.array([x - (len(r) - 1) * b.page_size for x, r in zip(suf, rows)], dtype=np.int32)
    cas = pk.CascadePlan().plan(b.qo_indptr, b.meta["shared_pages"], b.page_size, si, sx, sl,
                                num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads, head_dim=b.head_dim,
                                page_size=b.page_size)
    lse = torch.empty(st["q"].shape[:2], dtype=torch.float32, device=device)
    flat_ms, mode = kernel_ms(lambda: flat.run(st["q"], st["cache"], out=st["out"]))
    cas_ms, _ = kernel_ms(lambda: cas.run(st["q"], st["cache"], out=st["out"], lse=lse))
    row_bytes = b.num_kv_heads * b.head_dim * 2 * 2
    flat_bytes = int(b.kv_len.sum()) * row_bytes
    unique_bytes = (b.meta["shared_prefix"] + int(suf.sum())) * row_bytes
    out["cascade_decode"] = {
        "workload": "shared_prefix_decode: batch 64, 32q/8kv, D 128, page 16, shared prefix 4096 + own suffix U[1,512]",
        "flat_decode_ms": round(flat_ms, 4), "cascade_ms": round(cas_ms, 4),
        "speedup": round(flat_ms / cas_ms, 3),
        "flat_kv_bytes": flat_bytes, "unique_kv_bytes": unique_bytes,
        "flat_gbs": round(flat_bytes / (flat_ms * 1e-3) / 1e9, 1),
        "cascade_unique_gbs": round(unique_bytes / (cas_ms * 1e-3) / 1e9, 1),
        "cascade_equivalent_gbs": round(flat_bytes / (cas_ms * 1e-3) / 1e9, 1),
        "launches": 2 + (1 if cas.shared.info()["num_prefill_partials"] else 0), "timing": mode,
        "how": "pkv_cascade_run: the suffix decode into (o, lse), then the shared non-causal pass merged in its epilogue",
        "plans": {"shared_ctas": cas.shared.info()["num_work"], "suffix_ctas": cas.suffix.info()["num_work"]}}
    del st, flat, cas, lse
    torch.cuda.empty_cache()

    # (3) long prefix, short extend: 2 requests x 256 new tokens after a 32768-token prefix (64 items
    #     on 152 SMs), with and without prefill split-KV
    b = W.make_batch([32768 + 256] * 2, [256] * 2, 16, 32, 8, 128, seed=1107, name="long_prefix_extend")
    st = _device_state(b, device)
    pk.kv_store(st["k_new"], st["v_new"], st["slots"], st["cache"])
    flops = 4.0 * b.head_dim * b.num_qo_heads * _visible_pairs(b.kv_len, b.q_len)
    res = {"workload": "long_prefix_extend: batch 2, prefix 32768, 256 new tokens, page 16, 32q/8kv, D 128"}
    for key, ms_ in (("split", 0), ("no_split", 1)):
        pl_ = pk.Plan().plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, max_splits=ms_, **_plan_kw(b))
        t, mode = kernel_ms(lambda: pl_.run(st["q"], st["cache"], out=st["out"]), reps=10, iters=5)
        res[key] = {"ms": round(t, 4), "tflops": round(flops / (t * 1e-3) / 1e12, 2),
                    "ctas": pl_.info()["num_work"], "partials": pl_.info()["num_prefill_partials"]}
    res["timing"] = mode
    out["long_prefix_extend"] = res
    del st
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--only-prefill", action="store_true", help="measure the prefill workload alone (profiling)")
    ap.add_argument("--no-other-decode", action="store_true", help="skip the other decode workloads")
    ap.add_argument("--no-next", action="store_true", help="skip the extend-by-merge / cascade / split measurements")
    ap.add_argument("--only-next", action="store_true", help="measure those alone")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return reference_arm(args, world, rank)
    if args.only_next:
        import torch

        import paged_kv_attention_slot_gb300 as pk

        torch.cuda.set_device(local_rank)
        pk._lib.lib()
        hbm, tf_burst, _, _ = _peaks()
        res = next_rows_measure(torch.device("cuda", local_rank), tf_burst, hbm)
        res["device_error"] = pk.device_error()
        print(json.dumps(res))
        return
    if args.only_prefill:
        import torch

        import paged_kv_attention_slot_gb300 as pk

        torch.cuda.set_device(local_rank)
        pk._lib.lib()
        res = prefill_measure(torch.device("cuda", local_rank), args.steps, args.warmup, _peaks()[1])
        res["device_error"] = pk.device_error()
        print(json.dumps(res))
        return

    import torch

    import paged_kv_attention_slot_gb300 as pk
    import workloads as W

    # the oracle pool is spawned before the first GPU call
    pool = OraclePool((2,) if args.no_prefill else (2, 3), 0) if (
        rank == 0 and world == 1 and not args.no_cpu_baseline) else None
    if pool is not None:
        pool.wait_ready()

    dist_on = world > 1
    if dist_on:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    pk._lib.lib()
    hbm, tf_burst, tf_sust, peak_src = _peaks()

    b = rank_batch(2, rank)
    st = _device_state(b, device)
    plan = pk.Plan()
    plan.plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, **_plan_kw(b))
    info = plan.info()

    clocks = ClockSampler(local_rank)
    clocks.start()
    total_ms, _ = run_steps(b, st, plan, args.steps, args.warmup, dist_on)
    clk = clocks.stop()
    max_ms = max_over_ranks(total_ms, device)
    kv_bytes = b.kv_bytes_read()
    value = aggregate_gbs(kv_bytes, args.steps, world, max_ms)

    e2e_steps = max(20, args.steps)
    e2e_dts, h2d, d2h, e2e_diff = run_e2e(b, st, plan, e2e_steps, 3)
    e2e_runs = [kv_bytes * e2e_steps / t / 1e9 for t in e2e_dts]
    e2e_val = statistics.median(e2e_runs)
    err = pk.device_error()

    _, run_ms = run_steps(b, st, plan, min(args.steps, 10), 1, False, record_run_events=True)  # diagnostic
    run_avg = statistics.mean(run_ms)
    plan_us = plan_host_us(b, plan)
    k_ms, k_mode = kernel_ms(lambda: plan.run(st["q"], st["cache"], out=st["out"]))
    achieved = kv_bytes / (k_ms * 1e-3) / 1e9
    launches_per_step = 3  # plan metadata copy + kv_store + decode (the split-KV merge runs inside decode)

    prefill = None
    if not args.no_prefill and rank == 0:
        prefill = prefill_measure(device, max(5, args.steps // 2), 3, tf_burst)
    other = None
    if not args.no_other_decode and rank == 0:
        other = decode_other_configs(device, hbm)
    nxt = None
    if not args.no_next and rank == 0:
        nxt = next_rows_measure(device, tf_burst, hbm)

    cpu = None
    if pool is not None:
        cpu = cpu_baseline(b, pool)
        if prefill is not None and "unavailable" not in prefill:
            prefill["cpu_baseline"] = cpu_baseline_prefill(pool)
        pool.close()

    if rank == 0:
        line = {
            "metric": "paged decode KV-read GB/s (% of HBM) and prefill TFLOP/s (% of bf16 peak)",
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(max_ms / args.steps, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 values, random page permutation)",
            "config": {
                "workload": DECODE_WORKLOAD,
                "batch": b.batch_size, "kv_tokens": int(b.kv_len.sum()), "kv_bytes_per_step": kv_bytes,
                "l2": "inputs larger than L2 (KV pool %.0f MB > 129 MB), no flush" % (
                    2 * st["k_pool"].numel() * 2 / 1e6),
                "parallelism": f"dp{world} (independent batches per GPU)",
                "plan": {"ctas": info["num_work"], "merge_units": info["num_merge"], "kv_chunk": info["kv_chunk"],
                         "host_us": plan_us},
            },
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm, "unit": "GB/s",
                         "frac": round(achieved / hbm, 4), "peak_source": peak_src,
                         "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                         "kernel": "decode_kernel (split-KV merge fused), one launch per decode_run",
                         "kernel_ms": round(k_ms, 4), "timing": k_mode,
                         "run_ms_mean_in_steps": round(run_avg, 4),
                         "traffic": _traffic("decode", DECODE_SOURCES)},
            "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps, "runs": [round(v, 1) for v in e2e_runs],
                    "max_abs_vs_device_path": round(e2e_diff, 5)},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu,
            "prefill": prefill,
            "decode_other_configs": other,
            "next_rows": nxt,
            "device_error": pk.device_error() if err == 0 else err,
        }
        print(json.dumps(line))
    if dist_on:
        torch.distributed.destroy_process_group()


def reference_arm(args, world, rank):
    """The oracle, as it stands, on the host cores; same workload, metric and unit as the GPU arm."""
    if rank != 0:
        return
    import workloads as W

    pool = OraclePool((2,), 0)
    pool.wait_ready()
    b = W.workload(2)
    ids = list(range(b.batch_size))
    per_step = ids[:8]  # bounded sample per step: 8 of the 64 requests
    for _ in range(args.warmup):
        pool.run(b, per_step[:2])
    total = 0.0
    for _ in range(args.steps):
        total += pool.run(b, per_step)
    pool.close()
    kv = _kv_bytes(b, per_step)
    value = kv * args.steps / total / 1e9
    sample = (f"each step: the attention of 8 of the 64 requests of the llama8b_decode batch ({kv / 1e6:.1f} MB of KV), "
              f"fp64 numpy oracle, one request per task on a spawn pool of {pool.cores} single-threaded processes")
    line = {
        "impl": "reference",
        "metric": "paged decode KV-read GB/s (% of HBM) and prefill TFLOP/s (% of bf16 peak)",
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 values, random page permutation)",
        "config": {"workload": DECODE_WORKLOAD},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": pool.cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
