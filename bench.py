#!/usr/bin/env python
"""Decode throughput of the QSA sparse path on GB300: rows/s of one decode
step (qsa_select_paged_tokens + qsa_sparse_attention) and the achieved HBM
bandwidth of the selection stage against the measured copy bandwidth.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 4]

Workload (default): 256 rows x 131072 tokens -- 32768 compressed keys per row
(256 compressed pages), 256 K/V pages of 512 tokens per row, pages randomly
permuted, FP16, about 34 GB resident per GPU; every step streams ~2.7 GB, far
more than the 129 MB L2, so no L2 flush is needed between steps.

Timing: W warm-up steps, then K steps bracketed by a barrier and a device
synchronize, timed with CUDA events on the launching stream (none inside the
loop); max over ranks.  The per-stage split (the roofline's selection time)
comes from a second loop with an event before, between and after the calls.
N > 1 (torchrun): every rank runs its own 256 rows (weak scaling, no
collective on the data path); value = all ranks' rows / max time.

--impl reference times the CPU oracle (test infrastructure, plain C) on the
host cores on a bounded sample of rows of the same workload.
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode rows/s (select+sparse attend) and achieved HBM GB/s vs GB300 peak"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic_R256_L131072.json")
NOMINAL_HBM_GBS = 7900.0      # GB300 HBM3e nominal (context; the roofline uses the measured copy rate)
SELECTION_SOURCES = ("qsa_select.cu", "qsa_select_impl.cuh", "qsa_device.cuh", "qsa_internal.h")


def _selection_traffic(workload: int, rows: int):
    """DRAM bytes per selection launch from the committed ncu summary, or
    None when the selection kernels changed since the capture (the hashes of
    their sources differ) or the workload is not the one captured."""
    import hashlib
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        if workload != 4 or rows != d["rows_scaled_to"]:
            return None
        csrc = os.path.join(ROOT, "sparse_paged_attention_qsa_gb300", "csrc")
        for name, digest in d["sources_sha256"].items():
            if name not in SELECTION_SOURCES:     # the figure covers the selection kernels
                continue
            with open(os.path.join(csrc, name), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != digest:
                    return None
        return int(d["selection_stage_bytes_per_launch"])
    except Exception:
        return None


def _peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# --- algorithmic bytes (what the method must move; duplicates once) ----------

def select_bytes_per_row(seq_len: int, pos: int) -> int:
    """visible keys (256 B each) + q_sel + page-table entries + index write +
    row metadata (request id, seq_len, position)."""
    V = max(0, min((pos + 1) // 4, seq_len // 4))
    return 256 * V + 4 * 128 * 2 + 4 * math.ceil(V / 128) + 4 * 2051 + 4 + 4 + 8


def select_bytes_per_row_fp8(seq_len: int, pos: int) -> int:
    """select_bytes_per_row with 1-byte (E4M3) compressed keys."""
    V = max(0, min((pos + 1) // 4, seq_len // 4))
    return 128 * V + 4 * 128 * 2 + 4 * math.ceil(V / 128) + 4 * 2051 + 4 + 4 + 8


def attend_bytes_per_row(idx_row: np.ndarray) -> int:
    """distinct valid tokens (1 KiB K+V each) + q + out + index read + the
    K/V page-table entries touched + request id."""
    v = np.unique(idx_row[idx_row >= 0])
    pages = np.unique(v // 512).size
    return 1024 * v.size + 3 * 256 * 2 * 2 + 4 * idx_row.size + 4 * pages + 4


# --- clocks during the timed region ----------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(parts)
            except Exception:
                pass
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


# --- distributed plumbing (host-side only) -----------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def max_over_ranks(x: float, world: int, device) -> float:
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


# --- CPU oracle baseline -----------------------------------------------------

class OracleSample:
    """Host copies of a few rows of a workload (their queries, tables and the
    pages they reference) so the CPU oracle can run one decode row at a time."""

    def __init__(self, w, rows):
        import oracle
        oracle.build()
        self.oracle = oracle
        self.rows = list(rows)
        t2r = w.token_to_request.cpu().numpy()
        self.cpt = w.cmp_page_table.cpu().numpy()
        self.kpt = w.kv_page_table.cpu().numpy()
        reqs = sorted({int(t2r[r]) for r in self.rows})
        self.q = w.q_sel.cpu().numpy()
        self.qa = w.q_attn.cpu().numpy()
        self.t2r, self.sl = t2r, w.seq_lens.cpu().numpy()
        self.qp = w.query_positions.cpu().numpy()
        self.cpool = self._pool(w.cmp_cache, self.cpt[reqs].ravel(), 128 * 128)
        self.kpool = self._pool(w.kv_cache, self.kpt[reqs].ravel(), 512 * 512)

    def _pool(self, cache, ids, halves):
        P = cache.shape[0]
        ids = sorted({int(p) for p in ids if 0 <= int(p) < P})
        sel = torch.tensor(ids, dtype=torch.long, device=cache.device)
        host = cache.index_select(0, sel).cpu().numpy().reshape(len(ids), -1)
        return self.oracle.PagePool({p: host[i] for i, p in enumerate(ids)}, num_pages=P,
                                    page_halves=halves)

    def run_row(self, k: int):
        """One decode row on the oracle: selection, then attention on it."""
        r = self.rows[k % len(self.rows)]
        o = self.oracle
        idx, _ = o.select(self.q[r:r + 1], self.cpool, self.cpt, self.t2r[r:r + 1], self.sl,
                          self.qp[r:r + 1])
        o.attention(self.qa[r:r + 1], self.kpool, self.kpt, self.t2r[r:r + 1], idx)


def host_cores():
    """(cores of the host, cores this process may run on): the oracle runs one
    thread per usable core."""
    total = os.cpu_count() or 1
    try:
        usable = len(os.sched_getaffinity(0))
    except Exception:
        usable = total
    return total, max(1, usable)


def oracle_rate(sample: OracleSample, n_rows: int, threads: int):
    """Rows/s of the oracle over n_rows decode rows spread over `threads` OS
    threads (the C code releases the GIL); returns (rows/s, wall seconds)."""
    from concurrent.futures import ThreadPoolExecutor
    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(sample.run_row, range(n_rows)))
    dt = time.perf_counter() - t0
    return n_rows / dt, dt


def _sample_workload(workload: int, rows: int, rank: int):
    from sparse_paged_attention_qsa_gb300 import workloads as W
    if torch.cuda.is_available():
        dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
        torch.cuda.set_device(dev)
        w = W.config(workload, device=dev, seed=1000 + workload + 7919 * rank)
    else:
        w = W.config(workload, device="cpu", rows=rows, seed=1000 + workload + 7919 * rank)
    return w


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle as it stands, on the host cores.  One
    step = one decode row of the workload (select + attend); the K timed steps
    run spread over the host threads."""
    if rank != 0:
        return 0
    from sparse_paged_attention_qsa_gb300 import workloads as W
    total_cores, threads = host_cores()
    w = _sample_workload(args.workload, threads, rank)
    sample = OracleSample(w, range(min(threads, w.R)))
    del w
    oracle_rate(sample, min(args.warmup, threads), threads)      # warm-up rows
    value, dt = oracle_rate(sample, args.steps, threads)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32/f64",
        "data": "synthetic",
        "config": {"workload": W.CONFIG_NAMES[args.workload], "rows_per_step": 1},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": threads,
                         "threads": threads, "host_cores": total_cores, "kind": "oracle",
                         "sample": f"{args.steps} decode rows (select+attend) cycling over "
                                   f"{len(sample.rows)} rows of {W.CONFIG_NAMES[args.workload]}, "
                                   f"plain C oracle on {threads} threads, {dt:.1f} s wall"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --- our arm -----------------------------------------------------------------

def run_ours(args, world, rank, local):
    import sparse_paged_attention_qsa_gb300 as qsa
    from sparse_paged_attention_qsa_gb300 import build as qbuild
    from sparse_paged_attention_qsa_gb300 import workloads as W

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the product path has no CPU fallback)")
    qbuild.build()
    qsa.load_library()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")

    w = W.config(args.workload, device=dev, seed=1000 + args.workload + 7919 * rank,
                 rows=args.rows)
    R = w.R
    stream = torch.cuda.current_stream(dev)
    idx = torch.empty((R, 2051), dtype=torch.int32, device=dev)
    out = torch.empty((R, 3, 256), dtype=torch.float16, device=dev)
    sel_ws = torch.empty(qsa.qsa_select_workspace_bytes(R, w.cmp_page_table.shape[1]),
                         dtype=torch.uint8, device=dev)
    att_ws = torch.empty(qsa.qsa_attention_workspace_bytes(R, 2051), dtype=torch.uint8,
                         device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    k_view, v_view = w.k_view, w.v_view

    def select():
        qsa.qsa_select_paged_tokens(w.q_sel, w.cmp_cache, w.cmp_page_table, w.token_to_request,
                                    w.seq_lens, w.query_positions, out=idx, workspace=sel_ws,
                                    error_word=err, stream=stream)

    def attend():
        qsa.qsa_sparse_attention(w.q_attn, k_view, v_view, w.kv_page_table, w.token_to_request,
                                 idx, out=out, workspace=att_ws, error_word=err, stream=stream)

    for _ in range(args.warmup):
        select()
        attend()
    torch.cuda.synchronize(dev)
    if int(err.item()) != 0:
        raise SystemExit(f"bench.py: device error word {int(err.item())}")

    # algorithmic bytes of this workload (from the produced index lists)
    seq = w.seq_lens.cpu().numpy()
    pos = w.query_positions.cpu().numpy()
    t2r = w.token_to_request.cpu().numpy()
    idx_h = idx.cpu().numpy()
    sel_bytes = sum(select_bytes_per_row(int(seq[t2r[r]]), int(pos[r])) for r in range(R))
    att_bytes = sum(attend_bytes_per_row(idx_h[r]) for r in range(R))

    # the step: K decode steps back to back, events only around the loop (an
    # event between the stages would itself cost time on the stream)
    K = args.steps
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        start.record(stream)
        for i in range(K):
            select()
            attend()
        end.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    total_ms = start.elapsed_time(end)
    t_step = max_over_ranks(total_ms / K, world, dev)
    value = R * world / (t_step * 1e-3)

    # the stages: a second loop with an event around each stage (the
    # selection stage's time is the roofline's)
    Ks = max(1, min(K, 200))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(Ks)]
    torch.cuda.synchronize(dev)
    for i in range(Ks):
        ev[i][0].record(stream)
        select()
        ev[i][1].record(stream)
        attend()
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    sel_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    att_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    staged_ms = statistics.mean(e[0].elapsed_time(e[2]) for e in ev)

    # end to end through the public API: one qsa_select_attend call per step
    # (the call a serving loop makes), every step's inputs from pinned host
    # memory and its results back to pinned host memory, inside the timed
    # region.  Pipelined like a serving loop: step i+1's inputs are copied in
    # (one copy stream) and step i's results read back (another) while step i
    # computes; inputs and outputs are double-buffered.
    names = ("q_sel", "q_attn", "token_to_request", "seq_lens", "query_positions",
             "cmp_page_table", "kv_page_table")
    h_in = {n: getattr(w, n).cpu().pin_memory() for n in names}
    d_in = [{n: getattr(w, n) for n in names},
            {n: torch.empty_like(getattr(w, n)) for n in names}]
    d_idx = [idx, torch.empty_like(idx)]
    d_out = [out, torch.empty_like(out)]
    h_idx = [torch.empty((R, 2051), dtype=torch.int32).pin_memory() for _ in range(2)]
    h_out = [torch.empty((R, 3, 256), dtype=torch.float16).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = h_idx[0].numel() * 4 + h_out[0].numel() * 2
    Ke = max(1, min(K, args.e2e_steps))
    one_ws = torch.empty(qsa.qsa_select_attend_workspace_bytes(R, w.cmp_page_table.shape[1]),
                         dtype=torch.uint8, device=dev)
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]      # inputs of buffer b are on the device
    ev_done = [torch.cuda.Event() for _ in range(2)]    # step on buffer b finished computing
    ev_read = [torch.cuda.Event() for _ in range(2)]    # results of buffer b are on the host
    for b in range(2):
        ev_done[b].record(stream)
        ev_read[b].record(stream)

    def e2e_step(i):
        b = i % 2
        s_in.wait_event(ev_done[b])               # the step that last read these inputs is done
        with torch.cuda.stream(s_in):
            for n, t in h_in.items():
                d_in[b][n].copy_(t, non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_read[b])             # the previous results of buffer b are read
        x = d_in[b]
        qsa.qsa_select_attend(x["q_sel"], w.cmp_cache, x["cmp_page_table"],
                              x["token_to_request"], x["seq_lens"], x["query_positions"],
                              x["q_attn"], k_view, v_view, x["kv_page_table"], indices=d_idx[b],
                              out=d_out[b], workspace=one_ws, error_word=err, stream=stream)
        ev_done[b].record(stream)
        s_out.wait_event(ev_done[b])
        with torch.cuda.stream(s_out):
            h_idx[b].copy_(d_idx[b], non_blocking=True)
            h_out[b].copy_(d_out[b], non_blocking=True)
        ev_read[b].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(Ke):
        e2e_step(i)
    stream.wait_event(ev_read[(Ke - 1) % 2])      # the last results are on the host
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_step_ms = max_over_ranks(e0.elapsed_time(e1) / Ke, world, dev)
    e2e_value = R * world / (e2e_step_ms * 1e-3)
    if int(err.item()) != 0:
        raise SystemExit(f"bench.py: device error word {int(err.item())}")
    if not np.array_equal(h_idx[(Ke - 1) % 2].numpy(), idx_h):
        raise SystemExit("bench.py: end-to-end indices differ from the device-timed step's")

    peak, peak_kind = _peaks()
    one_call = None
    if not args.no_one_call:
        one_call = one_call_variant(args, w, R, world, dev, stream, idx, out, err, peak,
                              sel_bytes + att_bytes)
    fp8 = None
    if not args.no_fp8:
        fp8 = fp8_variant(args, w, R, world, dev, stream, idx, out, att_ws, err, peak)
    meta = metadata_timing(args, R, world, dev, stream, w.cmp_page_table, w.seq_lens)
    r1 = None
    if not args.no_r1 and args.workload == 4:
        r1 = r1_latency(args, dev, stream)
    small = None
    if not args.no_r1 and args.workload == 4:
        small = small_batches(args, w, dev, stream, peak)
    spec = None
    if not args.no_spec and args.workload == 4:
        spec = spec_variant(args, R, world, rank, dev, stream, peak)
    indexer = None
    if not args.no_indexer and args.workload == 4:
        indexer = indexer_variant(args, world, rank, dev, stream, peak)
    sel_gbs = sel_bytes / (sel_ms * 1e-3) / 1e9
    att_gbs = att_bytes / (att_ms * 1e-3) / 1e9
    step_gbs = (sel_bytes + att_bytes) / (total_ms / K * 1e-3) / 1e9

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        total_cores, threads = host_cores()
        sample = OracleSample(w, range(min(threads, R)))
        rate0, _ = oracle_rate(sample, 2 * len(sample.rows), threads)   # calibration
        n = max(2 * len(sample.rows), int(rate0 * 10.0))                 # about 10 s of rows
        rate, dt = oracle_rate(sample, n, threads)
        n1 = max(2, int(rate / threads * 3.0))                           # about 3 s on one core
        rate1, _ = oracle_rate(sample, n1, 1)
        # the GPU step timed again after the CPU leg (GPU, CPU, GPU): its
        # drift from the first timing, in percent
        Kd = max(1, min(K, 100))
        d0 = torch.cuda.Event(enable_timing=True)
        d1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        d0.record(stream)
        for _ in range(Kd):
            select()
            attend()
        d1.record(stream)
        torch.cuda.synchronize(dev)
        drift = (d0.elapsed_time(d1) / Kd / (total_ms / K) - 1.0) * 100.0
        cpu = {"value": rate, "unit": "rows/s", "cores": threads, "threads": threads,
               "host_cores": total_cores, "kind": "oracle",
               "single_thread_value": rate1,
               "gpu_step_drift_pct": drift,
               "sample": f"{n} decode rows (select+attend) over {len(sample.rows)} rows of "
                         f"this workload, plain C oracle on {threads} threads, {dt:.1f} s wall"}

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": t_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": W.CONFIG_NAMES[args.workload], "rows_per_gpu": R,
                   "seq_len": int(seq[0]), "storage_dtype": "f16",
                   "l2": "inputs larger than L2 (each step streams "
                         f"{(sel_bytes + att_bytes) / 1e9:.2f} GB of a "
                         f"{(w.cmp_cache.numel() + w.kv_cache.numel()) * 2 / 1e9:.1f} GB "
                         "resident set; no flush)",
                   "step_hbm_gbs": step_gbs, "step_frac_of_peak": step_gbs / peak,
                   "step_frac_of_nominal": step_gbs / NOMINAL_HBM_GBS,
                   "select_ms": sel_ms, "attend_ms": att_ms, "attend_hbm_gbs": att_gbs,
                   "staged_step_ms": staged_ms,
                   "stage_timing": f"{Ks} steps with an event before, between and after the "
                                   "two calls (the step itself is timed without them)",
                   "algorithmic_bytes_per_step": sel_bytes + att_bytes,
                   "parallelism": f"rows sharded over {world} GPU(s), no collective"},
        "roofline": {"bound": "hbm", "kernel": "selection stage (score + top-k launches)",
                     "achieved": sel_gbs, "peak": peak, "unit": "GB/s",
                     "frac": sel_gbs / peak, "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": sel_bytes,
                     "traffic": _selection_traffic(args.workload, R)},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "rows/s", "api": "qsa_select_attend (one call per step)",
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_step_ms, "steps": Ke,
                "pipelining": "inputs of step i+1 and results of step i move on two copy "
                              "streams while step i computes (double-buffered)"},
        "one_call_select_attend": one_call,
        "fp8_compressed_cache": fp8,
        "metadata_builder": meta,
        "latency_R1": r1,
        "small_batches_L131072": small,
        "speculative_decode": spec,
        "paged_mqa_indexer": indexer,
        "gpu_launches": 4 * K,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def one_call_variant(args, w, R, world, dev, stream, idx, out, err, peak, step_bytes):
    """One decode step through qsa_select_attend (one fused kernel for a small
    batch, else the two calls' kernels from one call and one workspace), on
    the same workload and outputs."""
    import sparse_paged_attention_qsa_gb300 as qsa
    ws = torch.empty(qsa.qsa_select_attend_workspace_bytes(R, w.cmp_page_table.shape[1]),
                     dtype=torch.uint8, device=dev)

    def step():
        qsa.qsa_select_attend(w.q_sel, w.cmp_cache, w.cmp_page_table, w.token_to_request,
                              w.seq_lens, w.query_positions, w.q_attn, w.k_view, w.v_view,
                              w.kv_page_table, indices=idx, out=out, workspace=ws,
                              error_word=err, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    K = max(1, min(args.steps, 500))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    if int(err.item()) != 0:
        raise SystemExit(f"bench.py: device error word {int(err.item())} (one-call path)")
    ms = max_over_ranks(e0.elapsed_time(e1) / K, world, dev)
    gbs = step_bytes / (ms * 1e-3) / 1e9
    cs = qsa.qsa_select_attend_fused_cluster(R, w.cmp_page_table.shape[1], w.cmp_cache.dtype)
    return {"value": R * world / (ms * 1e-3), "unit": "rows/s", "ms_per_step": ms, "steps": K,
            "step_hbm_gbs": gbs, "step_frac_of_peak": gbs / peak,
            "path": f"fused (one cluster of {cs} CTAs per row)" if cs else "chained kernels",
            "launches_per_step": 1 if cs else 4}


def fp8_variant(args, w, R, world, dev, stream, idx, out, att_ws, err, peak):
    """The same decode step with the compressed keys stored as FP8 E4M3 (the
    optional e4m3 compressed indexer cache): the same draws rounded to E4M3,
    K/V and everything else shared.  Timed like the main measurement."""
    import sparse_paged_attention_qsa_gb300 as qsa
    cmp8 = w.cmp_cache.to(torch.float8_e4m3fn)
    sel_ws = torch.empty(qsa.qsa_select_workspace_bytes(R, w.cmp_page_table.shape[1]),
                         dtype=torch.uint8, device=dev)

    def step():
        qsa.qsa_select_paged_tokens(w.q_sel, cmp8, w.cmp_page_table, w.token_to_request,
                                    w.seq_lens, w.query_positions, out=idx, workspace=sel_ws,
                                    error_word=err, stream=stream)
        e_mid.record(stream) if e_mid is not None else None
        qsa.qsa_sparse_attention(w.q_attn, w.k_view, w.v_view, w.kv_page_table,
                                 w.token_to_request, idx, out=out, workspace=att_ws,
                                 error_word=err, stream=stream)

    e_mid = None
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    K = max(1, min(args.steps, 200))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    barrier(world)
    for i in range(K):
        ev[i][0].record(stream)
        e_mid = ev[i][1]
        step()
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    total = sum(e[0].elapsed_time(e[2]) for e in ev) / K
    sel_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    t_step = max_over_ranks(total, world, dev)
    seq = w.seq_lens.cpu().numpy()
    pos = w.query_positions.cpu().numpy()
    t2r = w.token_to_request.cpu().numpy()
    sel_bytes = sum(select_bytes_per_row_fp8(int(seq[t2r[r]]), int(pos[r])) for r in range(R))
    gbs = sel_bytes / (sel_ms * 1e-3) / 1e9
    del cmp8
    return {"value": R * world / (t_step * 1e-3), "unit": "rows/s", "ms_per_step": t_step,
            "steps": K, "select_ms": sel_ms, "select_hbm_gbs": gbs, "select_frac": gbs / peak,
            "select_algorithmic_bytes": sel_bytes}


def _time_calls(fn, n, stream, dev, world):
    for _ in range(3):
        fn()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        fn()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    return max_over_ranks(e0.elapsed_time(e1) / n, world, dev)


def r1_latency(args, dev, stream):
    """Single-row decode latency on the pages' two R=1 cases (519 tokens over
    two compressed pages; 9215 tokens, 2303 blocks in a pool of 8192 pages):
    microseconds per call of selection, attention, the two-call step and the
    one-call step.  Before every timed call a 256 MiB buffer is written so
    the call starts with its inputs out of L2; median and min of 50 calls.
    Also per call back to back: 64 steps captured in one CUDA graph (no host
    work between them; the row's inputs stay in L2), median of 10 replays."""
    import sparse_paged_attention_qsa_gb300 as qsa
    from sparse_paged_attention_qsa_gb300 import workloads as W
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {}
    for cfg in (0, 1):
        w = W.config(cfg, device=dev)
        idx = torch.empty((1, 2051), dtype=torch.int32, device=dev)
        o = torch.empty((1, 3, 256), dtype=torch.float16, device=dev)
        cols = w.cmp_page_table.shape[1]
        sws = torch.empty(qsa.qsa_select_workspace_bytes(1, cols), dtype=torch.uint8, device=dev)
        aws = torch.empty(qsa.qsa_attention_workspace_bytes(1, 2051), dtype=torch.uint8,
                          device=dev)
        fws = torch.empty(qsa.qsa_select_attend_workspace_bytes(1, cols), dtype=torch.uint8,
                          device=dev)

        def sel(s=stream):
            qsa.qsa_select_paged_tokens(w.q_sel, w.cmp_cache, w.cmp_page_table,
                                        w.token_to_request, w.seq_lens, w.query_positions,
                                        out=idx, workspace=sws, stream=s)

        def att(s=stream):
            qsa.qsa_sparse_attention(w.q_attn, w.k_view, w.v_view, w.kv_page_table,
                                     w.token_to_request, idx, out=o, workspace=aws,
                                     stream=s)

        def both(s=stream):
            sel(s)
            att(s)

        def fused(s=stream):
            qsa.qsa_select_attend(w.q_sel, w.cmp_cache, w.cmp_page_table, w.token_to_request,
                                  w.seq_lens, w.query_positions, w.q_attn, w.k_view, w.v_view,
                                  w.kv_page_table, indices=idx, out=o, workspace=fws,
                                  stream=s)

        res = {}
        for name, fn in (("select", sel), ("attend", att), ("two_call_step", both),
                         ("one_call_step", fused)):
            for _ in range(5):
                fn()
            ts = []
            for _ in range(50):
                flush.fill_(1)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                b.synchronize()
                ts.append(a.elapsed_time(b) * 1e3)
            res[name] = {"us_median": statistics.median(ts), "us_min": min(ts)}
        side = torch.cuda.Stream(dev)
        for name, fn in (("two_call_step", both), ("one_call_step", fused)):
            g = torch.cuda.CUDAGraph()
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                fn(side)
                side.synchronize()
                with torch.cuda.graph(g, stream=side):
                    for _ in range(64):
                        fn(side)
            stream.wait_stream(side)
            g.replay()
            ts = []
            for _ in range(10):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                g.replay()
                b.record(stream)
                b.synchronize()
                ts.append(a.elapsed_time(b) * 1e3 / 64)
            res[name]["back_to_back_us"] = statistics.median(ts)
            del g
        out[W.CONFIG_NAMES[cfg]] = res
    # the launch floor of this measurement: a one-element kernel timed the
    # same way (after the flush), for context
    one = torch.zeros(1, device=dev)
    ts = []
    for _ in range(50):
        flush.fill_(1)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        one.add_(1.0)
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b) * 1e3)
    out["trivial_kernel_after_flush"] = {"us_median": statistics.median(ts), "us_min": min(ts)}
    return out


def small_batches(args, w, dev, stream, peak):
    """Decode steps of a few rows (the first R rows of the long-context
    workload, 131072 tokens each) through qsa_select_attend -- one fused
    kernel while the device holds a cluster per row, the chained kernels
    above -- and through the two calls.  A 256 MiB buffer is written before every timed call, so
    each starts with its inputs out of L2; median of 30 calls.  frac = the
    step's algorithmic bytes at the measured HBM rate / the step's time."""
    import sparse_paged_attention_qsa_gb300 as qsa
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    seq = w.seq_lens.cpu().numpy()
    pos = w.query_positions.cpu().numpy()
    t2r = w.token_to_request.cpu().numpy()
    cols = w.cmp_page_table.shape[1]
    res = {}
    for R in (1, 2, 4, 8, 16, 24, 32, 40, 48, 56, 64, 72, 76, 96, 128, 144, 152):
        if R > w.R:
            break
        cs = qsa.qsa_select_attend_fused_cluster(R, cols)
        x = {n: getattr(w, n)[:R] for n in ("q_sel", "q_attn", "token_to_request",
                                            "query_positions")}
        idx = torch.empty((R, 2051), dtype=torch.int32, device=dev)
        o = torch.empty((R, 3, 256), dtype=torch.float16, device=dev)
        fws = torch.empty(qsa.qsa_select_attend_workspace_bytes(R, cols), dtype=torch.uint8,
                          device=dev)
        sws = torch.empty(qsa.qsa_select_workspace_bytes(R, cols), dtype=torch.uint8,
                          device=dev)
        aws = torch.empty(qsa.qsa_attention_workspace_bytes(R, 2051), dtype=torch.uint8,
                          device=dev)

        def one():
            qsa.qsa_select_attend(x["q_sel"], w.cmp_cache, w.cmp_page_table,
                                  x["token_to_request"], w.seq_lens, x["query_positions"],
                                  x["q_attn"], w.k_view, w.v_view, w.kv_page_table, indices=idx,
                                  out=o, workspace=fws, stream=stream)

        def two():
            qsa.qsa_select_paged_tokens(x["q_sel"], w.cmp_cache, w.cmp_page_table,
                                        x["token_to_request"], w.seq_lens, x["query_positions"],
                                        out=idx, workspace=sws, stream=stream)
            qsa.qsa_sparse_attention(x["q_attn"], w.k_view, w.v_view, w.kv_page_table,
                                     x["token_to_request"], idx, out=o, workspace=aws,
                                     stream=stream)

        row = {}
        for name, fn in (("one_call", one), ("two_call", two)):
            for _ in range(3):
                fn()
            ts = []
            for _ in range(30):
                flush.fill_(1)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                b.synchronize()
                ts.append(a.elapsed_time(b) * 1e3)
            row[name + "_us"] = statistics.median(ts)
        idx_h = idx.cpu().numpy()
        nbytes = sum(select_bytes_per_row(int(seq[t2r[r]]), int(pos[r])) +
                     attend_bytes_per_row(idx_h[r]) for r in range(R))
        floor_us = nbytes / (peak * 1e9) * 1e6
        row.update({"rows_per_s": R / (row["one_call_us"] * 1e-6),
                    "hbm_floor_us": floor_us, "frac_of_floor": floor_us / row["one_call_us"],
                    "path": (f"fused (one cluster of {cs} CTAs per row)" if cs
                             else "chained kernels")})
        res[f"R{R}"] = row
    return res


def metadata_timing(args, R, world, dev, stream, cmp_pt, seq):
    """The side-cache metadata builder (one launch) on this workload's batch:
    one query token per request, compressed-key slot map and work list."""
    import sparse_paged_attention_qsa_gb300 as qsa
    qsl = torch.arange(R + 1, dtype=torch.int32, device=dev)
    common = torch.arange(R, dtype=torch.int64, device=dev)
    outs = qsa.qsa_build_metadata(qsl, seq, cmp_pt, R, storage_block_size=128,
                                  compress_ratio=4, common_slot_mapping=common,
                                  num_mapped_tokens=R, max_num_work=2 * R, stream=stream)

    def call():
        qsa.qsa_build_metadata(qsl, seq, cmp_pt, R, storage_block_size=128, compress_ratio=4,
                               common_slot_mapping=common, num_mapped_tokens=R,
                               max_num_work=2 * R, out=outs, stream=stream)

    n = 2000
    ms = _time_calls(call, n, stream, dev, world)
    return {"us_per_call": ms * 1e3, "tokens": R, "requests": R, "work_items": 2 * R,
            "calls": n, "bound": "launch latency (a few KB per call)"}


def spec_variant(args, R, world, rank, dev, stream, peak):
    """Speculative / multi-token decode: R rows as R/4 requests x 4 query
    tokens (positions L-4 .. L-1, L = 131072).  One step = the metadata
    builder (token -> request, positions) + selection + attention, all on
    the device.  Inputs drawn like the main workload (own pools)."""
    import sparse_paged_attention_qsa_gb300 as qsa
    from sparse_paged_attention_qsa_gb300 import workloads as W
    nreq = max(1, R // 4)
    w = W.build("spec_R%d_%dx4_L131072" % (4 * nreq, nreq), [131072] * nreq,
                query_lens=[4] * nreq, cmp_pool=256 * nreq, kv_pool=256 * nreq,
                seed=4242 + 7919 * rank, device=dev)
    T = w.R
    common = torch.zeros(T, dtype=torch.int64, device=dev)
    meta = qsa.qsa_build_metadata(w.query_start_loc, w.seq_lens, w.cmp_page_table, T,
                                  storage_block_size=128, compress_ratio=4,
                                  common_slot_mapping=common, num_mapped_tokens=T,
                                  stream=stream)
    idx = torch.empty((T, 2051), dtype=torch.int32, device=dev)
    out = torch.empty((T, 3, 256), dtype=torch.float16, device=dev)
    sel_ws = torch.empty(qsa.qsa_select_workspace_bytes(T, w.cmp_page_table.shape[1]),
                         dtype=torch.uint8, device=dev)
    att_ws = torch.empty(qsa.qsa_attention_workspace_bytes(T, 2051), dtype=torch.uint8,
                         device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        qsa.qsa_build_metadata(w.query_start_loc, w.seq_lens, w.cmp_page_table, T,
                               storage_block_size=128, compress_ratio=4,
                               common_slot_mapping=common, num_mapped_tokens=T, out=meta,
                               stream=stream)
        qsa.qsa_decode(w.q_sel, w.cmp_cache, w.cmp_page_table, meta["token_to_req"],
                       w.seq_lens, meta["logical_positions"], w.q_attn, w.k_view, w.v_view,
                       w.kv_page_table, indices=idx, out=out, sel_workspace=sel_ws,
                       att_workspace=att_ws, error_word=err, stream=stream)

    K = max(1, min(args.steps, 200))
    ms = _time_calls(step, K, stream, dev, world)
    if int(err.item()) != 0:
        raise SystemExit(f"bench.py: device error word {int(err.item())} (speculative decode)")
    pos = meta["logical_positions"].cpu().numpy()
    idx_h = idx.cpu().numpy()
    row_sel = sum(select_bytes_per_row(131072, int(pos[r])) for r in range(T))
    # each request's keys once: the floor when the rows of a request share
    # one pass over its pages
    uniq_sel = sum(select_bytes_per_row(131072, 131071) for _ in range(nreq))
    att = sum(attend_bytes_per_row(idx_h[r]) for r in range(T))
    del w, idx, out, sel_ws, att_ws
    return {"workload": "R%d_%dreq_x4tok_L131072" % (T, nreq), "value": T * world / (ms * 1e-3),
            "unit": "rows/s", "ms_per_step": ms, "steps": K,
            "launches_per_step": 5,
            "algorithmic_bytes_rows_separate": row_sel + att,
            "algorithmic_bytes_keys_shared": uniq_sel + att,
            "frac_of_peak_rows_separate": (row_sel + att) / (ms * 1e-3) / 1e9 / peak,
            "frac_of_peak_keys_shared": (uniq_sel + att) / (ms * 1e-3) / 1e9 / peak}


def run_indexer_only(args, world, rank, local):
    """Only the indexer measurement, printed as its own JSON object (a small,
    self-contained case for profiling its kernels)."""
    import sparse_paged_attention_qsa_gb300 as qsa
    from sparse_paged_attention_qsa_gb300 import build as qbuild
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the product path has no CPU fallback)")
    qbuild.build()
    qsa.load_library()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    peak, _ = _peaks()
    res = indexer_variant(args, world, rank, dev, torch.cuda.current_stream(dev), peak)
    if rank == 0:
        print(json.dumps({"paged_mqa_indexer": res}), flush=True)
    return 0


def indexer_variant(args, world, rank, dev, stream, peak):
    """The weighted paged MQA indexer decode step (DeepSeek-V3.2 style):
    128 requests x 2 query tokens x 64 heads over 65536 cached tokens each
    (block size 64), FP8 tensor-core logits then the per-row top-2048.
    Inputs resident (1.1 GB of cache); each step streams the whole cache."""
    import sparse_paged_attention_qsa_gb300 as qsa
    from sparse_paged_attention_qsa_gb300 import workloads as W
    B, next_n, H, ctx, topk = 128, 2, 64, 65536, 2048
    ib = W.indexer_batch("indexer_B128_n2_H64_L65536", [ctx] * B, next_n=next_n, heads=H,
                         block_size=64, max_model_len=ctx, extra_blocks=0,
                         seed=777 + 7919 * rank, device=dev)
    rows = B * next_n
    logits = torch.empty((rows, ctx), dtype=torch.float32, device=dev)
    idx = torch.empty((rows, topk), dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def lg():
        qsa.qsa_paged_mqa_logits(ib.q, ib.kv_cache, ib.weights, ib.context_lens,
                                 ib.block_tables, next_n, ctx, block_size=64, out=logits,
                                 error_word=err, stream=stream)

    def tk():
        qsa.qsa_top_k_per_row_decode(logits, next_n, ib.context_lens, topk, out=idx,
                                     stream=stream)

    for _ in range(args.warmup):
        lg()
        tk()
    torch.cuda.synchronize(dev)
    if int(err.item()) != 0:
        raise SystemExit(f"bench.py: device error word {int(err.item())} (indexer)")
    K = max(1, min(args.steps, 200))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    barrier(world)
    for i in range(K):
        ev[i][0].record(stream)
        lg()
        ev[i][1].record(stream)
        tk()
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    lg_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    tk_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    step = max_over_ranks(statistics.mean(e[0].elapsed_time(e[2]) for e in ev), world, dev)
    cache_bytes = B * ctx * 132
    lg_bytes = cache_bytes + rows * H * (128 + 4) + rows * ctx * 4 + B * 4 + B * (ctx // 64) * 4
    tk_bytes = rows * ctx * 4 + rows * topk * 4 + B * 4
    flops = 2.0 * rows * ctx * H * 128
    gbs = lg_bytes / (lg_ms * 1e-3) / 1e9
    del ib, logits, idx
    return {"workload": "B128_nextn2_H64_L65536_bs64_top2048", "value": rows * world / (step * 1e-3),
            "unit": "rows/s", "ms_per_step": step, "steps": K, "logits_ms": lg_ms,
            "topk_ms": tk_ms, "logits_algorithmic_bytes": lg_bytes, "logits_hbm_gbs": gbs,
            "logits_frac_of_peak": gbs / peak, "logits_fp8_tflops": flops / (lg_ms * 1e-3) / 1e12,
            "topk_algorithmic_bytes": tk_bytes,
            "topk_gbs": tk_bytes / (tk_ms * 1e-3) / 1e9, "launches_per_step": 3}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=4, choices=[0, 1, 2, 3, 4])
    ap.add_argument("--rows", type=int, default=None,
                    help="keep only the first rows of a multi-row workload (profiling cases)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp8", action="store_true",
                    help="skip the FP8-E4M3 compressed-cache measurement")
    ap.add_argument("--no-r1", action="store_true",
                    help="skip the single-row latency measurement (workloads 0 and 1)")
    ap.add_argument("--no-one-call", "--no-fused", dest="no_one_call", action="store_true",
                    help="skip the one-call select+attend (qsa_select_attend) measurement")
    ap.add_argument("--no-spec", action="store_true",
                    help="skip the speculative-decode (4 tokens per request) measurement")
    ap.add_argument("--no-indexer", action="store_true",
                    help="skip the paged MQA indexer measurement")
    ap.add_argument("--indexer-only", action="store_true",
                    help="run only the paged MQA indexer measurement (profiling case)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("bench.py: at least 3 warm-up steps are required")
    world, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.indexer_only:
        return run_indexer_only(args, world, rank, local)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
