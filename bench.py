#!/usr/bin/env python
"""Benchmark: paged decode attention on GB300, one JSON line on stdout.

A step is one pass of the whole decode hot path over one batch: the cache
write of every sequence's new token (pa_reshape_and_cache), then the two
stream operations of pa_decode's balanced path: the zero fill of the arrival
counters (pa_decode_workspace_clear) and the persistent decode launch
(pa_decode_balanced), whose CTAs also combine the contexts cut between them.
With --path cascade (workloads whose block tables share prefix blocks) the
decode is pa_decode_cascade instead: the shared prefix for all query heads at
once, each sequence's own pages, and the combine. With --path int8 the same
batch is held as an INT8 cache with one fp32 scale per token and kv head: the
write is pa_reshape_and_cache_int8 and the decode pa_decode_int8 (counter
clear + the balanced decode launch).
Default workload: the
Mistral-7B-shaped bf16 batch (32 sequences, 32 query / 8 kv heads, head_dim
128, block_size 32, context lengths U[512, 4096], shuffled block pool).

value  = algorithmic bytes of a step (K/V of the attended tokens, q, output,
         block-table entries, context lengths, the new rows written) * steps
         / device time of the timed region, summed over ranks, in GB/s.
e2e    = the same metric through pa_decode with host buffers: per step the
         query, new K/V rows, slot mapping, lengths and tables are copied from
         pinned host memory, and the output is copied back.
roofline = the persistent decode kernel alone (CUDA events around each launch).

L2: the K/V caches are replicated 4 times (each replica larger than the
129 MB L2) and consecutive steps use different replicas.

--impl reference times the CPU oracle (fp64 C, all host cores) on a bounded
sample of the same workload, per step, and prints the same line.
"""
from __future__ import annotations

import argparse
import ctypes
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention: achieved HBM GB/s (% of GB300 peak) and seqs/s"
NOMINAL_HBM_GBS = 8000.0


# ------------------------------------------------------------------ traffic
def csrc_digest() -> str:
    """First 16 hex digits of sha256 over the library's CUDA sources."""
    import glob
    import hashlib
    m = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "paged_kv_cache_context_gb300", "csrc", "*"))):
        m.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            m.update(fh.read())
    return m.hexdigest()[:16]


def measured_traffic(key: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    capture keyed `key` (the workload for the balanced decode, else
    workload/path), or None when there is none or the sources changed since."""
    path = os.path.join(ROOT, "profiles", "paged_decode_kernel_traffic.txt")
    if not os.path.exists(path):
        return None
    digest = csrc_digest()
    with open(path) as fh:
        for line in fh:
            parts = line.split()
            if len(parts) == 3 and not line.startswith("#") and parts[0] == key \
                    and parts[1] == digest:
                return int(parts[2])
    return None


# ------------------------------------------------------------------ ranks
def rank_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def all_reduce(value: float, op: str, device=None) -> float:
    """max / sum of a float over the ranks of the default process group (the
    value itself when not distributed)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        window = [l for (t, l) in self.lines if t0 - 0.06 <= t <= t1 + 0.06] or \
                 [l for (_, l) in self.lines]
        for line in window:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ workload bytes
def step_bytes(case) -> dict:
    """Algorithmic bytes of one decode step."""
    S, Hq, Hkv, D, bs = (case.num_seqs, case.num_heads, case.num_kv_heads, case.head_dim,
                         case.block_size)
    qb = torch.finfo(case.q_dtype).bits // 8
    cb = 1 if case.kv_dtype in ("fp8_e4m3", "int8") else qb
    sb = torch.finfo(case.kv_src_dtype).bits // 8
    kv = case.kv_bytes()  # with an INT8 cache, the rows' scales too
    pages = sum(-(-case.attended(s) // bs) for s in range(S))
    new_rows = int((case.new_pos >= 0).sum())
    # what the decode launch must move: K/V of the attended rows once per kv
    # head, the queries read and the outputs written, one table entry per
    # page of a sequence, the context lengths
    kernel = kv + S * Hq * D * 2 * qb + pages * 4 + S * 4
    row_scale = 4 if case.kv_dtype == "int8" else 0
    write = new_rows * Hkv * (D * (sb + cb) + row_scale) * 2 + S * 8
    total = kernel + write
    return {"kv": kv, "kernel": kernel, "write": write, "total": total}


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


# ------------------------------------------------------------------ oracle timing
def oracle_step_time(case, rows_per_step: int, reps: int, build_all: bool = True):
    """Seconds per oracle step (write of the sample's new rows + decode of the
    sample's rows) on the host cores; the sample is the first rows_per_step
    (sequence, head) rows in sequence order."""
    import oracle  # test infrastructure: only this CPU-baseline leg uses it
    from paged_kv_cache_context_gb300 import workloads as wl
    Hq = case.num_heads
    nseq = min(case.num_seqs, -(-rows_per_step // Hq))
    kc, vc = wl.empty_caches(case)
    int8 = case.kv_dtype == "int8"
    ks, vs = wl.empty_scales(case) if int8 else (None, None)

    def write(key, val, sm):
        if int8:
            oracle.reshape_and_cache_int8(key, val, kc, vc, ks, vs, sm, case.block_size)
        else:
            oracle.reshape_and_cache(key, val, kc, vc, sm, case.block_size, case.kv_dtype,
                                     case.k_scale, case.v_scale)

    for s in range(nseq):
        pos, key, val = case.tokens_of(s)
        sm, _ = oracle.slot_mapping(case.block_tables, torch.full_like(pos, s), pos,
                                    case.block_size, case.window)
        write(key[:-1], val[:-1], sm[:-1])
    new_sm, _ = oracle.slot_mapping(case.block_tables, None, case.new_pos, case.block_size,
                                    case.window)
    new_sm[nseq:] = -1
    nk, nv = case.new_key.cpu(), case.new_value.cpu()
    q = case.query.cpu()
    rows = list(range(min(rows_per_step, case.num_seqs * Hq)))
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        write(nk, nv, new_sm)
        oracle.decode(q, kc, vc, case.block_tables, case.context_lens, case.num_kv_heads,
                      case.block_size, case.scale, case.window, case.kv_dtype, case.k_scale,
                      case.v_scale, rows=rows, k_scales=ks, v_scales=vs)
        times.append(time.perf_counter() - t0)
    # the same algorithmic bytes as the GPU step: the K/V rows a (sequence,
    # kv head) attends count once for the G query-head rows that share them
    G = Hq // case.num_kv_heads
    sample_bytes = 0
    for r in rows:
        s = r // Hq
        elem = (1 if case.kv_dtype in ("fp8_e4m3", "int8")
                else torch.finfo(case.q_dtype).bits // 8)
        sample_bytes += case.attended(s) * 2 * (case.head_dim * elem + (4 if int8 else 0))
    return times, sample_bytes / G, len(rows)


def cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, local_rank, world):
    from paged_kv_cache_context_gb300 import build, pa
    from paged_kv_cache_context_gb300 import workloads as wl
    build.build()
    L = pa.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    sp = ctypes.c_void_p(stream.cuda_stream)

    case = wl.config(args.workload, value_device=str(dev),
                     seed=None if rank == 0 else 50_000 + rank)
    int8 = args.path == "int8"
    if int8:
        if case.kv_dtype != "auto" or case.q_dtype == torch.float32:
            raise SystemExit("--path int8 needs a workload with a bf16/f16 native cache")
        case = dataclasses.replace(case, kv_dtype="int8")
    if args.path == "cascade" and args.cascade_kv != "auto":
        if case.kv_dtype != "auto" or case.q_dtype == torch.float32:
            raise SystemExit("--cascade-kv needs a workload with a bf16/f16 native cache")
        if args.cascade_kv == "int8":
            case = dataclasses.replace(case, kv_dtype="int8")
        else:
            # per-tensor scales amax / 448 over every row written, in fp32
            def amax(ts):
                return max(float(t.float().abs().max()) for t in ts if t.numel())
            case = dataclasses.replace(case, kv_dtype="fp8_e4m3",
                                       k_scale=amax([case.pre_key, case.new_key]) / 448.0,
                                       v_scale=amax([case.pre_value, case.new_value]) / 448.0)
    int8_cache = case.kv_dtype == "int8"  # rows written with per-row scales
    S, Hq, Hkv, D, bs = (case.num_seqs, case.num_heads, case.num_kv_heads, case.head_dim,
                         case.block_size)
    MB, NB = case.max_blocks_per_seq, case.num_blocks
    bt = case.block_tables.to(dev)
    cl = case.context_lens.to(dev)
    q = case.query.to(dev).contiguous()

    # caches: prefill rows written by the library itself
    kc, vc = wl.empty_caches(case, device=str(dev))
    ks, vs = wl.empty_scales(case, device=str(dev)) if int8_cache else (None, None)
    for a, b in case.pre_chunks:
        if b > a:
            sm = torch.empty(b - a, dtype=torch.int64, device=dev)
            pa.slot_mapping(sm, bt, case.pre_seq[a:b].to(dev), case.pre_pos[a:b].to(dev), bs,
                            case.window)
            if int8_cache:
                pa.reshape_and_cache_int8(case.pre_key[a:b].contiguous(),
                                          case.pre_value[a:b].contiguous(), kc, vc, ks, vs, sm)
            else:
                pa.reshape_and_cache(case.pre_key[a:b].contiguous(),
                                     case.pre_value[a:b].contiguous(), kc, vc, sm, case.kv_dtype,
                                     case.k_scale, case.v_scale)
    new_sm = torch.empty(S, dtype=torch.int64, device=dev)
    pa.slot_mapping(new_sm, bt, None, case.new_pos.to(dev), bs, case.window)
    new_k = case.new_key.to(dev).contiguous()
    new_v = case.new_value.to(dev).contiguous()
    torch.cuda.synchronize()
    def clone(t):
        return None if t is None else t.clone()
    reps = [(kc, vc, ks, vs)] + [tuple(clone(t) for t in (kc, vc, ks, vs))
                                 for _ in range(args.replicas - 1)]

    qd = pa._DTYPE[case.q_dtype]
    kvd = pa._KV[case.kv_dtype]
    out = torch.empty(S, Hq, D, dtype=case.q_dtype, device=dev)
    ws_bytes = pa.decode_workspace_size(S, Hq, Hkv, D, bs, MB, case.window)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    num_ctas = ctypes.c_int(0)

    # pre-bound C calls (marshalling once, outside the timed loop)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    def ptr(t):
        return P(t.data_ptr())
    write_args, dec_args = [], []
    for (k_, v_, _, _) in reps:
        write_args.append((ptr(new_k), ptr(new_v), ptr(k_), ptr(v_), ptr(new_sm), I(S), I(Hkv),
                           I(D), I(bs), I(NB), I(pa._DTYPE[new_k.dtype]), I(kvd),
                           F(case.k_scale), F(case.v_scale), sp))
        dec_args.append((ptr(out), ptr(q), ptr(k_), ptr(v_), ptr(bt), ptr(cl), I(S), I(Hq),
                         I(Hkv), I(D), I(bs), I(NB), I(MB), F(case.scale), I(case.window), I(qd),
                         I(kvd), F(case.k_scale), F(case.v_scale), ptr(ws), Z(ws_bytes),
                         P(ctypes.addressof(num_ctas)), sp))
    f_write, f_clear, f_dec = (L.pa_reshape_and_cache, L.pa_decode_workspace_clear,
                               L.pa_decode_balanced)
    clear_args = (ptr(ws), Z(ws_bytes), sp)
    if not int8_cache and (f_clear(*clear_args) or f_dec(*dec_args[0])):
        raise RuntimeError("pa_decode_balanced failed")
    if int8_cache:
        # pa_reshape_and_cache_int8: codes and row scales
        write_args = [(ptr(new_k), ptr(new_v), ptr(k_), ptr(v_), ptr(ks_), ptr(vs_),
                       ptr(new_sm), I(S), I(Hkv), I(D), I(bs), I(NB),
                       I(pa._DTYPE[new_k.dtype]), sp) for (k_, v_, ks_, vs_) in reps]
        f_write = L.pa_reshape_and_cache_int8
    launches_per_step = 3  # cache write, counter clear, decode
    prefix_pages = case.shared_prefix_tokens // bs
    if args.path == "cascade":
        # pa_decode_cascade: prefix attention + suffix decode + reduce
        if prefix_pages < 1:
            raise SystemExit("--path cascade needs a workload with a shared prefix")
        ws_bytes = pa.decode_cascade_workspace_size(S, Hq, Hkv, D, bs, prefix_pages)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        if case.kv_dtype == "fp8_e4m3":
            dec_args = [(ptr(out), ptr(q), ptr(k_), ptr(v_), ptr(bt), ptr(cl), I(S), I(Hq),
                         I(Hkv), I(D), I(bs), I(NB), I(MB), F(case.scale), F(case.k_scale),
                         F(case.v_scale), I(qd), I(prefix_pages), ptr(ws), Z(ws_bytes), sp)
                        for (k_, v_, _, _) in reps]
            f_dec = L.pa_decode_cascade_fp8
        elif int8_cache:
            dec_args = [(ptr(out), ptr(q), ptr(k_), ptr(v_), ptr(ks_), ptr(vs_), ptr(bt),
                         ptr(cl), I(S), I(Hq), I(Hkv), I(D), I(bs), I(NB), I(MB), F(case.scale),
                         I(qd), I(prefix_pages), ptr(ws), Z(ws_bytes), sp)
                        for (k_, v_, ks_, vs_) in reps]
            f_dec = L.pa_decode_cascade_int8
        else:
            dec_args = [(ptr(out), ptr(q), ptr(k_), ptr(v_), ptr(bt), ptr(cl), I(S), I(Hq),
                         I(Hkv), I(D), I(bs), I(NB), I(MB), F(case.scale), I(qd),
                         I(prefix_pages), ptr(ws), Z(ws_bytes), sp) for (k_, v_, _, _) in reps]
            f_dec = L.pa_decode_cascade
        if f_write(*write_args[0]) or f_dec(*dec_args[0]):
            raise RuntimeError("pa_decode_cascade failed")
        launches_per_step = 4  # cache write, prefix attention, suffix decode, reduce
    if int8:
        # pa_reshape_and_cache_int8, then pa_decode_int8 (counter clear + balanced decode)
        write_args = [(ptr(new_k), ptr(new_v), ptr(k_), ptr(v_), ptr(ks_), ptr(vs_),
                       ptr(new_sm), I(S), I(Hkv), I(D), I(bs), I(NB),
                       I(pa._DTYPE[new_k.dtype]), sp) for (k_, v_, ks_, vs_) in reps]
        dec_args = [(ptr(out), ptr(q), ptr(k_), ptr(v_), ptr(ks_), ptr(vs_), ptr(bt), ptr(cl),
                     I(S), I(Hq), I(Hkv), I(D), I(bs), I(NB), I(MB), F(case.scale),
                     I(case.window), I(qd), ptr(ws), Z(ws_bytes), sp)
                    for (k_, v_, ks_, vs_) in reps]
        f_write, f_dec = L.pa_reshape_and_cache_int8, L.pa_decode_int8
        if f_write(*write_args[0]) or f_dec(*dec_args[0]):
            raise RuntimeError("pa_decode_int8 failed")
        launches_per_step = 3  # cache write, counter clear, decode

    def step(i, ev_a=None, ev_b=None):
        r = i % len(reps)
        rc = f_write(*write_args[r])
        if args.path == "balanced":
            rc |= f_clear(*clear_args)
        if ev_a is not None:
            ev_a.record(stream)
        rc |= f_dec(*dec_args[r])
        if ev_b is not None:
            ev_b.record(stream)
        if rc:
            raise RuntimeError(f"library call failed: {rc}")

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if pa.get_device_error():
        raise RuntimeError("device error word set after warm-up")

    K = args.steps
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    vis = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    phys = int(vis[local_rank]) if local_rank < len(vis) and vis[local_rank].strip().isdigit() \
        else local_rank
    clocks = ClockSampler(phys)
    clocks.start()
    time.sleep(0.3)
    barrier(dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e0.record(stream)
    for i in range(K):
        step(i, ev_a[i], ev_b[i])
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    barrier(dev)
    clk = clocks.stop(t0, t1)
    if pa.get_device_error():
        raise RuntimeError("device error word set in the timed region")
    elapsed = e0.elapsed_time(e1) / 1e3
    split_ms = [a.elapsed_time(b) for a, b in zip(ev_a, ev_b)]

    sb = step_bytes(case)
    if args.path == "cascade":
        # HBM bytes the cascade must move: the prefix K/V once per kv head for
        # the whole batch, each sequence's own K/V, q and out, and the
        # partials (fp32, written and read once) of the prefix ranges and the
        # suffix
        nslots = ws_bytes // (4 * S * Hq * (D + 2))
        elem = torch.finfo(case.q_dtype).bits // 8
        row_b = D * (1 if case.kv_dtype != "auto" else elem) + (4 if int8_cache else 0)
        unique_kv = (case.shared_prefix_tokens + sum(
            case.attended(s) - case.shared_prefix_tokens for s in range(S))) * Hkv * 2 * row_b
        sb["kernel"] = (unique_kv + S * Hq * D * 2 * elem + 2 * S * Hq * nslots * (D + 2) * 4 +
                        S * MB * 4 + S * 4)
    elapsed_max = all_reduce(elapsed, "max", dev)
    bytes_all = all_reduce(float(sb["total"] * K), "sum", dev)
    seqs_all = all_reduce(float(S * K), "sum", dev)
    split_mean = statistics.mean(split_ms) / 1e3
    peak, peak_kind = peaks()
    achieved = sb["kernel"] / split_mean / 1e9

    # ---- the cache write at prefill scale: every context token of the batch
    write_prefill = None
    if not int8_cache and case.pre_key.shape[0] > 0:
        write_prefill = prefill_scale_write(case, pa, dev, stream, bt, reps)

    # ---- e2e: the public pa_decode call with host buffers
    e2e = run_e2e(args, case, pa, L, dev, stream, reps, new_sm, bt, cl, q, new_k, new_v, out,
                  sb, world)

    result = {
        "metric": METRIC, "value": round(bytes_all / elapsed_max / 1e9, 2), "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(elapsed_max / K * 1e3, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "impl": "ours",
        "config": {"workload": args.workload, "num_seqs": S, "num_heads": Hq,
                   "num_kv_heads": Hkv, "head_dim": D, "block_size": bs,
                   "window": case.window, "cache_dtype": case.kv_dtype if case.kv_dtype != "auto"
                   else str(case.q_dtype).replace("torch.", ""),
                   "storage_dtype": str(case.q_dtype).replace("torch.", ""),
                   "decode_path": args.path,
                   "decode_ctas": num_ctas.value if args.path == "balanced" else None,
                   "workspace_bytes": ws_bytes,
                   "kv_bytes_per_step": sb["kv"], "bytes_per_step": sb["total"],
                   "l2": f"{args.replicas} rotating cache replicas of "
                         f"{kc.numel() * kc.element_size() * 2 / 1e6:.0f} MB (> L2)",
                   "parallelism": f"replicas x{world} (independent batches, no collective)"},
        "seqs_per_s": round(seqs_all / elapsed_max, 1),
        "pct_of_nominal_8tbs": round(100 * bytes_all / elapsed_max / 1e9 / NOMINAL_HBM_GBS, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": (measured_traffic(args.workload) if args.path == "balanced"
                                 else measured_traffic(f"{args.workload}/{args.path}")
                                 if args.path == "int8" else None),
                     "kernel": {"cascade": {"auto": "pa_decode_cascade",
                                            "fp8_e4m3": "pa_decode_cascade_fp8",
                                            "int8": "pa_decode_cascade_int8"}[case.kv_dtype] +
                                           ": prefix attention + suffix decode + reduce",
                                "int8": "pa_decode_int8: counter clear + paged_decode_kernel "
                                        "(balanced mode, INT8 rows and row scales)",
                                "balanced": "paged_decode_kernel (balanced mode)"}[args.path],
                     "kernel_bytes_per_launch": sb["kernel"],
                     "kernel_us_mean": round(split_mean * 1e6, 2),
                     "kernel_us_median": round(statistics.median(split_ms) * 1e3, 2)},
        "e2e": e2e,
        "write_prefill_scale": write_prefill,
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
        "wall_s_timed": round(t1 - t0, 4),
    }
    if rank == 0:
        result["cpu_baseline"] = (None if args.skip_cpu_baseline else cpu_baseline(case, args))
        print(json.dumps(result), flush=True)


def prefill_scale_write(case, pa, dev, stream, bt, reps):
    """pa_reshape_and_cache of every context token of the batch in one call
    (T = sum of the context lengths minus the step's new tokens), timed with
    CUDA events on the launching stream, alternating cache replicas."""
    S, Hkv, D = case.num_seqs, case.num_kv_heads, case.head_dim
    T = int(case.pre_key.shape[0])
    key = case.pre_key.to(dev).contiguous()
    val = case.pre_value.to(dev).contiguous()
    sm = torch.empty(T, dtype=torch.int64, device=dev)
    pa.slot_mapping(sm, bt, case.pre_seq.to(dev), case.pre_pos.to(dev), case.block_size,
                    case.window)
    sb = key.element_size()
    cb = 1 if case.kv_dtype == "fp8_e4m3" else sb
    nbytes = T * Hkv * D * (sb + cb) * 2 + T * 8
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(8)]
    for i in range(3 + len(ev)):
        k_, v_ = reps[i % len(reps)][:2]
        if i >= 3:
            ev[i - 3][0].record(stream)
        pa.reshape_and_cache(key, val, k_, v_, sm, case.kv_dtype, case.k_scale, case.v_scale,
                             stream=stream)
        if i >= 3:
            ev[i - 3][1].record(stream)
    torch.cuda.synchronize()
    us = statistics.median(a.elapsed_time(b) for a, b in ev) * 1e3
    peak, kind = peaks()
    return {"tokens": T, "bytes": nbytes, "us": round(us, 2),
            "value": round(nbytes / us / 1e3, 1), "unit": "GB/s",
            "frac": round(nbytes / us / 1e3 / peak, 4), "peak_kind": kind,
            "what": "pa_reshape_and_cache of every context token (read rows, write pages, "
                    "slots), one call, CUDA events, median of 8"}


def run_e2e(args, case, pa, L, dev, stream, reps, new_sm, bt, cl, q, new_k, new_v, out, sb,
            world):
    """pa_reshape_and_cache + pa_decode from pinned host buffers, output back
    to pinned host memory, every step."""
    S, Hq, Hkv, D = case.num_seqs, case.num_heads, case.num_kv_heads, case.head_dim
    host = {n: t.cpu().pin_memory() for n, t in
            (("q", q), ("k", new_k), ("v", new_v), ("sm", new_sm), ("cl", cl), ("bt", bt))}
    dev_bufs = {n: torch.empty_like(t, device=dev) for n, t in host.items()}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    prefix_pages = case.shared_prefix_tokens // case.block_size
    if args.path == "cascade":
        wsb = pa.decode_cascade_workspace_size(S, Hq, Hkv, D, case.block_size, prefix_pages)
    else:
        wsb = pa.decode_workspace_size(S, Hq, Hkv, D, case.block_size, case.max_blocks_per_seq,
                                       case.window)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size()
    K = args.steps

    def step(i):
        k_, v_, ks_, vs_ = reps[i % len(reps)]
        for n, t in host.items():
            dev_bufs[n].copy_(t, non_blocking=True)
        if args.path == "int8":
            pa.reshape_and_cache_int8(dev_bufs["k"], dev_bufs["v"], k_, v_, ks_, vs_,
                                      dev_bufs["sm"])
            pa.decode_int8(out, dev_bufs["q"], k_, v_, ks_, vs_, dev_bufs["bt"], dev_bufs["cl"],
                           Hkv, case.scale, case.window, ws)
            out_h.copy_(out, non_blocking=True)
            return
        if case.kv_dtype == "int8":
            pa.reshape_and_cache_int8(dev_bufs["k"], dev_bufs["v"], k_, v_, ks_, vs_,
                                      dev_bufs["sm"])
        else:
            pa.reshape_and_cache(dev_bufs["k"], dev_bufs["v"], k_, v_, dev_bufs["sm"],
                                 case.kv_dtype, case.k_scale, case.v_scale)
        if args.path == "cascade" and case.kv_dtype == "fp8_e4m3":
            pa.decode_cascade_fp8(out, dev_bufs["q"], k_, v_, dev_bufs["bt"], dev_bufs["cl"],
                                  Hkv, case.scale, case.k_scale, case.v_scale, prefix_pages, ws)
        elif args.path == "cascade" and case.kv_dtype == "int8":
            pa.decode_cascade_int8(out, dev_bufs["q"], k_, v_, ks_, vs_, dev_bufs["bt"],
                                   dev_bufs["cl"], Hkv, case.scale, prefix_pages, ws)
        elif args.path == "cascade":
            pa.decode_cascade(out, dev_bufs["q"], k_, v_, dev_bufs["bt"], dev_bufs["cl"], Hkv,
                              case.scale, prefix_pages, ws)
        else:
            pa.decode(out, dev_bufs["q"], k_, v_, dev_bufs["bt"], dev_bufs["cl"], Hkv,
                      case.scale, case.window, case.kv_dtype, case.k_scale, case.v_scale, ws)
        out_h.copy_(out, non_blocking=True)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(K):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    el = all_reduce(e0.elapsed_time(e1) / 1e3, "max", dev)
    tot = all_reduce(float(sb["total"] * K), "sum", dev)
    return {"value": round(tot / el / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(el / K * 1e3, 5)}


def cpu_baseline(case, args):
    """The oracle on the host cores, bounded to ~10-20 s: the whole batch on
    every core, then a sample of rows on one thread."""
    import oracle  # test infrastructure: only this CPU-baseline leg uses it
    rows_total = case.num_seqs * case.num_heads
    times, sbytes, nrows = oracle_step_time(case, rows_total, 1)
    per = times[0]
    reps = max(1, min(20, int(12.0 / max(per, 1e-3))))
    if reps > 1:
        times, sbytes, nrows = oracle_step_time(case, rows_total, reps)
    t = statistics.median(times)
    # one thread, on the rows of the first sequences (about 5 s of work)
    per_row = t * cores() / max(nrows, 1)
    rows1 = max(1, min(rows_total, int(5.0 / max(per_row, 1e-6))))
    prev = oracle.set_threads(1)
    try:
        t1, b1, n1 = oracle_step_time(case, rows1, 1)
    finally:
        oracle.set_threads(prev)
    one = {"value": round(b1 / t1[0] / 1e9, 4), "unit": "GB/s", "cores": 1,
           "seconds_per_step": round(t1[0] / n1 * rows_total, 4),
           "sample": f"{n1} of {rows_total} sequence-head rows; seconds_per_step "
                     "scales the sample's time per row to the whole batch"}
    return {"value": round(sbytes / t / 1e9, 4), "unit": "GB/s", "cores": cores(),
            "kind": "oracle", "seconds_per_step": round(t, 4),
            "sample": f"whole batch ({nrows} sequence-head rows) x {len(times)} reps: oracle "
                      "write of the new rows + fp64 decode, OpenMP over rows",
            "single_thread": one}


# ------------------------------------------------------------------ paged prefill
def run_prefill(args, rank, local_rank, world):
    """--path prefill: pa_prefill, causal multi-query attention over the paged
    cache, on the workload's batch with its whole context already cached: the
    last --prefill-tokens positions of every sequence (fewer when shorter) are
    the query chunk. A dense contraction, so the roofline is the tensor pipe:
    algorithmic FLOPs = 4 * D * Hq * sum over query tokens of (position + 1)
    (Q K^T and P V, two operations per multiply-add), against the measured
    bf16 tensor throughput."""
    from paged_kv_cache_context_gb300 import build, pa
    from paged_kv_cache_context_gb300 import workloads as wl
    build.build()
    pa.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    case = wl.config(args.workload, value_device=str(dev),
                     seed=None if rank == 0 else 50_000 + rank)
    if case.kv_dtype != "auto" or case.q_dtype == torch.float32 or case.window:
        raise SystemExit("--path prefill needs a bf16/f16 workload without a window")
    S, Hq, Hkv, D, bs = (case.num_seqs, case.num_heads, case.num_kv_heads, case.head_dim,
                         case.block_size)
    int8 = args.prefill_int8
    fp8 = args.prefill_fp8 and not int8
    if int8:
        case = dataclasses.replace(case, kv_dtype="int8")
    if fp8:
        # per-tensor scales amax / 448 over every row written, in fp32
        def amax(chunks):
            return max(float(t.float().abs().max()) for t in chunks if t.numel())
        ksc = amax([case.pre_key, case.new_key]) / 448.0
        vsc = amax([case.pre_value, case.new_value]) / 448.0
        case = dataclasses.replace(case, kv_dtype="fp8_e4m3", k_scale=ksc, v_scale=vsc)
    bt = case.block_tables.to(dev)
    cl = case.context_lens.to(dev)
    kc, vc = wl.empty_caches(case, device=str(dev))
    ks, vs = wl.empty_scales(case, device=str(dev)) if int8 else (None, None)
    for seq, pos, key, val in [(case.pre_seq[a:b], case.pre_pos[a:b], case.pre_key[a:b],
                                case.pre_value[a:b]) for a, b in case.pre_chunks if b > a] + \
            [(None, case.new_pos, case.new_key, case.new_value)]:
        sm = torch.empty(pos.numel(), dtype=torch.int64, device=dev)
        pa.slot_mapping(sm, bt, None if seq is None else seq.to(dev), pos.to(dev), bs, 0)
        if int8:
            pa.reshape_and_cache_int8(key.to(dev).contiguous(), val.to(dev).contiguous(), kc, vc,
                                      ks, vs, sm)
        else:
            pa.reshape_and_cache(key.to(dev).contiguous(), val.to(dev).contiguous(), kc, vc, sm,
                                 case.kv_dtype, case.k_scale, case.v_scale)
    reps = [(kc, vc, ks, vs)] + [(kc.clone(), vc.clone(),
                                  None if ks is None else ks.clone(),
                                  None if vs is None else vs.clone())
                                 for _ in range(args.replicas - 1)]
    query, q_seq, q_pos = wl.prefill_queries(case, args.prefill_tokens, seed=7001)
    q_lens = [int((q_seq == s_).sum()) for s_ in range(S)]
    cu = torch.tensor([0] + list(torch.cumsum(torch.tensor(q_lens), 0).tolist()),
                      dtype=torch.int32)
    max_q = max(q_lens)
    T = query.shape[0]
    qd = query.to(dev).contiguous()
    cud = cu.to(dev)
    out = torch.empty(T, Hq, D, dtype=case.q_dtype, device=dev)
    flops = 4.0 * D * Hq * float((q_pos.to(torch.int64) + 1).sum())
    elem = 1 if int8 or fp8 else torch.finfo(case.q_dtype).bits // 8
    kv_bytes = sum(-(-int(n) // bs) for n in case.context_lens.tolist()) * bs * Hkv * 2 * \
        (D * elem + (4 if int8 else 0))

    def run(i, q_, bt_, cu_, cl_):
        k_, v_, ks_, vs_ = reps[i % len(reps)]
        if int8:
            pa.prefill_int8(out, q_, k_, v_, ks_, vs_, bt_, cu_, cl_, Hkv, max_q, case.scale,
                            stream=stream)
        elif fp8:
            pa.prefill_fp8(out, q_, k_, v_, bt_, cu_, cl_, Hkv, max_q, case.scale, case.k_scale,
                           case.v_scale, stream=stream)
        else:
            pa.prefill(out, q_, k_, v_, bt_, cu_, cl_, Hkv, max_q, case.scale, stream=stream)

    def launch(i):
        run(i, qd, bt, cud, cl)

    for i in range(args.warmup):
        launch(i)
    torch.cuda.synchronize()
    if pa.get_device_error():
        raise RuntimeError("device error word set after warm-up")
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    vis = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    phys = int(vis[local_rank]) if local_rank < len(vis) and vis[local_rank].strip().isdigit() \
        else local_rank
    clocks = ClockSampler(phys)
    clocks.start()
    time.sleep(0.3)
    barrier(dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(K):
        evs[i][0].record(stream)
        launch(i)
        evs[i][1].record(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    barrier(dev)
    clk = clocks.stop(t0, t1)
    if pa.get_device_error():
        raise RuntimeError("device error word set in the timed region")
    elapsed = all_reduce(e0.elapsed_time(e1) / 1e3, "max", dev)
    per = statistics.mean(a.elapsed_time(b) for a, b in evs) / 1e3
    flops_all = all_reduce(flops * K, "sum", dev)
    peak_tf, peak_kind = 1907.2, "fallback"
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak_tf, peak_kind = float(json.load(f)["bf16_tflops"]), "measured (burst)"
    except (OSError, KeyError, ValueError):
        pass
    achieved = flops / per / 1e12

    # e2e: query chunk, offsets, lengths and tables from pinned host memory,
    # output back to pinned host memory, every step
    host = {n: t.cpu().pin_memory() for n, t in (("q", query), ("cu", cu), ("cl", cl), ("bt", bt))}
    dbuf = {n: torch.empty_like(t, device=dev) for n, t in host.items()}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def e2e_step(i):
        for n, t in host.items():
            dbuf[n].copy_(t, non_blocking=True)
        run(i, dbuf["q"], dbuf["bt"], dbuf["cu"], dbuf["cl"])
        out_h.copy_(out, non_blocking=True)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a_.record(stream)
    for i in range(K):
        e2e_step(i)
    b_.record(stream)
    torch.cuda.synchronize()
    e2e_t = all_reduce(a_.elapsed_time(b_) / 1e3, "max", dev)
    result = {
        "metric": "paged prefill attention: achieved TFLOP/s", "value":
        round(flops_all / elapsed / 1e12, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(elapsed / K * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "impl": "ours",
        "config": {"workload": args.workload, "path": "prefill",
                   "cache_dtype": case.kv_dtype if int8 or fp8
                   else str(case.q_dtype).replace("torch.", ""),
                   "num_seqs": S,
                   "num_heads": Hq, "num_kv_heads": Hkv, "head_dim": D, "block_size": bs,
                   "query_tokens": T, "max_q_len": max_q, "flops_per_step": flops,
                   "kv_bytes_per_step": kv_bytes,
                   "l2": f"{args.replicas} rotating cache replicas (> L2)"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak_tf,
                     "peak_kind": peak_kind, "unit": "TFLOP/s",
                     "frac": round(achieved / peak_tf, 4),
                     "traffic": measured_traffic(f"{args.workload}/prefill" +
                                                 ("_int8" if int8 else "_fp8" if fp8 else "")),
                     "kernel": "prefill_tc_kernel (tcgen05 kind::f16, TMEM accumulators" +
                               (", INT8 codes widened to f16 in shared memory)" if int8 else
                                ", E4M3 codes widened to f16 in shared memory)" if fp8 else ")"),
                     "kernel_us_mean": round(per * 1e6, 2)},
        "e2e": {"value": round(flops_all / e2e_t / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host.values()),
                "d2h_bytes_per_step": out_h.numel() * out_h.element_size()},
        "gpu_launches": K, "clocks": clk, "wall_s_timed": round(t1 - t0, 4),
    }
    if rank == 0 and args.skip_cpu_baseline:
        print(json.dumps(result), flush=True)
    elif rank == 0:
        import oracle  # test infrastructure: only this CPU-baseline leg uses it
        ko, vo = kc.cpu(), vc.cpu()
        kso = None if ks is None else ks.cpu()
        vso = None if vs is None else vs.cpu()
        pick = torch.nonzero(q_seq == 0).flatten()[:64]
        tq = time.perf_counter()
        reps_o = 0
        while time.perf_counter() - tq < 10.0 and reps_o < 50:
            oracle.prefill(query[pick], q_seq[pick], q_pos[pick], ko, vo, case.block_tables, Hkv,
                           bs, case.scale, case.kv_dtype, case.k_scale, case.v_scale,
                           k_scales=kso, v_scales=vso)
            reps_o += 1
        t_o = (time.perf_counter() - tq) / reps_o
        f_o = 4.0 * D * Hq * float((q_pos[pick].to(torch.int64) + 1).sum())
        result["cpu_baseline"] = {"value": round(f_o / t_o / 1e12, 6), "unit": "TFLOP/s",
                                  "cores": cores(), "kind": "oracle",
                                  "sample": f"{pick.numel()} query tokens of sequence 0 "
                                            f"(all heads) x {reps_o} reps"}
        print(json.dumps(result), flush=True)


# ------------------------------------------------------------------ reference arm
def run_reference(args, rank, world):
    if rank != 0:
        return
    from paged_kv_cache_context_gb300 import workloads as wl
    case = wl.config(args.workload)
    rows_total = case.num_seqs * case.num_heads
    # calibrate the cost of a row, then size each step's sample to fit the budget
    t_cal, _, n_cal = oracle_step_time(case, min(rows_total, 64), 1)
    per_row = t_cal[0] / n_cal
    budget = 120.0
    rows = max(1, min(rows_total, int(budget / max(1, args.steps + args.warmup) / per_row)))
    times, sbytes, nrows = oracle_step_time(case, rows, args.steps + args.warmup)
    times = times[args.warmup:]
    el = sum(times)
    value = sbytes * len(times) / el / 1e9
    sb = step_bytes(case)
    out = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / len(times) * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": args.workload, "num_seqs": case.num_seqs,
                   "num_heads": case.num_heads, "num_kv_heads": case.num_kv_heads,
                   "head_dim": case.head_dim, "block_size": case.block_size,
                   "bytes_per_step_full_batch": sb["total"]},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores(),
                         "kind": "oracle",
                         "sample": f"{nrows} of {rows_total} sequence-head rows per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="mistral_bf16",
                    choices=("tiny", "mistral_bf16", "ring_bf16", "fp8_phi3", "prefix_bf16"))
    ap.add_argument("--replicas", type=int, default=4)
    ap.add_argument("--skip-cpu-baseline", action="store_true",
                    help="leave out the oracle timing (for profiler runs of the same line)")
    ap.add_argument("--prefill-tokens", type=int, default=512,
                    help="--path prefill: query tokens per sequence (its last positions)")
    ap.add_argument("--cascade-kv", choices=("auto", "fp8_e4m3", "int8"), default="auto",
                    help="with --path cascade: the cache held as FP8 E4M3 codes with per-tensor "
                         "scales (pa_decode_cascade_fp8) or INT8 codes with row scales "
                         "(pa_decode_cascade_int8)")
    ap.add_argument("--prefill-fp8", action="store_true",
                    help="--path prefill over an FP8 E4M3 cache with per-tensor scales "
                         "(pa_prefill_fp8)")
    ap.add_argument("--prefill-int8", action="store_true",
                    help="with --path prefill: the cache held as INT8 codes with row scales "
                         "(pa_prefill_int8)")
    ap.add_argument("--path", choices=("balanced", "cascade", "int8", "prefill"),
                    default="balanced",
                    help="entry point timed: pa_decode's balanced path, "
                         "pa_decode_cascade (workloads with a shared prefix), "
                         "pa_decode_int8 over the workload held as an INT8 cache, or "
                         "pa_prefill over the workload's last --prefill-tokens positions")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, local_rank, world = rank_info()
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        elif args.path == "prefill":
            run_prefill(args, rank, local_rank, world)
        else:
            run_ours(args, rank, local_rank, world)
    finally:
        import torch.distributed as dist
        if dist.is_available() and dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
