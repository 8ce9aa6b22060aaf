#!/usr/bin/env python
"""Benchmark of one decode step (KV append + plan + decode + combine) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama3_8b] [--no-cpu-baseline]

Prints ONE JSON line (rank 0).  A step is one pass of the whole hot path over
one batch: the append of the step's new K/V row per sequence (at position
L_b - 1), the plan, the decode and the combine -- one paged_decode_step call
through the C ABI (three kernel launches on one CUDA stream).

value      = algorithmic bytes of the step / device time of the step, GB/s:
             unique K+V bytes read + q read + out written + append bytes
             (k_new/v_new read and written into the pool).
e2e        = the same metric through paged_decode_step_host: the step's
             inputs (q, k_new, v_new, page table, lengths, positions) in
             pinned host memory, read by the kernels across the host-device
             link each step, and the output stored into pinned host memory,
             all inside the timed region (with a host sync per step);
             e2e.copy_engine: the same with copy-engine copies in and out
             around paged_decode_step.
roofline   = the decode kernel alone: its algorithmic bytes (K+V+q+out) over
             its duration (CUDA events around paged_decode_run on its stream,
             in a second region of the same steps issued as separate calls),
             against the measured HBM copy peak.
cpu_baseline = the float64 oracle on the host cores, on a bounded sample.

--impl reference times the oracle itself as the reference arm (same metric,
workload and unit, each step a bounded sample).

Multi-GPU: the path does not exchange data between GPUs; N>1 runs N
independent replicas (one per rank) and reports the aggregate.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged GQA decode attn: achieved HBM GB/s (% of peak) and decode seqs/s"
UNIT = "GB/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
DECODE_SOURCES = ["paged_kv_decode_16_gb300/csrc/decode.cuh",
                  "paged_kv_decode_16_gb300/csrc/decode_mma.cuh",
                  "paged_kv_decode_16_gb300/csrc/schedule.cuh",
                  "paged_kv_decode_16_gb300/csrc/merge.cuh",
                  "paged_kv_decode_16_gb300/csrc/common.cuh"]
TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "decode_llama3_8b_shape.md")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama3_8b")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--num-workers", type=int, default=0)
    ap.add_argument("--variant", choices=["auto", "cuda_cores", "tensor_cores", "tcgen05"],
                    default="auto",
                    help="decode kernel (auto = tensor cores)")
    ap.add_argument("--report", action="store_true",
                    help="per-configuration results instead of the bench line: for each named "
                         "workload the step's GPU time (L2 flushed by a read of twice its size, "
                         "median of 50 after 10 warm-up; and back to back), GB/s, %% of the same-run copy peak, "
                         "seqs/s, max abs / rel error of every output against the oracle, and "
                         "the oracle's time on all host cores and on one (median of 3 after 1)")
    ap.add_argument("--profile-only", action="store_true",
                    help="only the warm-up and timed steps (for profiler captures): no copy "
                         "peak, clock sampling, end-to-end leg or CPU baseline")
    ap.add_argument("--profile-path", choices=["step", "prefix", "multi"], default="step",
                    help="with --profile-only: 'prefix' runs, on the prefix_sharing workload, "
                         "warmup + steps calls of paged_decode_attention_prefix and then one "
                         "paged_decode_attention (4 launches per call, then 3); 'multi' runs "
                         "warmup + steps calls of paged_decode_attention_multi with 8 query "
                         "tokens per sequence on the step's cache (3 launches per call)")
    return ap.parse_args()


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(dist, x: float, device) -> float:
    """The largest of the ranks' values: a replicated job takes as long as its
    slowest rank.  dist is None on one process."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(world: int, bytes_per_step: float, ms_per_step: float) -> float:
    """Whole-job throughput: every rank moves bytes_per_step per step."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def decode_source_hash() -> str:
    """Hash of the decode kernel's sources with comments and blank space
    removed: an edit of a comment keeps a profile taken on the same code."""
    h = hashlib.sha256()
    for rel in DECODE_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def traffic_from_profile():
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current decode kernel source (else None)."""
    try:
        text = open(TRAFFIC_SUMMARY).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith(("traffic_bytes_per_launch", "kernel_source_sha")):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha") != decode_source_hash():
        return None
    try:
        return int(float(vals["traffic_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms in the background."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.t_start = self.t_end = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        self.wall = []

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def finish(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = []
        for rec in csv.reader(io.StringIO(out)):
            if len(rec) < 10:
                continue
            rec = [x.strip() for x in rec]
            try:
                ts = time.mktime(time.strptime(rec[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
            except Exception:
                ts = None
            rows.append((ts, rec))
        # samples inside the timed region (1 s slack for the timestamp granularity)
        inside = [r for ts, r in rows
                  if ts is not None and self.t_start is not None
                  and self.t_start - 1.0 <= ts <= self.t_end + 1.0]
        use = inside or [r for _, r in rows]
        sm = []
        smax = None
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in use:
            try:
                sm.append(float(r[2]))
                smax = float(r[3])
            except ValueError:
                pass
            for name, val in zip(names, r[6:10]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(use),
                "samples_in_region": len(inside)}


# ---------------------------------------------------------------------------
def step_bytes(w) -> dict:
    kv = w.kv_bytes_unique()
    qo = w.qo_bytes()
    app = w.append_bytes()
    return {"kv_unique": kv, "kv_logical": w.kv_bytes_logical(), "qo": qo, "append": app,
            "step": kv + qo + app, "decode": kv + qo}


def copy_peak_gbs(torch, dev) -> float:
    """Same-run device copy bandwidth (read + write bytes), 1 GiB bf16, best of 10."""
    n = 1 << 29
    a = torch.empty(n, dtype=torch.bfloat16, device=dev)
    b = torch.empty_like(a)
    a.fill_(1.0)
    best = float("inf")
    for _ in range(12):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        b.copy_(a)
        e.record()
        e.synchronize()
        best = min(best, s.elapsed_time(e))
    del a, b
    return 2 * n * 2 / (best * 1e-3) / 1e9


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def _oracle_rate(w, q, kp, vp, target_s: float):
    """Sequences one by one (all query heads), in a fixed random order, for
    about target_s seconds: (bytes, sequences, seconds)."""
    import numpy as np

    import oracle

    per_tok = w.n_kv_heads * w.head_dim * 4
    seqs = 0
    nbytes = 0
    t0 = time.perf_counter()
    order = np.random.default_rng(0).permutation(w.batch)
    i = 0
    while time.perf_counter() - t0 < target_s and seqs < 100 * w.batch:
        b = int(order[i % w.batch])
        i += 1
        rows = np.array([(b, h) for h in range(w.n_q_heads)], dtype=np.int32)
        oracle.paged_decode_rows(q, kp, vp, w.page_table, w.context_lens, w.scale, w.dtype_name,
                                 rows)
        seqs += 1
        nbytes += int(w.context_lens[b]) * per_tok + 2 * w.n_q_heads * w.head_dim * 2
    return nbytes, seqs, time.perf_counter() - t0


def oracle_full_median(w, q, kp, vp, reps: int = 3) -> float:
    """Seconds of one float64 oracle pass over the whole batch: the median of
    `reps` passes after one warm-up pass (input generation and copies excluded)."""
    import oracle

    times = []
    for i in range(reps + 1):
        t0 = time.perf_counter()
        oracle.paged_decode(q, kp, vp, w.page_table, w.context_lens, w.scale, w.dtype_name)
        if i:
            times.append(time.perf_counter() - t0)
    return statistics.median(times)


def cpu_oracle_sample(w, one_core: bool = True):
    """Time the oracle on host copies of the whole workload, on all host cores
    (the reported value) and then on one core: median of 3 passes after one
    warm-up pass each."""
    import oracle
    from paged_kv_decode_16_gb300 import workloads as wl

    q = wl.to_bits(w.q)
    kp, vp = wl.to_bits(w.k_pool), wl.to_bits(w.v_pool)
    by = step_bytes(w)["decode"]
    cores = oracle.max_threads()
    dt = oracle_full_median(w, q, kp, vp)
    res = {"value": by / dt / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
           "cpu_model": cpu_model(), "seconds_per_pass": dt, "seqs_per_s": w.batch / dt,
           "sample": f"the whole {w.name} batch ({w.batch} sequences x {w.n_q_heads} query "
                     f"heads), float64 oracle with OpenMP over query rows; median of 3 passes "
                     f"after 1 warm-up pass"}
    if one_core:
        oracle.set_threads(1)
        try:
            dt1 = oracle_full_median(w, q, kp, vp)
        finally:
            oracle.set_threads(cores)
        res["one_core"] = {"value": by / dt1 / 1e9, "unit": UNIT, "seqs_per_s": w.batch / dt1,
                           "seconds_per_pass": dt1,
                           "sample": "the same passes on 1 thread (median of 3 after 1)"}
    return res


def host_sample(fn, *args) -> dict:
    """A host-only side measurement: its failure is reported under its own key
    instead of costing the whole line."""
    try:
        return fn(*args)
    except Exception as e:  # noqa: BLE001 (reported in the line)
        return {"error": f"{type(e).__name__}: {e}"}


def prefix_cache_sample(seed: int) -> dict:
    """The host prefix cache on a serving-like request stream: 512 requests,
    each one of 16 system prompts of 1024 tokens plus a private 512-token
    suffix (page size 16); per request the longest cached prefix is matched,
    the missing pages allocated, the prompt inserted, and the request's own
    references released.  The pool is bookkeeping only (its addresses are never
    touched)."""
    import ctypes

    import numpy as np

    import paged_kv_decode_16_gb300 as pkv

    lib = pkv.load_library()
    h = ctypes.c_void_p()
    if lib.kv_pool_create(65536, 16, 8, 128, 1, ctypes.c_void_p(1 << 20),
                          ctypes.c_void_p(1 << 40), ctypes.byref(h)) != 0:
        return {"error": "kv_pool_create"}
    rng = np.random.default_rng(seed)
    systems = [rng.integers(0, 128000, size=1024).astype(np.int32) for _ in range(16)]
    reqs = [np.concatenate([systems[int(rng.integers(16))],
                            rng.integers(0, 128000, size=512).astype(np.int32)])
            for _ in range(512)]
    cache = pkv.PrefixCache(h)
    t_match = t_insert = 0.0
    matched = total = 0
    for toks in reqs:
        t0 = time.perf_counter()
        got = cache.match(toks)
        t1 = time.perf_counter()
        need = len(toks) // 16 - len(got)
        fresh = (ctypes.c_int32 * need)()
        lib.kv_pool_alloc_pages(h, need, fresh)
        row = np.array(got + list(fresh), dtype=np.int32)
        t2 = time.perf_counter()
        cache.insert(toks, row)
        t3 = time.perf_counter()
        lib.kv_pool_release_pages(h, row.ctypes.data, len(row))
        t_match += t1 - t0
        t_insert += t3 - t2
        matched += len(got)
        total += len(toks) // 16
    pages = cache.pages()
    cache.destroy()
    lib.kv_pool_destroy(h)
    n = len(reqs)
    return {"what": "host radix prefix cache (pkv_prefix_cache_*): match + insert per request, "
                    "through the Python binding",
            "requests": n, "tokens_per_request": 1536, "us_per_match": t_match / n * 1e6,
            "us_per_insert": t_insert / n * 1e6, "matched_page_fraction": matched / total,
            "cached_pages": pages}


# ---------------------------------------------------------------------------
def reference_step(w, q, kp, vp, target_s: float) -> dict:
    """One reference-arm step: the oracle over sequences of the workload (all
    query heads each, fixed random order) for about target_s seconds."""
    nbytes, seqs, dt = _oracle_rate(w, q, kp, vp, target_s)
    return {"value": nbytes / dt / 1e9, "seqs_per_s": seqs / dt,
            "sample": f"{seqs} sequences x all {w.n_q_heads} query heads of the {w.name} "
                      f"workload, float64 oracle with OpenMP over query heads, {dt:.2f} s"}


def run_reference(args):
    """Reference arm: the float64 oracle on the host cores, same metric/unit."""
    ws, rank, _ = dist_info()
    if rank != 0:
        return 0
    import torch  # noqa: F401  (workload tensors live on the CPU here)

    import oracle
    from paged_kv_decode_16_gb300 import workloads as wl
    w = wl.make(args.workload, seed=args.seed, device="cpu")
    kp, vp = wl.to_bits(w.k_pool), wl.to_bits(w.v_pool)
    if w.append:
        kp, vp = oracle.kv_append(kp, vp, wl.to_bits(w.k_new), wl.to_bits(w.v_new),
                                  w.page_table, w.positions)
    q = wl.to_bits(w.q)
    # about 150 s in all: each step samples at least one sequence (a few ms)
    budget = min(12.0, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        reference_step(w, q, kp, vp, budget)
    vals, seqs = [], []
    r = None
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r = reference_step(w, q, kp, vp, budget)
        vals.append(r["value"])
        seqs.append(r["seqs_per_s"])
    wall = time.perf_counter() - t0
    value = statistics.mean(vals) if vals else 0.0
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": wall / max(1, args.steps) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "batch": w.batch, "n_q_heads": w.n_q_heads,
                   "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "page_size": w.page_size,
                   "storage_dtype": w.dtype_name, "seed": args.seed},
        "seqs_per_s": statistics.mean(seqs) if seqs else 0.0,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(),
                         "cpu_model": cpu_model(), "kind": "oracle",
                         "sample": r["sample"] if r else ""},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_ours(args):
    import numpy as np
    import torch

    import paged_kv_decode_16_gb300 as pkv
    from paged_kv_decode_16_gb300 import workloads as wl

    world, rank, local = dist_info()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pkv.load_library()

    w = wl.make(args.workload, seed=args.seed, device=dev)
    B = w.batch
    table = torch.from_numpy(w.page_table).to(dev)
    lens = torch.from_numpy(w.context_lens).to(dev)
    pos = torch.from_numpy(w.positions).to(dev)
    pool = pkv.kv_pool_create(w.num_pages, w.page_size, w.n_kv_heads, w.head_dim, w.dtype,
                              w.k_pool, w.v_pool)
    out = torch.empty_like(w.q)
    nw = args.num_workers
    # tcgen05 runs several query tokens per sequence only: the profile of the
    # multi-query call; the step itself keeps the automatic kernel
    multi_var = None
    if args.variant == "tcgen05":
        if not (args.profile_only and args.profile_path == "multi"):
            raise SystemExit("--variant tcgen05 needs --profile-only --profile-path multi")
        multi_var = pkv.VARIANT_TCGEN05
    var = {"auto": pkv.VARIANT_AUTO, "cuda_cores": pkv.VARIANT_CUDA_CORES,
           "tensor_cores": pkv.VARIANT_TENSOR_CORES,
           "tcgen05": pkv.VARIANT_AUTO}[args.variant]
    ws = pkv.alloc_workspace(B, w.n_q_heads, w.n_kv_heads, w.head_dim, nw, device=dev,
                             variant=var)
    stream = torch.cuda.current_stream(dev)
    by = step_bytes(w)

    def step():
        # one C-ABI call: append fused into the plan launch, decode, combine
        pkv.paged_decode_step(w.k_new, w.v_new, pos, w.q, w.k_pool, w.v_pool, table, lens,
                              w.scale, out, ws, nw, variant=var)

    def split_step(ev0, ev1):
        # the same work as separate calls, with events around the decode kernel
        pkv.kv_append(pool, w.k_new, w.v_new, table, pos)
        pkv.paged_decode_plan(lens, w.n_q_heads, w.n_kv_heads, w.head_dim, w.page_size,
                              table.shape[1], ws, nw, variant=var)
        ev0.record(stream)
        pkv.paged_decode_run(w.q, w.k_pool, w.v_pool, table, w.scale, out, ws, nw, variant=var)
        ev1.record(stream)
        pkv.paged_decode_combine(out, w.n_kv_heads, ws, nw, variant=var)

    peak, peak_kind = measured_peak()
    if args.profile_only and args.profile_path == "multi":
        gq = torch.Generator(device=dev).manual_seed(args.seed + 8)
        qm = torch.randn(B, 8, w.n_q_heads, w.head_dim, generator=gq, device=dev,
                         dtype=torch.float32).to(w.dtype)
        om = torch.empty_like(qm)
        mv = multi_var if multi_var is not None else var
        wsm = pkv.alloc_multi_workspace(B, 8, w.n_q_heads, w.n_kv_heads, w.head_dim, nw,
                                        device=dev, variant=mv)
        for _ in range(args.warmup + args.steps):
            pkv.paged_decode_attention_multi(qm, w.k_pool, w.v_pool, table, lens, w.scale, om,
                                             wsm, nw, variant=mv)
        torch.cuda.synchronize()
        status = pkv.pkv_read_device_status(wsm)
        if rank == 0:
            print(json.dumps({"profile_only": True, "workload": args.workload, "path": "multi",
                              "steps": args.steps, "warmup": args.warmup,
                              "device_status": status}))
        pool.destroy()
        if dist:
            dist.destroy_process_group()
        return 0 if status == 0 else 1
    if args.profile_only and args.profile_path == "prefix":
        wp = wl.make("prefix_sharing", seed=args.seed, device=dev)
        tp = torch.from_numpy(wp.page_table).to(dev)
        lp = torch.from_numpy(wp.context_lens).to(dev)
        op = torch.empty_like(wp.q)
        wsc = pkv.alloc_prefix_workspace(wp.batch, wp.n_q_heads, wp.n_kv_heads, wp.head_dim, nw,
                                         device=dev, variant=var)
        wsp = pkv.alloc_workspace(wp.batch, wp.n_q_heads, wp.n_kv_heads, wp.head_dim, nw,
                                  device=dev, variant=var)
        for _ in range(args.warmup + args.steps):
            pkv.paged_decode_attention_prefix(wp.q, wp.k_pool, wp.v_pool, tp, lp, wp.scale,
                                              wp.prefix_len, op, wsc, nw, variant=var)
        pkv.paged_decode_attention(wp.q, wp.k_pool, wp.v_pool, tp, lp, wp.scale, op, wsp, nw,
                                   variant=var)
        torch.cuda.synchronize()
        status = pkv.pkv_read_device_status(wsc) | pkv.pkv_read_device_status(wsp)
        if rank == 0:
            print(json.dumps({"profile_only": True, "workload": "prefix_sharing",
                              "path": "prefix", "steps": args.steps, "warmup": args.warmup,
                              "device_status": status}))
        pool.destroy()
        if dist:
            dist.destroy_process_group()
        return 0 if status == 0 else 1
    if args.profile_only:
        for _ in range(args.warmup + args.steps):
            step()
        torch.cuda.synchronize()
        status = pkv.pkv_read_device_status(ws)
        if rank == 0:
            print(json.dumps({"profile_only": True, "workload": args.workload,
                              "steps": args.steps, "warmup": args.warmup,
                              "device_status": status}))
        pool.destroy()
        if dist:
            dist.destroy_process_group()
        return 0 if status == 0 else 1
    same_run_copy = copy_peak_gbs(torch, dev)
    sampler = ClockSampler(local)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if pkv.pkv_read_device_status(ws):
        raise RuntimeError("device status set during warm-up")

    # An untimed read of twice the L2 size (a read, not a write: dirty lines
    # would be written back inside the next timed region) before each run of
    # flushed_ms and before each flushed decode launch: second figures of the
    # step and of the decode kernel, where no run finds anything of its own in L2.
    flush = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def flushed_ms(fn, n):
        """Mean of n runs of fn, each timed by its own events after a flush."""
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for a, b in evs:
            flush.amax()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs) / n

    def timed_loop(fn, n):
        """Mean of n runs of fn back to back (after warm-up)."""
        for _ in range(max(3, args.warmup)):
            fn()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(dist, e0.elapsed_time(e1) / n, dev)

    K = args.steps
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.mark_start()
    t_start.record(stream)
    for _ in range(K):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    sampler.mark_end()
    if dist:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    ms_step = total_ms / K
    ms_step = max_over_ranks(dist, ms_step, dev)
    # the same step with L2 flushed before each
    KF = max(1, min(K, 2000))
    ms_flushed = max_over_ranks(dist, flushed_ms(step, KF), dev)
    clocks = sampler.finish()

    # ---- the same step with the rotary embedding of q and k_new fused into
    # the append (paged_decode_step_rope), same timing discipline ----
    KR = max(1, min(K, 2000))
    rope_theta = 500000.0

    def rope_step():
        pkv.paged_decode_step_rope(w.k_new, w.v_new, pos, w.q, w.k_pool, w.v_pool, table, lens,
                                   w.scale, rope_theta, out, ws, nw, variant=var)

    rope_ms = timed_loop(rope_step, KR)
    # the same with the per-head RMS norm of q and k before the rotation
    gn = torch.Generator(device=dev).manual_seed(args.seed + 2)
    wq = (1.0 + 0.3 * torch.randn(w.head_dim, generator=gn, device=dev)).to(w.dtype)
    wk = (1.0 + 0.3 * torch.randn(w.head_dim, generator=gn, device=dev)).to(w.dtype)

    def rope_norm_step():
        pkv.paged_decode_step_rope(w.k_new, w.v_new, pos, w.q, w.k_pool, w.v_pool, table, lens,
                                   w.scale, rope_theta, out, ws, nw, variant=var,
                                   q_norm_weight=wq, k_norm_weight=wk, norm_eps=1e-6)

    rope_norm_ms = timed_loop(rope_norm_step, KR)

    # ---- shared-prefix decode on the prefix-sharing workload (64 sequences,
    # one 2048-token prefix): the cascade against the plain decode ----
    wp = wl.make("prefix_sharing", seed=args.seed, device=dev)
    tp = torch.from_numpy(wp.page_table).to(dev)
    lp = torch.from_numpy(wp.context_lens).to(dev)
    op = torch.empty_like(wp.q)
    wsp_plain = pkv.alloc_workspace(wp.batch, wp.n_q_heads, wp.n_kv_heads, wp.head_dim, nw,
                                    device=dev, variant=var)
    wsp = pkv.alloc_prefix_workspace(wp.batch, wp.n_q_heads, wp.n_kv_heads, wp.head_dim, nw,
                                     device=dev, variant=var)

    KP = max(1, min(K, 2000))
    prefix_ms = timed_loop(lambda: pkv.paged_decode_attention_prefix(
        wp.q, wp.k_pool, wp.v_pool, tp, lp, wp.scale, wp.prefix_len, op, wsp, nw,
        variant=var), KP)
    plain_ms = timed_loop(lambda: pkv.paged_decode_attention(
        wp.q, wp.k_pool, wp.v_pool, tp, lp, wp.scale, op, wsp_plain, nw, variant=var), KP)
    # its unique K/V (84 MB) fits in L2: the same two calls with L2 flushed before each
    prefix_ms_flushed = max_over_ranks(dist, flushed_ms(lambda: pkv.paged_decode_attention_prefix(
        wp.q, wp.k_pool, wp.v_pool, tp, lp, wp.scale, wp.prefix_len, op, wsp, nw,
        variant=var), KP), dev)
    plain_ms_flushed = max_over_ranks(dist, flushed_ms(lambda: pkv.paged_decode_attention(
        wp.q, wp.k_pool, wp.v_pool, tp, lp, wp.scale, op, wsp_plain, nw, variant=var), KP), dev)
    pby = step_bytes(wp)
    del wp, tp, lp, op, wsp, wsp_plain

    # ---- several query tokens per sequence (four draft tokens, causal) on the
    # step's own cache, against the one-query decode of the same batch ----
    QN = 4
    multi = None
    if var != pkv.VARIANT_CUDA_CORES:
        def multi_ms_for(qn, mvar=var):
            gq = torch.Generator(device=dev).manual_seed(args.seed + qn)
            qm = torch.randn(B, qn, w.n_q_heads, w.head_dim, generator=gq, device=dev,
                             dtype=torch.float32).to(w.dtype)
            om = torch.empty_like(qm)
            wsm = pkv.alloc_multi_workspace(B, qn, w.n_q_heads, w.n_kv_heads, w.head_dim, nw,
                                            device=dev, variant=mvar)
            return timed_loop(lambda: pkv.paged_decode_attention_multi(
                qm, w.k_pool, w.v_pool, table, lens, w.scale, om, wsm, nw, variant=mvar), KP)

        multi_ms = multi_ms_for(QN)
        multi8_ms = multi_ms_for(8)
        # the tcgen05 kernel (transposed products, units of up to 64 rows)
        tc5 = {qn: multi_ms_for(qn, pkv.VARIANT_TCGEN05) for qn in (4, 8, 16)}
        multi16_ms = multi_ms_for(16)
        one_ms = timed_loop(lambda: pkv.paged_decode_attention(
            w.q, w.k_pool, w.v_pool, table, lens, w.scale, out, ws, nw, variant=var), KP)
        mbytes = by["kv_unique"] + QN * by["qo"]
        multi = {"what": f"paged_decode_attention_multi with {QN} causal query tokens per "
                         "sequence (each K/V chunk read once for all of them) vs "
                         "paged_decode_attention with one, same cache; 8 tokens: units of "
                         "32 rows, two m16 tiles per warp",
                 "n_queries": QN, "ms_multi": multi_ms, "ms_one_query": one_ms, "steps": KP,
                 "gbs_multi": mbytes / (multi_ms * 1e-3) / 1e9,
                 "tokens_per_s_multi": B * QN / (multi_ms * 1e-3),
                 "tokens_per_s_one_query": B / (one_ms * 1e-3),
                 "ms_multi_8": multi8_ms,
                 "tokens_per_s_multi_8": B * 8 / (multi8_ms * 1e-3),
                 "ms_multi_16": multi16_ms,
                 "tcgen05": {"what": "the same calls with variant PKV_VARIANT_TCGEN05",
                             "ms_multi_4": tc5[4], "ms_multi_8": tc5[8],
                             "ms_multi_16": tc5[16]}}

    # ---- the same step on the other full-size workloads: one sequence-long
    # context per (sequence, KV head) split over many warps, and the mixed
    # batch whose append writes position L and attends L + 1 tokens ----
    others = {}
    for oname in ("long_context", "mixed_append"):
        w2 = wl.make(oname, seed=args.seed, device=dev)
        t2 = torch.from_numpy(w2.page_table).to(dev)
        l2 = torch.from_numpy(w2.context_lens).to(dev)
        p2 = torch.from_numpy(w2.positions).to(dev)
        o2 = torch.empty_like(w2.q)
        ws2 = pkv.alloc_workspace(w2.batch, w2.n_q_heads, w2.n_kv_heads, w2.head_dim, nw,
                                  device=dev, variant=var)
        ms2 = timed_loop(lambda: pkv.paged_decode_step(
            w2.k_new, w2.v_new, p2, w2.q, w2.k_pool, w2.v_pool, t2, l2, w2.scale, o2, ws2, nw,
            variant=var), KP)
        b2 = step_bytes(w2)
        others[oname] = {
            "ms_per_step": ms2, "value": aggregate_gbs(world, b2["step"], ms2), "unit": UNIT,
            "pct_of_peak": 100.0 * b2["step"] / (ms2 * 1e-3) / 1e9 / peak, "steps": KP,
            "batch": w2.batch, "bytes_per_step": b2["step"],
            "device_status": pkv.pkv_read_device_status(ws2)}
        del w2, t2, l2, p2, o2, ws2

    # ---- the decode kernel alone: events around its launch on its stream,
    # in steps run back to back as in the timed region (the roofline), and
    # each after an L2 flush (reported beside it) ----
    KD = max(1, min(K, 2000))

    def decode_ms(flushed):
        dec0 = [torch.cuda.Event(enable_timing=True) for _ in range(KD)]
        dec1 = [torch.cuda.Event(enable_timing=True) for _ in range(KD)]
        torch.cuda.synchronize()
        for i in range(KD):
            if flushed:
                flush.amax()
            split_step(dec0[i], dec1[i])
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in zip(dec0, dec1))

    dec_avg = decode_ms(False)
    dec_avg_flushed = decode_ms(True)

    # ---- end to end through host buffers (pinned), one sync per step ----
    # paged_decode_step_host: the step's inputs sit in pinned host memory and
    # its kernels read them (and store the result into pinned host memory)
    # across the host-device link themselves.  Beside it, the same step with
    # copy-engine copies: the inputs as one packed pinned buffer copied in,
    # paged_decode_step, the output copied out.  Each is recorded once into a
    # CUDA graph; a step replays it and waits for the result.
    def graph_of(body):
        body()
        torch.cuda.synchronize()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                body()
        stream.wait_stream(cap)
        torch.cuda.synchronize()
        return g

    KE = max(1, min(args.e2e_steps, K))

    def e2e_time(g):
        def e2e_step():
            g.replay()
            torch.cuda.current_stream(dev).synchronize()
        for _ in range(10):
            e2e_step()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(KE):
            e2e_step()
        return max_over_ranks(dist, (time.perf_counter() - t0) * 1e3 / KE, dev)

    srcs = [w.q, w.k_new, w.v_new, table, lens, pos]
    pinned = [t.detach().cpu().contiguous().pin_memory() for t in srcs]
    q_h, kn_h, vn_h, tb_h, ln_h, ps_h = pinned
    out_h = torch.empty_like(out, device="cpu").pin_memory()
    ws_host = pkv.alloc_step_host_workspace(B, w.n_q_heads, w.n_kv_heads, w.head_dim,
                                            table.shape[1], nw, device=dev, variant=var)
    h2d = sum(t.numel() * t.element_size() for t in pinned)
    d2h = out.numel() * out.element_size()

    def e2e_host_body():
        pkv.paged_decode_step_host(kn_h, vn_h, ps_h, q_h, w.k_pool, w.v_pool, tb_h, ln_h, w.scale,
                                   out_h, ws_host, nw, variant=var)

    e2e_ms = e2e_time(graph_of(e2e_host_body))
    host_status = pkv.pkv_read_device_status(ws_host)

    offs, total = [], 0
    for t in srcs:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    in_h = torch.empty(total, dtype=torch.uint8).pin_memory()
    in_d = torch.empty(total, dtype=torch.uint8, device=dev)
    views_d = []
    for t, o in zip(srcs, offs):
        nb = t.numel() * t.element_size()
        in_h[o:o + nb].copy_(t.detach().cpu().reshape(-1).view(torch.uint8))
        views_d.append(in_d[o:o + nb].view(t.dtype).view(t.shape))
    q_d, kn_d, vn_d, tb_d, ln_d, ps_d = views_d
    out_h2 = torch.empty_like(out, device="cpu").pin_memory()

    def e2e_copy_body():
        in_d.copy_(in_h, non_blocking=True)
        pkv.paged_decode_step(kn_d, vn_d, ps_d, q_d, w.k_pool, w.v_pool, tb_d, ln_d, w.scale,
                              out, ws, nw, variant=var)
        out_h2.copy_(out, non_blocking=True)

    e2e_copy_ms = e2e_time(graph_of(e2e_copy_body))
    status = pkv.pkv_read_device_status(ws)

    value = aggregate_gbs(world, by["step"], ms_step)
    achieved = by["decode"] / (dec_avg * 1e-3) / 1e9
    traffic = traffic_from_profile()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype_name, "data": "synthetic",
        "config": {
            "workload": args.workload, "batch": B, "n_q_heads": w.n_q_heads,
            "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "page_size": w.page_size,
            "context_lens": f"uniform [512, 4096], mean {float(w.context_lens.mean()):.0f}"
            if args.workload == "llama3_8b" else f"mean {float(w.context_lens.mean()):.0f}",
            "seed": args.seed, "num_workers": nw or "auto", "variant": args.variant,
            "parallelism": "replicas" if world > 1 else "single GPU",
            "l2": (f"inputs larger than L2: {by['kv_unique'] / 2**20:.0f} MiB of K/V per step "
                   f"vs 129 MB L2; no flush") if by["kv_unique"] > L2_BYTES
            else "inputs smaller than L2 (warm numbers)",
            "step": "paged_decode_step: append fused into the plan launch, decode, combine "
                    "(3 launches chained by programmatic dependent launch)",
        },
        "seqs_per_s": world * B / (ms_step * 1e-3),
        "l2_flushed": {"ms_per_step": ms_flushed, "steps": KF,
                       "value": aggregate_gbs(world, by["step"], ms_flushed), "unit": UNIT,
                       "what": "the same step, each run after an untimed read of twice the "
                               "L2 size, timed by its own events"},
        "pct_of_peak": 100.0 * value / world / peak,
        "bytes_per_step": by,
        "decode_kernel_ms": dec_avg,
        "same_run_copy_gbs": same_run_copy,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "kernel": "pkv::decode_kernel (CUDA cores)"
                     if var == pkv.VARIANT_CUDA_CORES else "pkv::decode_mma_kernel (tensor cores)",
                     "algorithmic_bytes": by["decode"],
                     "timing": f"CUDA events around paged_decode_run on its stream, mean of "
                               f"{KD} steps run back to back right after the timed region",
                     "decode_kernel_ms_l2_flushed": dec_avg_flushed,
                     "frac_l2_flushed": by["decode"] / (dec_avg_flushed * 1e-3) / 1e9 / peak},
        "e2e": {"value": aggregate_gbs(world, by["step"], e2e_ms), "unit": UNIT,
                "mode": "CUDA graph replay per step of paged_decode_step_host (the step's "
                        "inputs in pinned host memory, read by the plan launch across the "
                        "host-device link; the output stored by the kernels into pinned host "
                        "memory), then a host sync",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "steps": KE, "device_status": host_status,
                "copy_engine": {"value": aggregate_gbs(world, by["step"], e2e_copy_ms),
                                "unit": UNIT, "ms_per_step": e2e_copy_ms,
                                "mode": "CUDA graph replay per step: the packed pinned inputs "
                                        "copied in, paged_decode_step, the output copied out, "
                                        "then a host sync"}},
        "rope_step": {"value": aggregate_gbs(world, by["step"], rope_ms), "unit": UNIT,
                      "ms_per_step": rope_ms, "steps": KR, "rope_theta": rope_theta,
                      "ms_per_step_with_qk_norm": rope_norm_ms,
                      "what": "paged_decode_step_rope: rotary embedding of q and k_new fused "
                              "into the append CTAs of the plan launch, same bytes"},
        "prefix_sharing": {
            "what": "paged_decode_attention_prefix (shared prefix attended once per KV head "
                    "for all queries, then the suffixes, then the merge) vs "
                    "paged_decode_attention on the prefix_sharing workload",
            "ms_prefix": prefix_ms, "ms_plain": plain_ms, "steps": KP,
            "ms_prefix_l2_flushed": prefix_ms_flushed, "ms_plain_l2_flushed": plain_ms_flushed,
            "gbs_unique_prefix": (pby["kv_unique"] + pby["qo"]) / (prefix_ms * 1e-3) / 1e9,
            "gbs_logical_prefix": (pby["kv_logical"] + pby["qo"]) / (prefix_ms * 1e-3) / 1e9,
            "gbs_logical_plain": (pby["kv_logical"] + pby["qo"]) / (plain_ms * 1e-3) / 1e9},
        "multi_query": multi,
        "other_workloads": others,
        "prefix_cache": host_sample(prefix_cache_sample, args.seed),
        "gpu_launches": 3 * K,
        "clocks": clocks,
        "device_status": status,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(w)
    elif rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = None
    if rank == 0:
        print(json.dumps(line))
    pool.destroy()
    if dist:
        dist.destroy_process_group()
    return 0


def _errors(got, ref):
    """max |gpu - ref| and max |gpu - ref| / max(|ref|, 0.2) over every element."""
    import numpy as np
    err = np.abs(got - ref)
    return float(err.max(initial=0.0)), float((err / np.maximum(np.abs(ref), 0.2)).max(initial=0.0))


def run_report(args):
    """Per-configuration results of the five named workloads (one GPU)."""
    import numpy as np
    import torch

    import oracle
    import paged_kv_decode_16_gb300 as pkv
    from paged_kv_decode_16_gb300 import workloads as wl

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pkv.load_library()
    stream = torch.cuda.current_stream(dev)
    copy_peak = copy_peak_gbs(torch, dev)
    # L2 flush: a read of twice the L2 size, so the lines it leaves are clean
    # (a write would leave dirty lines whose write-back lands in the timed step)
    flush = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def cold_ms(fn, n=50, warm=10):
        for _ in range(warm):
            fn()
        ts = []
        for _ in range(n):
            flush.amax()  # untimed read of twice the L2 size
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    def warm_ms(fn, n=500):
        for _ in range(20):
            fn()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / n

    rows = []
    for name in wl.NAMES:
        w = wl.make(name, seed=args.seed, device=dev)
        table = torch.from_numpy(w.page_table).to(dev)
        lens = torch.from_numpy(w.context_lens).to(dev)
        pos = torch.from_numpy(w.positions).to(dev)
        out = torch.empty_like(w.q)
        ws = pkv.alloc_workspace(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, device=dev)
        kb, vb = wl.to_bits(w.k_pool), wl.to_bits(w.v_pool)

        def step():
            pkv.paged_decode_step(w.k_new, w.v_new, pos, w.q, w.k_pool, w.v_pool, table, lens,
                                  w.scale, out, ws)

        step()
        torch.cuda.synchronize()
        status = pkv.pkv_read_device_status(ws)
        kp, vp = oracle.kv_append(kb, vb, wl.to_bits(w.k_new), wl.to_bits(w.v_new),
                                  w.page_table, w.positions)
        append_exact = bool(np.array_equal(kp, wl.to_bits(w.k_pool)) and
                            np.array_equal(vp, wl.to_bits(w.v_pool)))
        q_bits = wl.to_bits(w.q)
        ref = oracle.paged_decode(q_bits, kp, vp, w.page_table, w.context_lens, w.scale,
                                  w.dtype_name)
        got = out.float().cpu().numpy().astype(np.float64)
        max_abs, max_rel = _errors(got, ref)
        by = step_bytes(w)
        t_cold, t_warm = cold_ms(step), warm_ms(step)
        cores = oracle.max_threads()
        cpu_all = oracle_full_median(w, q_bits, kp, vp)
        oracle.set_threads(1)
        try:
            cpu_one = oracle_full_median(w, q_bits, kp, vp)
        finally:
            oracle.set_threads(cores)
        r = {"workload": name, "call": "paged_decode_step (append + plan + decode + combine)",
             "batch": w.batch, "bytes": by["step"], "ms_cold": t_cold, "ms_warm": t_warm,
             "gbs_cold": by["step"] / (t_cold * 1e-3) / 1e9,
             "gbs_warm": by["step"] / (t_warm * 1e-3) / 1e9,
             "pct_of_copy_peak_cold": 100.0 * by["step"] / (t_cold * 1e-3) / 1e9 / copy_peak,
             "seqs_per_s_cold": w.batch / (t_cold * 1e-3), "max_abs_err": max_abs,
             "max_rel_err": max_rel, "append_bit_exact": append_exact, "device_status": status,
             "cpu_oracle_s_all_cores": cpu_all, "cpu_oracle_s_one_core": cpu_one,
             "cpu_cores": cores}
        rows.append(r)
        print(json.dumps(r), flush=True)
        if name == "prefix_sharing":
            wsp = pkv.alloc_prefix_workspace(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim,
                                             device=dev)
            out2 = torch.empty_like(w.q)

            def cascade():
                pkv.paged_decode_attention_prefix(w.q, w.k_pool, w.v_pool, table, lens, w.scale,
                                                  w.prefix_len, out2, wsp)

            cascade()
            torch.cuda.synchronize()
            st2 = pkv.pkv_read_device_status(wsp)
            a2, r2 = _errors(out2.float().cpu().numpy().astype(np.float64), ref)
            c_cold, c_warm = cold_ms(cascade), warm_ms(cascade)
            uniq = by["kv_unique"] + by["qo"]
            r = {"workload": name, "call": "paged_decode_attention_prefix (cascade, no append)",
                 "batch": w.batch, "bytes": uniq, "ms_cold": c_cold, "ms_warm": c_warm,
                 "gbs_cold": uniq / (c_cold * 1e-3) / 1e9, "gbs_warm": uniq / (c_warm * 1e-3) / 1e9,
                 "pct_of_copy_peak_cold": 100.0 * uniq / (c_cold * 1e-3) / 1e9 / copy_peak,
                 "seqs_per_s_cold": w.batch / (c_cold * 1e-3), "max_abs_err": a2,
                 "max_rel_err": r2, "device_status": st2}
            rows.append(r)
            print(json.dumps(r), flush=True)
        del w, table, lens, pos, out, ws
        torch.cuda.empty_cache()
    print(json.dumps({"copy_peak_gbs": copy_peak, "cpu_model": cpu_model(),
                      "gpu": torch.cuda.get_device_name(dev)}))
    print("| config | call | GPU µs (L2 flushed / warm) | GB/s (flushed) | % of copy peak | "
          "seqs/s | max abs err | max rel err | oracle s (all cores / 1 core) |")
    print("|---|---|---|---|---|---|---|---|---|")
    for r in rows:
        cpu = (f"{r['cpu_oracle_s_all_cores']:.3f} / {r['cpu_oracle_s_one_core']:.2f}"
               if "cpu_oracle_s_all_cores" in r else "—")
        print(f"| {r['workload']} | {r['call'].split(' ')[0]} | {r['ms_cold'] * 1e3:.1f} / "
              f"{r['ms_warm'] * 1e3:.1f} | {r['gbs_cold']:.0f} | {r['pct_of_copy_peak_cold']:.1f} | "
              f"{r['seqs_per_s_cold']:.3g} | {r['max_abs_err']:.2e} | {r['max_rel_err']:.2e} | "
              f"{cpu} |")
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.report:
        return run_report(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
