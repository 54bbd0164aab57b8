"""Benchmark of the paged-attention hot path on GB300.

One step = one decode step of the whole path on one batch: pa_append_kv
writes each request's new K/V token into the page pool by slot_mapping, then
pa_attention (which routes L = 1 to the split-KV decode kernel) attends over
every request's paged context. Inputs are seeded synthetic batches shaped
like the pages' decode workloads (no datasets, no weights).

Prints one JSON line. ``value`` is decode K/V GB/s over the whole step
(algorithmic bytes / device time), with the inputs resident in HBM; four or
more rotating copies of the page pool keep every step's K/V reads cold in L2.

    python bench.py [--gpus N --steps K --warmup W] [--workload NAME]
    python bench.py --impl reference ...   (the fp64 CPU oracle, timed)

Under torchrun (N > 1) every rank runs its own replica of the workload (the
path has no exchange step; "scaling": "weak") and value sums all ranks' bytes
over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "paged decode K/V GB/s & tokens/s (% HBM peak); prefill TFLOP/s (% bf16 peak)"
DEFAULT_WORKLOAD = "decode_b32_gqa7_ps16"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def timed_region(dist, sync, run):
    """Runs `run()` between a barrier and a device synchronize on both sides
    (every rank enters and leaves together). Returns run()'s result."""
    if dist is not None:
        dist.barrier()
    sync()
    out = run()
    sync()
    if dist is not None:
        dist.barrier()
    return out


def max_over_ranks(dist, value, device=None):
    """The largest `value` over all ranks, returned on every rank (the value
    itself with one rank): the whole job is as slow as its slowest replica."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world, bytes_per_step, ms_per_step):
    """GB/s of the whole job: every replica moves `bytes_per_step` per step and
    a step takes the slowest rank's `ms_per_step`."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


def step_bytes(b: wl.PagedBatch):
    """Algorithmic bytes of one step: (decode kernel, append kernel)."""
    n = b.context_lens.astype(np.int64)
    kv = int(n.sum()) * b.H_kv * b.D * 2 * 2
    qo = 2 * b.B * b.H_q * b.L * b.D * 2
    tables = int(np.ceil(n / b.page_size).sum()) * 4 + b.B * 4
    decode = kv + qo + tables
    append = 2 * (2 * b.B * b.H_kv * b.L_new * b.D * 2) + b.B * b.L_new * 4
    return decode, append


def prefill_flops(b: wl.PagedBatch) -> float:
    """Causal-useful FLOPs: 4 * D per (query row, visible key) pair."""
    total = 0
    for n in b.context_lens.astype(np.int64):
        for i in range(b.L):
            p = int(n) - b.L + i
            vis = min(int(n), p + 1) if b.causal else int(n)
            total += max(0, vis)
    return 4.0 * b.D * b.H_q * total


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def source_digest(rel):
    """Digest of a source file's code: comments and white space removed, so a
    comment edit keeps a capture valid and any code change invalidates it."""
    import re
    with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    text = " ".join(text.split())
    return hashlib.sha256(text.encode()).hexdigest()[:16]


def committed_traffic(kernel_key, workload):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)[kernel_key]
    except Exception:
        return None
    if t.get("workload") != workload:
        return None
    if t.get("source_sha") != source_digest(t["source"]):
        return None
    return t.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.rows = []
        self.marks = []
        self.proc = None
        self.gpu = gpu_index
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def mark(self, name):
        self.marks.append((name, time.time()))

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        parsed = []
        for ts, line in self.rows:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                parsed.append((ts, float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        window = [p for p in parsed if t0 <= p[0] <= t1]
        scope = "timed"
        if not window:          # very short timed region: widen to the whole run
            window, scope = parsed, "run"
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in window for i, v in enumerate(p[3])
                          if v.lower().startswith("active")})
        return {"sm_mhz": float(np.median([p[1] for p in window])),
                "sm_max_mhz": float(max(p[2] for p in window)),
                "reasons": reasons, "samples": len(window), "window": scope}


class OracleSampler:
    """The fp64 CPU oracle on the same workload, on bounded samples: whole
    (request, KV head) groups (all query heads of the group, every query row)
    in batch order, `chunk` groups per oracle call (rows spread over
    `n_threads` threads). The append is applied once, up front."""

    def __init__(self, b: wl.PagedBatch, n_threads: int):
        import oracle
        self.oracle = oracle
        self.b = b
        self.n_threads = n_threads
        self.kp, self.vp = b.key_pages.copy(), b.value_pages.copy()
        oracle.append_kv(b.key_new, b.value_new, self.kp, self.vp, b.slot_mapping, b.page_size)
        self.G = b.H_q // b.H_kv
        self.groups = [(r, h) for r in range(b.B) for h in range(b.H_kv)]
        self.k = 0

    def run(self, budget_s: float, chunk=None):
        """Runs calls until budget_s has passed (at least one call).
        Returns (GB/s of K/V read, groups done, seconds)."""
        b, G = self.b, self.G
        if chunk is None:
            chunk = max(1, min(len(self.groups), -(-self.n_threads // (G * b.L))))
        done_bytes, n_groups, t_start = 0, 0, time.perf_counter()
        while True:
            sel = [self.groups[(self.k + j) % len(self.groups)] for j in range(chunk)]
            self.k += chunk
            rows = np.asarray([(r, h * G + g, i) for r, h in sel for g in range(G)
                               for i in range(b.L)], dtype=np.int32)
            self.oracle.attention(b.query, self.kp, self.vp, b.block_table, b.context_lens,
                                  b.page_size, scale=b.scale, causal=b.causal, rows=rows,
                                  n_threads=self.n_threads)
            done_bytes += sum(int(b.context_lens[r]) * b.D * 2 * 2 for r, _ in sel)
            n_groups += len(sel)
            el = time.perf_counter() - t_start
            if el >= budget_s:
                return done_bytes / el / 1e9, n_groups, el


def cpu_model() -> str:
    """The host CPU's model name: /proc/cpuinfo's "model name" (x86), else
    lscpu's "Model name" (Arm hosts such as Grace), else the Arm implementer
    and part codes of /proc/cpuinfo."""
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip().lower(), v.strip())
    except OSError:
        pass
    if fields.get("model name"):
        return fields["model name"]
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    if "cpu implementer" in fields:
        return f"implementer {fields['cpu implementer']} part {fields.get('cpu part', '?')}"
    return "unknown"


def decode_cpu_baseline(b: wl.PagedBatch, budget_s: float):
    """The oracle on bounded samples of the decode workload, single-threaded
    and on every host core (rates in GB/s of K/V read)."""
    cores = os.cpu_count() or 1
    sampler = OracleSampler(b, 1)
    r1, g1, t1 = sampler.run(0.35 * budget_s, chunk=1)
    sampler.n_threads = cores
    ra, ga, ta = sampler.run(0.65 * budget_s)
    return {"value": round(ra, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{b.name}: whole (request, KV head) groups (all {b.H_q // b.H_kv} query "
                      f"heads each) in batch order; {ga} groups in {ta:.1f} s on {cores} "
                      f"threads, {g1} groups in {t1:.1f} s on 1 thread; GB/s of K/V read",
            "threads_1": {"value": round(r1, 4), "groups": g1, "seconds": round(t1, 2)},
            "threads_all": {"value": round(ra, 4), "threads": cores, "groups": ga,
                            "seconds": round(ta, 2)},
            "cpu_model": cpu_model()}


def prefill_cpu_baseline(b: wl.PagedBatch, budget_s: float, tile: int = 128):
    """The oracle on sampled query tiles of the prefill chunk (after its
    append), single-threaded and on every host core. A unit is one (request,
    query head, 128-row query tile); units are drawn in a seeded random
    order. Rate: causal-useful GFLOP/s (4 * D per visible (row, key) pair)."""
    import oracle
    cores = os.cpu_count() or 1
    kp, vp = b.key_pages.copy(), b.value_pages.copy()
    oracle.append_kv(b.key_new, b.value_new, kp, vp, b.slot_mapping, b.page_size)
    n_tiles = -(-b.L // tile)
    units = [(r, h, t) for r in range(b.B) for h in range(b.H_q) for t in range(n_tiles)]
    order = np.random.default_rng(b.seed + 11).permutation(len(units))

    def run(threads, budget, k0):
        flops, done, k, t_start = 0.0, 0, k0, time.perf_counter()
        while True:
            r, h, t = units[int(order[k % len(units)])]
            k += 1
            rows = np.asarray([(r, h, i) for i in range(t * tile, min(b.L, (t + 1) * tile))],
                              dtype=np.int32)
            oracle.attention(b.query, kp, vp, b.block_table, b.context_lens, b.page_size,
                             scale=b.scale, causal=b.causal, rows=rows, n_threads=threads)
            n = int(b.context_lens[r])
            vis = [min(n, n - b.L + i + 1) if b.causal else n for i in rows[:, 2]]
            flops += 4.0 * b.D * sum(max(0, v) for v in vis)
            done += 1
            el = time.perf_counter() - t_start
            if el >= budget:
                return flops / el / 1e9, done, el, k

    g1, u1, t1, k = run(1, 0.35 * budget_s, 0)
    ga, ua, ta, _ = run(cores, 0.65 * budget_s, k)
    return {"value": round(ga, 4), "unit": "GFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{b.name}: (request, query head, {tile}-row query tile) units in a "
                      f"seeded random order; {ua} units in {ta:.1f} s on {cores} threads, "
                      f"{u1} in {t1:.1f} s on 1 thread; causal-useful GFLOP/s",
            "threads_1": {"value": round(g1, 4), "units": u1, "seconds": round(t1, 2)},
            "threads_all": {"value": round(ga, 4), "threads": cores, "units": ua,
                            "seconds": round(ta, 2)},
            "cpu_model": cpu_model()}


def run_reference(args, rank, world):
    """The reference arm: the fp64 CPU oracle, as it stands, on the host cores."""
    if rank != 0:
        return 0
    b = wl.make_workload(args.workload)
    cores = os.cpu_count() or 1
    dec_bytes, _ = step_bytes(b)
    total_budget = 150.0
    per_step = max(0.02, total_budget / max(1, args.steps + args.warmup))
    sampler = OracleSampler(b, cores)
    for _ in range(args.warmup):
        sampler.run(per_step, chunk=1)
    t0 = time.perf_counter()
    rates = []
    groups = 0
    for _ in range(args.steps):
        r, g, _ = sampler.run(per_step, chunk=1)
        rates.append(r)
        groups += g
    el = time.perf_counter() - t0
    value = float(np.mean(rates))
    sample = (f"{args.workload}: per step, whole (request, KV head) groups of the batch "
              f"(all query heads and rows of each) for ~{per_step:.3f} s; {groups} groups over "
              f"{args.steps} steps; GB/s of K/V read")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * el / max(1, args.steps), 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(b, world, "none (CPU)"),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                             "kind": "oracle", "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _bench_lib(binding):
    """ctypes view of the native step loops (bench_loop.cpp)."""
    import ctypes
    from paged_kv_attention_06_gb300 import build as pkg_build
    lib = ctypes.CDLL(pkg_build.BENCH_LIB)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    pvp = ctypes.POINTER(ctypes.c_void_p)
    lib.pa_bench_steps.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, pvp, pvp,
                                   vp, i32,
                                   binding.pa_shape, vp, vp, vp, f32, ctypes.c_int, vp,
                                   binding.pa_shape, i32, vp, sz, vp,
                                   ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)]
    lib.pa_bench_steps.restype = ctypes.c_int
    lib.pa_bench_e2e_steps.argtypes = [ctypes.c_int, ctypes.c_int, pvp, pvp,
                                       ctypes.POINTER(ctypes.c_size_t), ctypes.c_int, vp, vp, sz,
                                       vp, vp, pvp, pvp, vp, i32, binding.pa_shape, vp, vp, vp,
                                       f32, ctypes.c_int, vp, binding.pa_shape, i32, vp, sz, vp,
                                       ctypes.POINTER(ctypes.c_float)]
    lib.pa_bench_e2e_steps.restype = ctypes.c_int
    lib.pa_bench_e2e_pipelined.argtypes = [ctypes.c_int, ctypes.c_int, vp, pvp, sz,
                                           ctypes.POINTER(ctypes.c_size_t), pvp, pvp, sz, pvp, pvp,
                                           i32, binding.pa_shape, f32, ctypes.c_int,
                                           binding.pa_shape, i32, vp, sz, vp, vp, vp,
                                           ctypes.POINTER(ctypes.c_float)]
    lib.pa_bench_e2e_pipelined.restype = ctypes.c_int
    lib.pa_bench_steps_fp8.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, pvp,
                                       pvp, vp, i32, binding.pa_shape, vp, vp, vp, f32, f32, f32,
                                       ctypes.c_int, vp, binding.pa_shape, i32, vp, sz, vp,
                                       ctypes.POINTER(ctypes.c_float),
                                       ctypes.POINTER(ctypes.c_float)]
    lib.pa_bench_steps_fp8.restype = ctypes.c_int
    lib.pa_bench_attention_calls.argtypes = [ctypes.c_int, ctypes.c_int, pvp, pvp, vp, vp, vp, i32,
                                             f32, ctypes.c_int, ctypes.c_int, f32, f32, vp,
                                             binding.pa_shape, i32, vp, sz, vp,
                                             ctypes.POINTER(ctypes.c_float)]
    lib.pa_bench_attention_calls.restype = ctypes.c_int
    return lib


CALL_WARMUP, CALL_BLOCK, CALL_BLOCKS = 5, 60, 4
PREFILL_BLOCK, PREFILL_BLOCKS = 20, 4


def time_calls(blib, n_copies, kps, vps, q, bt, cl, page_size, scale, causal, out, shape,
               max_ctx, ws, ws_bytes, stream, fp8=False, k_scale=1.0, v_scale=1.0):
    """Device time of one attention call: CALL_WARMUP untimed calls, then
    CALL_BLOCKS blocks of CALL_BLOCK back-to-back calls, each block bracketed
    by CUDA events (none between calls). Returns (median over blocks of the
    per-call ms, the blocks' per-call ms)."""
    import ctypes

    def block(n):
        total = ctypes.c_float(0)
        st = blib.pa_bench_attention_calls(n, n_copies, kps, vps, q, bt, cl, page_size, scale,
                                           int(causal), int(fp8), k_scale, v_scale, out, shape,
                                           max_ctx, ws, ws_bytes, stream, ctypes.byref(total))
        if st != 0:
            raise RuntimeError(f"native call loop failed with status {st}")
        return float(total.value) / n

    block(CALL_WARMUP)
    per = [block(CALL_BLOCK) for _ in range(CALL_BLOCKS)]
    return float(np.median(per)), per


def workload_config(b, world, l2_note):
    n = b.context_lens
    return {"workload": b.name, "B": b.B, "H_q": b.H_q, "H_kv": b.H_kv, "D": b.D,
            "page_size": b.page_size, "L": b.L, "L_new": b.L_new, "num_pages": b.num_pages,
            "context_lens": {"min": int(n.min()), "max": int(n.max()), "sum": int(n.sum())},
            "recipe": b.recipe, "seed": b.seed, "l2": l2_note,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-budget", type=float, default=8.0,
                    help="seconds of oracle work for the cpu_baseline leg")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--fp8-decode", action="store_true",
                    help="time only the decode step over e4m3 page pools of --workload and exit")
    ap.add_argument("--prefill-shapes", action="store_true",
                    help="time both prefill kernels on chunked-prefill shapes and exit")
    ap.add_argument("--shape", default=None, help="with --prefill-shapes: only this shape")
    ap.add_argument("--shapes-page-size", type=int, default=16,
                    help="with --prefill-shapes: tokens per page")
    ap.add_argument("--shapes-head-dim", type=int, default=128,
                    help="with --prefill-shapes: head_dim (128 or 64)")
    ap.add_argument("--shapes-heads", default="32x8",
                    help="with --prefill-shapes: query heads x KV heads, e.g. 28x4")
    ap.add_argument("--serving-trace", action="store_true",
                    help="run the synthetic serving trace through pa_kv_cache and exit")
    ap.add_argument("--dense-gather", action="store_true",
                    help="time direct paged decode against gather + dense decode and exit")
    ap.add_argument("--dispatch-sweep", action="store_true",
                    help="time decode vs prefill over query chunk lengths and exit")
    ap.add_argument("--sweep-L", default=None,
                    help="with --dispatch-sweep: comma-separated query chunk lengths only")
    ap.add_argument("--sweep-ctx", default=None,
                    help="with --dispatch-sweep: comma-separated context lengths only")
    ap.add_argument("--sweep-group", default=None,
                    help="with --dispatch-sweep: one head shape only, as H_qxH_kv (e.g. 28x4)")
    ap.add_argument("--no-other-decode", action="store_true",
                    help="skip the other decode workloads (secondary entries)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)

    rank = _env_int("RANK", 0)
    world = _env_int("WORLD_SIZE", 1)
    local_rank = _env_int("LOCAL_RANK", 0)
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    import paged_kv_attention_06_gb300 as pa
    from paged_kv_attention_06_gb300 import binding

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    if args.fp8_decode:
        import paged_kv_attention_06_gb300 as pa
        from paged_kv_attention_06_gb300 import binding
        stream = torch.cuda.current_stream()
        print(json.dumps({"fp8_decode": bench_decode_fp8(args.workload, pa, binding, torch, device,
                                                         stream, args.steps, args.warmup)}))
        return 0
    if args.prefill_shapes:
        hq, hkv = (int(x) for x in args.shapes_heads.split("x"))
        print(json.dumps({"prefill_shapes": prefill_shapes(
            torch, device, args.shape, heads=(hq, hkv), page_size=args.shapes_page_size,
            head_dim=args.shapes_head_dim)}))
        return 0
    if args.serving_trace:
        serving_trace(torch, device)            # warm-up run (builds, first calls)
        print(json.dumps({"serving_trace": serving_trace(torch, device),
                          "serving_trace_python_issue": serving_trace(torch, device, native=False)}))
        return 0
    if args.dense_gather:
        print(json.dumps({"dense_gather": dense_gather_bench(torch, device),
                          "timing": "CUDA graph of 20 calls over 4 rotating pools and dense "
                                    "buffers, replayed 3 times, events around the replays; "
                                    "median of 4"}))
        return 0
    if args.dispatch_sweep:
        kw = {}
        if args.sweep_L:
            kw["Ls"] = tuple(int(x) for x in args.sweep_L.split(","))
        if args.sweep_ctx:
            kw["ctxs"] = tuple(int(x) for x in args.sweep_ctx.split(","))
        if args.sweep_group:
            hq, hkv = (int(x) for x in args.sweep_group.lower().split("x"))
            kw["groups"] = ((hq, hkv),)
        print(json.dumps({"dispatch_sweep": dispatch_sweep(torch, device, **kw),
                          "timing": "CUDA graph of 16 calls over 4 rotating pool copies, "
                                    "replayed 3 times, events around the replays"}))
        return 0
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    b = wl.make_workload(args.workload)

    def to_dev(x):
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(np.ascontiguousarray(x)).to(device)

    dec_bytes, app_bytes = step_bytes(b)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    pool_bytes = 2 * b.key_pages.nbytes
    copies = max(4, math.ceil(4 * l2 / max(1, dec_bytes)))
    kp0, vp0 = to_dev(b.key_pages), to_dev(b.value_pages)
    pools = [(kp0, vp0)] + [(kp0.clone(), vp0.clone()) for _ in range(copies - 1)]
    q = to_dev(b.query)
    bt = to_dev(b.block_table)
    cl = to_dev(b.context_lens)
    kn, vn = to_dev(b.key_new), to_dev(b.value_new)
    sm = to_dev(b.slot_mapping)
    out = torch.empty_like(q)
    shape = pa.make_shape(q.shape, kp0.shape, bt.shape[1])
    app_shape = pa.pa_shape(b.B, 0, b.H_kv, b.D, b.L_new, b.num_pages, 0)
    ws, ws_need = pa.decode_workspace(shape, device)
    stream = torch.cuda.current_stream(device)
    sp = stream.cuda_stream
    max_ctx = int(b.context_lens.max())
    lib = binding._lib
    route = int(lib.pa_attention_route(shape, max_ctx))

    # The timed steps are issued from C (bench_loop.cpp) through the public
    # C ABI, so that no interpreter work sits between launches.
    import ctypes
    blib = _bench_lib(binding)
    kps = (ctypes.c_void_p * copies)(*[kp.data_ptr() for kp, _ in pools])
    vps = (ctypes.c_void_p * copies)(*[vp_.data_ptr() for _, vp_ in pools])

    def run_steps(n):
        """n steps with no event between them; returns their device ms."""
        total = ctypes.c_float(0)
        st = blib.pa_bench_steps(n, 0, copies, kn.data_ptr(), vn.data_ptr(), kps, vps,
                                 sm.data_ptr(), b.page_size, app_shape, q.data_ptr(),
                                 bt.data_ptr(), cl.data_ptr(), b.scale, int(b.causal),
                                 out.data_ptr(), shape, max_ctx, ws.data_ptr(), ws_need, sp,
                                 None, ctypes.byref(total))
        if st != 0:
            raise RuntimeError(f"native step loop failed with status {st}")
        return float(total.value)

    # The K timed steps run as up to four blocks of at least 25 steps, each
    # bracketed by events (none inside a block); the step time is their sum
    # over K, and the blocks' own per-step times give the repeat spread. A
    # block boundary breaks the kernels' launch overlap once, so short runs
    # take one block.
    n_blocks = max(1, min(4, args.steps // 25))
    block_sizes = [args.steps // n_blocks + (1 if i < args.steps % n_blocks else 0)
                   for i in range(n_blocks)]

    def run_blocks():
        return [run_steps(n) for n in block_sizes]

    run_steps(args.warmup)
    torch.cuda.synchronize()
    status, flags = pa.pa_get_device_error()
    if status:
        raise RuntimeError(f"device error during warm-up: {flags:#x}")

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    wall0 = time.time()
    host0 = time.perf_counter()
    block_ms = timed_region(dist, torch.cuda.synchronize, run_blocks)
    host_s = time.perf_counter() - host0
    wall1 = time.time()
    total_ms = max_over_ranks(dist, sum(block_ms), device)
    block_step_ms = [t / n for t, n in zip(block_ms, block_sizes)]

    # One decode call alone: blocks of back-to-back calls over the rotating
    # pool copies, events only around each block.
    call_ms, call_blocks = time_calls(blib, copies, kps, vps, q.data_ptr(), bt.data_ptr(),
                                      cl.data_ptr(), b.page_size, b.scale, b.causal,
                                      out.data_ptr(), shape, max_ctx, ws.data_ptr(), ws_need, sp)
    call_ms = max_over_ranks(dist, call_ms, device)
    status, flags = pa.pa_get_device_error()
    if status:
        raise RuntimeError(f"device error in the timed region: {flags:#x}")
    total_ms = max_over_ranks(dist, total_ms, device)

    # ---- e2e: same step through the C ABI from pinned host buffers ---------
    # The step's inputs (query, new K/V, slots, block table, context lengths)
    # sit at 256-byte-aligned offsets of one pinned host region and one device
    # region, so each step moves them with one host-to-device copy; the
    # kernels read them in place, and the output comes back with one copy.
    parts = [b.query, b.key_new, b.value_new, b.slot_mapping, b.block_table, b.context_lens]
    offs, packed = [], 0
    for x in parts:
        offs.append(packed)
        packed += -(-x.nbytes // 256) * 256
    h_in = torch.empty(packed, dtype=torch.uint8).pin_memory()
    for x, o in zip(parts, offs):
        h_in[o:o + x.nbytes] = torch.from_numpy(np.ascontiguousarray(x).reshape(-1).view(np.uint8))
    d_in = torch.empty(packed, dtype=torch.uint8, device=device)
    d_q, d_kn, d_vn, d_sm, d_bt, d_cl = [d_in.data_ptr() + o for o in offs]
    h_out = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    h2d = packed
    d2h = h_out.numel() * h_out.element_size()
    e2e_steps = max(10, min(args.steps, 2000))
    src = (ctypes.c_void_p * 1)(h_in.data_ptr())
    dst = (ctypes.c_void_p * 1)(d_in.data_ptr())
    szs = (ctypes.c_size_t * 1)(packed)

    def run_e2e(n):
        total = ctypes.c_float(0)
        st = blib.pa_bench_e2e_steps(n, copies, src, dst, szs, 1, out.data_ptr(),
                                     h_out.data_ptr(), d2h, d_kn, d_vn, kps, vps, d_sm,
                                     b.page_size, app_shape, d_q, d_bt, d_cl, b.scale,
                                     int(b.causal), out.data_ptr(), shape, max_ctx, ws.data_ptr(),
                                     ws_need, sp, ctypes.byref(total))
        if st != 0:
            raise RuntimeError(f"native e2e loop failed with status {st}")
        return float(total.value)

    run_e2e(3)
    serial_ms = max_over_ranks(dist, timed_region(dist, torch.cuda.synchronize,
                                                  lambda: run_e2e(e2e_steps)) / e2e_steps,
                               device)

    # The same steps with the copies of step k +- 1 overlapping step k's kernels
    # (a copy stream, two input regions and two output buffers on each side).
    d_in2 = [d_in, torch.empty(packed, dtype=torch.uint8, device=device)]
    outs2 = [out, torch.empty_like(q)]
    h_out2 = [h_out, torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()]
    copy_stream, out_stream = torch.cuda.Stream(device), torch.cuda.Stream(device)
    offs_c = (ctypes.c_size_t * 6)(*offs)
    din_c = (ctypes.c_void_p * 2)(*[t.data_ptr() for t in d_in2])
    dout_c = (ctypes.c_void_p * 2)(*[t.data_ptr() for t in outs2])
    hout_c = (ctypes.c_void_p * 2)(*[t.data_ptr() for t in h_out2])

    def run_e2e_pipelined(n):
        total = ctypes.c_float(0)
        st = blib.pa_bench_e2e_pipelined(n, copies, h_in.data_ptr(), din_c, packed, offs_c,
                                         dout_c, hout_c, d2h, kps, vps, b.page_size, app_shape,
                                         b.scale, int(b.causal), shape, max_ctx, ws.data_ptr(),
                                         ws_need, sp, copy_stream.cuda_stream,
                                         out_stream.cuda_stream, ctypes.byref(total))
        if st != 0:
            raise RuntimeError(f"native pipelined e2e loop failed with status {st}")
        return float(total.value)

    run_e2e_pipelined(3)
    e2e_ms = max_over_ranks(dist, timed_region(dist, torch.cuda.synchronize,
                                               lambda: run_e2e_pipelined(e2e_steps)) / e2e_steps,
                            device)

    # ---- secondary: the other decode workloads ------------------------------
    other_decode = []
    if not args.no_other_decode and world == 1:
        for name, n in (("decode_b64_ps128", 400), ("decode_long_b8", 200)):
            if name != args.workload:
                other_decode.append(bench_decode_config(name, pa, binding, torch, device,
                                                        stream, n))
    # the same decode step over e4m3 page pools (half the K/V bytes)
    fp8_decode = None
    if not args.no_other_decode and world == 1 and b.D == 128:
        fp8_decode = bench_decode_fp8(b.name, pa, binding, torch, device, stream, 2000)
        fp8_decode["other"] = [bench_decode_fp8(name, pa, binding, torch, device, stream, n)
                               for name, n in (("decode_b64_ps128", 400), ("decode_long_b8", 200))]

    # ---- secondary: chunked prefill TFLOP/s (prefill route) -----------------
    prefill = None
    if not args.no_prefill and world == 1:
        prefill = bench_prefill(pa, binding, torch, device, stream, cpu_budget=0.75 * args.cpu_budget)

    clocks.stop()
    ck = clocks.summary(wall0, wall1)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    ms_step = total_ms / args.steps
    value = whole_job_gbs(world, dec_bytes + app_bytes, ms_step)
    hbm_peak, bf16_peak, peak_kind = load_peaks()
    achieved = dec_bytes / (call_ms * 1e-3) / 1e9
    traffic = committed_traffic("decode_kernel", b.name)
    cpu = None
    if world == 1 or rank == 0:
        cpu = decode_cpu_baseline(b, args.cpu_budget)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": workload_config(
            b, world, f"{copies} rotating copies of the K/V pool "
                      f"({copies * pool_bytes / 1e6:.0f} MB vs {l2 / 1e6:.0f} MB L2): each "
                      f"step reads a copy last touched {copies - 1} steps earlier"),
        "tokens_per_s": round(world * b.B / (ms_step * 1e-3), 1),
        "step_blocks_ms_per_step": [round(t, 6) for t in block_step_ms],
        "step_median_of_blocks_ms": round(float(np.median(block_step_ms)), 6),
        "step_spread": round((max(block_step_ms) - min(block_step_ms)) /
                             float(np.median(block_step_ms)), 4),
        "decode_call_us": round(1e3 * call_ms, 3),
        "decode_call_blocks_us": [round(1e3 * t, 3) for t in call_blocks],
        "decode_call_spread": round((max(call_blocks) - min(call_blocks)) / float(np.median(
            call_blocks)), 4),
        "decode_call_timing": (f"{CALL_WARMUP} warm-up calls, then {CALL_BLOCKS} blocks of "
                               f"{CALL_BLOCK} back-to-back pa_attention calls over the rotating "
                               f"pool copies, CUDA events around each block only; median of "
                               f"the blocks' per-call times"),
        "route": "decode" if route == 0 else "prefill",
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                     "traffic": traffic, "peak_source": f"{peak_kind} hbm_gbs",
                     "kernel": "decode_kernel<128> + decode_merge_kernel<128> (one pa_decode call)",
                     "algorithmic_bytes_per_launch": dec_bytes},
        "cpu_baseline": cpu,
        "e2e": {"value": round(whole_job_gbs(world, dec_bytes + app_bytes, e2e_ms), 3),
                "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies_per_step": {"h2d": 1, "d2h": 1,
                                    "inputs": "query, new K/V, slots, block table and context "
                                              "lengths packed in one pinned region"},
                "pipelined": "step k's input copy runs while step k - 1 computes and its "
                             "output copy while step k + 1 computes (one stream for input "
                             "copies, one for output copies, double buffers); every step's "
                             "copies are inside the timed region",
                "serial_ms_per_step": round(serial_ms, 6),
                "ms_per_step": round(e2e_ms, 6), "steps": e2e_steps},
        "gpu_launches": (3 if route == 0 else 2) * args.steps,
        "timed_loop": "native C loop over the C ABI (bench_loop.cpp)",
        "host_wall_us_per_step": round(1e6 * host_s / args.steps, 2),
        "clocks": ck,
    }
    if other_decode:
        line["other_decode"] = other_decode
    if fp8_decode is not None:
        line["fp8_decode"] = fp8_decode
    if prefill is not None:
        prefill["roofline_frac_bf16"] = round(prefill["tflops"] / bf16_peak, 4)
        prefill["peak_source"] = f"{peak_kind} bf16_tflops"
        line["prefill"] = prefill
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def bench_decode_fp8(name, pa, binding, torch, device, stream, steps, warmup=10,
                     k_scale=0.05, v_scale=0.05):
    """The decode workload with e4m3 page pools (seeded random codes,
    per-tensor scales): pa_append_kv_fp8 + pa_decode_fp8 per step through the
    native loop, rotating pool copies; bytes counted at one byte per K/V
    element."""
    import ctypes
    b = wl.make_workload(name)
    rng = np.random.default_rng(b.seed + 7)

    def to_dev(x):
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(np.ascontiguousarray(x)).to(device)

    bf16_bytes, _ = step_bytes(b)
    kv_bf16 = int(b.context_lens.astype(np.int64).sum()) * b.H_kv * b.D * 2 * 2
    dec_bytes = bf16_bytes - kv_bf16 // 2
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    copies = max(4, math.ceil(4 * l2 / max(1, dec_bytes)))
    kp0 = to_dev(wl.random_e4m3_codes(rng, b.key_pages.shape))
    vp0 = to_dev(wl.random_e4m3_codes(rng, b.value_pages.shape))
    pools = [(kp0, vp0)] + [(kp0.clone(), vp0.clone()) for _ in range(copies - 1)]
    q, bt, cl = to_dev(b.query), to_dev(b.block_table), to_dev(b.context_lens)
    kn, vn, sm = to_dev(b.key_new), to_dev(b.value_new), to_dev(b.slot_mapping)
    out = torch.empty_like(q)
    shape = pa.make_shape(q.shape, kp0.shape, bt.shape[1])
    app_shape = pa.pa_shape(b.B, 0, b.H_kv, b.D, b.L_new, b.num_pages, 0)
    ws, ws_need = pa.decode_workspace(shape, device)
    blib = _bench_lib(binding)
    kps = (ctypes.c_void_p * copies)(*[kp.data_ptr() for kp, _ in pools])
    vps = (ctypes.c_void_p * copies)(*[vp_.data_ptr() for _, vp_ in pools])
    def run(n):
        total = ctypes.c_float(0)
        st = blib.pa_bench_steps_fp8(n, 0, copies, kn.data_ptr(), vn.data_ptr(), kps,
                                     vps, sm.data_ptr(), b.page_size, app_shape, q.data_ptr(),
                                     bt.data_ptr(), cl.data_ptr(), b.scale, k_scale, v_scale,
                                     int(b.causal), out.data_ptr(), shape,
                                     int(b.context_lens.max()), ws.data_ptr(), ws_need,
                                     stream.cuda_stream, None, ctypes.byref(total))
        if st != 0:
            raise RuntimeError(f"native fp8 step loop failed with status {st} on {name}")
        return float(total.value)

    run(warmup)
    torch.cuda.synchronize()
    total_ms = run(steps)
    dec_avg, _ = time_calls(blib, copies, kps, vps, q.data_ptr(), bt.data_ptr(), cl.data_ptr(),
                            b.page_size, b.scale, b.causal, out.data_ptr(), shape,
                            int(b.context_lens.max()), ws.data_ptr(), ws_need,
                            stream.cuda_stream, fp8=True, k_scale=k_scale, v_scale=v_scale)
    torch.cuda.synchronize()
    st, flags = pa.pa_get_device_error()
    if st:
        raise RuntimeError(f"device error in fp8 decode bench {name}: {flags:#x}")
    hbm_peak, _, peak_kind = load_peaks()
    ms_step = total_ms / steps
    res = {"workload": name, "pages": "e4m3, per-tensor scales", "ms_per_step": round(ms_step, 6),
           "tokens_per_s": round(b.B * b.L / (ms_step * 1e-3), 1),
           "decode_call_us": round(1e3 * dec_avg, 3),
           "decode_gbs": round(dec_bytes / (dec_avg * 1e-3) / 1e9, 2),
           "frac": round(dec_bytes / (dec_avg * 1e-3) / 1e9 / hbm_peak, 4),
           "peak_source": f"{peak_kind} hbm_gbs", "algorithmic_bytes_per_launch": dec_bytes,
           "kernel": "decode_kernel<128, e4m3> + decode_merge_kernel<128>",
           "steps": steps, "l2": f"{copies} rotating pool copies"}
    del pools, ws
    torch.cuda.empty_cache()
    return res


def bench_decode_config(name, pa, binding, torch, device, stream, steps, warmup=10):
    """One of the other decode workloads through the same native step loop
    (append + pa_attention per step, rotating pool copies): step time, the
    decode call's event time and its HBM roofline fraction."""
    import ctypes
    b = wl.make_workload(name)

    def to_dev(x):
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(np.ascontiguousarray(x)).to(device)

    dec_bytes, app_bytes = step_bytes(b)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    copies = max(4, math.ceil(4 * l2 / max(1, dec_bytes)))
    kp0, vp0 = to_dev(b.key_pages), to_dev(b.value_pages)
    pools = [(kp0, vp0)] + [(kp0.clone(), vp0.clone()) for _ in range(copies - 1)]
    q, bt, cl = to_dev(b.query), to_dev(b.block_table), to_dev(b.context_lens)
    kn, vn, sm = to_dev(b.key_new), to_dev(b.value_new), to_dev(b.slot_mapping)
    out = torch.empty_like(q)
    shape = pa.make_shape(q.shape, kp0.shape, bt.shape[1])
    app_shape = pa.pa_shape(b.B, 0, b.H_kv, b.D, b.L_new, b.num_pages, 0)
    ws, ws_need = pa.decode_workspace(shape, device)
    blib = _bench_lib(binding)
    kps = (ctypes.c_void_p * copies)(*[kp.data_ptr() for kp, _ in pools])
    vps = (ctypes.c_void_p * copies)(*[vp_.data_ptr() for _, vp_ in pools])
    def run(n):
        total = ctypes.c_float(0)
        st = blib.pa_bench_steps(n, 0, copies, kn.data_ptr(), vn.data_ptr(), kps, vps,
                                 sm.data_ptr(), b.page_size, app_shape, q.data_ptr(),
                                 bt.data_ptr(), cl.data_ptr(), b.scale, int(b.causal),
                                 out.data_ptr(), shape, int(b.context_lens.max()), ws.data_ptr(),
                                 ws_need, stream.cuda_stream, None, ctypes.byref(total))
        if st != 0:
            raise RuntimeError(f"native step loop failed with status {st} on {name}")
        return float(total.value)

    run(warmup)
    torch.cuda.synchronize()
    total_ms = run(steps)
    dec_avg, _ = time_calls(blib, copies, kps, vps, q.data_ptr(), bt.data_ptr(), cl.data_ptr(),
                            b.page_size, b.scale, b.causal, out.data_ptr(), shape,
                            int(b.context_lens.max()), ws.data_ptr(), ws_need,
                            stream.cuda_stream)
    torch.cuda.synchronize()
    st, flags = pa.pa_get_device_error()
    if st:
        raise RuntimeError(f"device error in decode bench {name}: {flags:#x}")
    hbm_peak, _, peak_kind = load_peaks()
    ms_step = total_ms / steps
    res = {"workload": name, "ms_per_step": round(ms_step, 6),
           "step_gbs": round((dec_bytes + app_bytes) / (ms_step * 1e-3) / 1e9, 2),
           "decode_call_us": round(1e3 * dec_avg, 3),
           "decode_gbs": round(dec_bytes / (dec_avg * 1e-3) / 1e9, 2),
           "frac": round(dec_bytes / (dec_avg * 1e-3) / 1e9 / hbm_peak, 4),
           "peak_source": f"{peak_kind} hbm_gbs", "algorithmic_bytes_per_launch": dec_bytes,
           "steps": steps, "l2": f"{copies} rotating pool copies"}
    del pools, ws
    torch.cuda.empty_cache()
    return res


def dispatch_sweep(torch, device, Ls=(1, 2, 4, 8, 12, 16, 24, 32, 48, 64, 96, 128),
                   ctxs=(1024, 4096), groups=((28, 4), (32, 8), (8, 8)), B=32, page_size=16,
                   copies=4, calls=16):
    """Time pa_decode and pa_prefill on the same inputs for query chunks of L
    rows (both are correct for every L): the data behind the L threshold of
    pa_attention_route. Each timing is a CUDA graph of `calls` calls over
    `copies` rotating pool copies, replayed 3 times, CUDA events around the
    replays (no interpreter between launches)."""
    import paged_kv_attention_06_gb300 as pa

    def to_dev(x):
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(np.ascontiguousarray(x)).to(device)

    rows = []
    for (H_q, H_kv) in groups:
        for ctx in ctxs:
            base = wl.build_batch(f"sweep_g{H_q // H_kv}_n{ctx}", B=B, H_q=H_q, H_kv=H_kv, D=128,
                                  page_size=page_size, L=1, context_lens=[ctx] * B,
                                  seed=4242 + ctx + H_q, L_new=1)
            kp0, vp0 = to_dev(base.key_pages), to_dev(base.value_pages)
            pools = [(kp0, vp0)] + [(kp0.clone(), vp0.clone()) for _ in range(copies - 1)]
            bt, cl = to_dev(base.block_table), to_dev(base.context_lens)
            for L in Ls:
                q = torch.randn(B, H_q, L, 128, device=device).to(torch.bfloat16)
                out = torch.empty_like(q)
                res = {}
                for kind in ("decode", "prefill"):
                    def call(c):
                        kp, vp_ = pools[c % copies]
                        if kind == "decode":
                            pa.pa_decode(q, kp, vp_, bt, cl, page_size, scale=base.scale, out=out,
                                         max_context_len=ctx)
                        else:
                            pa.pa_prefill(q, kp, vp_, bt, cl, page_size, scale=base.scale, out=out)
                    for c in range(3):
                        call(c)
                    torch.cuda.synchronize()
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g):
                        for c in range(calls):
                            call(c)
                    g.replay()
                    torch.cuda.synchronize()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    for _ in range(3):
                        g.replay()
                    e1.record()
                    torch.cuda.synchronize()
                    res[kind] = e0.elapsed_time(e1) * 1e3 / (3 * calls)
                    del g
                st, flags = pa.pa_get_device_error()
                if st:
                    raise RuntimeError(f"device error in the dispatch sweep: {flags:#x}")
                rows.append({"G": H_q // H_kv, "H_q": H_q, "H_kv": H_kv, "ctx": ctx, "L": L,
                             "decode_us": round(res["decode"], 2),
                             "prefill_us": round(res["prefill"], 2),
                             "faster": "decode" if res["decode"] <= res["prefill"] else "prefill"})
            del pools
            torch.cuda.empty_cache()
    return rows


def dense_gather_bench(torch, device, ctxs=(128, 1024), batches=(1, 32), H_q=32, H_kv=8,
                       page_size=128, copies=4, calls=20, repeats=4):
    """The pages' operator comparison (tiny-llm "Measure the Direct Page
    Walk": the dense path with its page-to-dense gather against the direct
    page walk, Qwen3-4B decode shape, contexts 128 and 1024, page size 128),
    on GB300: pa_decode over the pages, pa_gather_kv + pa_decode_dense, and
    pa_decode_dense alone. Each time: a CUDA graph of `calls` calls over
    `copies` rotating pools (and dense buffers), replayed 3 times, CUDA
    events around the replays; the median of `repeats` such measurements."""
    import paged_kv_attention_06_gb300 as pa

    def to_dev(x):
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(np.ascontiguousarray(x)).to(device)

    rows = []
    for B in batches:
        for ctx in ctxs:
            base = wl.build_batch(f"densegather_b{B}_n{ctx}", B=B, H_q=H_q, H_kv=H_kv, D=128,
                                  page_size=page_size, L=1, context_lens=[ctx] * B,
                                  seed=777 + B + ctx, L_new=1, placement="churn")
            kp0, vp0 = to_dev(base.key_pages), to_dev(base.value_pages)
            pools = [(kp0, vp0)] + [(kp0.clone(), vp0.clone()) for _ in range(copies - 1)]
            bt, cl = to_dev(base.block_table), to_dev(base.context_lens)
            q = to_dev(base.query)
            out = torch.empty_like(q)
            N = max(64, -(-ctx // 64) * 64)
            dense = [(torch.empty((B, H_kv, N, 128), dtype=torch.bfloat16, device=device),
                      torch.empty((B, H_kv, N, 128), dtype=torch.bfloat16, device=device))
                     for _ in range(copies)]
            for c in range(copies):
                pa.pa_gather_kv(pools[c][0], pools[c][1], bt, cl, page_size, N,
                                key_dense=dense[c][0], value_dense=dense[c][1])
            res = {}
            for kind in ("paged", "gather+dense", "dense_only"):
                def call(c):
                    kp, vp_ = pools[c % copies]
                    kd, vd = dense[c % copies]
                    if kind == "paged":
                        pa.pa_decode(q, kp, vp_, bt, cl, page_size, scale=base.scale, out=out,
                                     max_context_len=ctx)
                    else:
                        if kind == "gather+dense":
                            pa.pa_gather_kv(kp, vp_, bt, cl, page_size, N, key_dense=kd,
                                            value_dense=vd)
                        pa.pa_decode_dense(q, kd, vd, cl, scale=base.scale, out=out,
                                           max_context_len=ctx)
                for c in range(5):
                    call(c)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for c in range(calls):
                        call(c)
                ts = []
                for _ in range(repeats):
                    g.replay()
                    torch.cuda.synchronize()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    for _ in range(3):
                        g.replay()
                    e1.record()
                    torch.cuda.synchronize()
                    ts.append(e0.elapsed_time(e1) * 1e3 / (3 * calls))
                res[kind] = float(np.median(ts))
                del g
            st, flags = pa.pa_get_device_error()
            if st:
                raise RuntimeError(f"device error in the dense-gather bench: {flags:#x}")
            kv_bytes = 2 * B * ctx * H_kv * 128 * 2
            rows.append({"B": B, "ctx": ctx, "H_q": H_q, "H_kv": H_kv, "page_size": page_size,
                         "paged_us": round(res["paged"], 2),
                         "gather_plus_dense_us": round(res["gather+dense"], 2),
                         "dense_only_us": round(res["dense_only"], 2),
                         "paged_vs_gather_plus_dense": round(res["gather+dense"] / res["paged"], 3),
                         "kv_bytes": kv_bytes})
            del pools, dense
            torch.cuda.empty_cache()
    return rows


def serving_trace(torch, device, n_seqs=16, batch=4, prompt=(128, 1024), output=(32, 128),
                  chunk=128, H_q=32, H_kv=8, D=128, page_size=16, seed=2024, native=True):
    """A synthetic serving trace shaped like the pages' (16 requests, at most
    4 active, prompts U[128, 1024], outputs U[32, 128], prefill in chunks of
    128 tokens) through one attention layer: every step the C++ pa_kv_cache
    plans the step's block_table, context_lens and slot_mapping once, the
    tables go to the device from pinned buffers, the new K/V rows are
    appended, and attention runs (all decoding requests in one call with
    L = 1; each prefilling request's chunk in its own call). K/V rows and
    queries are seeded normal values (no model). native: each call is one
    pa_kv_cache_step (plan into pinned memory, one table copy, append and
    attention in one C call); otherwise plan, three copies, append and
    attention are issued from Python one by one."""
    import paged_kv_attention_06_gb300 as pa
    rng = np.random.default_rng(seed)
    prompts = rng.integers(prompt[0], prompt[1], size=n_seqs, endpoint=True)
    outputs = rng.integers(output[0], output[1], size=n_seqs, endpoint=True)
    max_ctx = int(prompts.max() + outputs.max())
    max_pages = -(-max_ctx // page_size)
    num_pages = batch * max_pages + 64
    cache = pa.KVCache(num_pages, page_size)
    gen = torch.Generator(device=device).manual_seed(seed)
    kp = torch.randn((num_pages, H_kv, page_size, D), generator=gen, device=device).to(torch.bfloat16)
    vp = torch.randn((num_pages, H_kv, page_size, D), generator=gen, device=device).to(torch.bfloat16)
    # flat buffers; a step uses the leading n * ... elements as a contiguous [n, ..] view
    flat = lambda n: torch.randn((n,), generator=gen, device=device).to(torch.bfloat16)
    k_flat, v_flat = flat(batch * H_kv * chunk * D), flat(batch * H_kv * chunk * D)
    q_flat = flat(batch * H_q * chunk * D)
    # one pinned staging region per call of a step (the copies are asynchronous)
    regions = batch + 1
    h_bt = torch.empty((regions, batch * max_pages), dtype=torch.int32).pin_memory()
    h_cl = torch.empty((regions, batch), dtype=torch.int32).pin_memory()
    h_sm = torch.empty((regions, batch * chunk), dtype=torch.int32).pin_memory()
    d_bt = torch.empty((batch * max_pages,), dtype=torch.int32, device=device)
    d_cl = torch.empty((batch,), dtype=torch.int32, device=device)
    d_sm = torch.empty((batch * chunk,), dtype=torch.int32, device=device)
    # native steps: packed tables, one pinned region per call of a step
    tab_bytes = pa.KVCache.step_table_bytes(batch, max_pages, chunk)
    h_tab = torch.empty((regions, tab_bytes), dtype=torch.uint8).pin_memory()
    d_tab = torch.empty((regions, tab_bytes), dtype=torch.uint8, device=device)
    o_flat = torch.empty((batch * H_q * chunk * D,), dtype=torch.bfloat16, device=device)
    ws, _ = pa.decode_workspace(pa.pa_shape(batch, H_q, H_kv, D, 1, num_pages, max_pages), device)
    pws, _ = pa.prefill_workspace(pa.pa_shape(1, H_q, H_kv, D, chunk, num_pages, max_pages),
                                  page_size, device)
    if pws is not None and pws.numel() > ws.numel():
        ws = pws

    def step_native(r, ids, toks, l_new, is_decode):
        n = len(ids)
        kv = (n, H_kv, l_new, D)
        e0, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        cache.step(ids, toks, l_new, max_pages, h_tab[r], d_tab[r],
                   k_flat[:n * H_kv * l_new * D].view(kv), v_flat[:n * H_kv * l_new * D].view(kv),
                   q_flat[:n * H_q * l_new * D].view(n, H_q, l_new, D), kp, vp,
                   out=o_flat[:n * H_q * l_new * D].view(n, H_q, l_new, D), workspace=ws)
        e2.record()
        events.append((e0, e0, e2, is_decode))

    def step(r, ids, toks, l_new, is_decode):
        bt, cl, sm = cache.plan(ids, toks, max_pages, l_new)
        n = len(ids)
        nb, ns = n * max_pages, n * l_new
        h_bt[r, :nb].copy_(torch.from_numpy(bt.reshape(-1)))
        h_cl[r, :n].copy_(torch.from_numpy(cl))
        h_sm[r, :ns].copy_(torch.from_numpy(np.ascontiguousarray(sm).reshape(-1)))
        d_bt[:nb].copy_(h_bt[r, :nb], non_blocking=True)
        d_cl[:n].copy_(h_cl[r, :n], non_blocking=True)
        d_sm[:ns].copy_(h_sm[r, :ns], non_blocking=True)
        kv = (n, H_kv, l_new, D)
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record()
        pa.pa_append_kv(k_flat[:n * H_kv * l_new * D].view(kv), v_flat[:n * H_kv * l_new * D].view(kv),
                        kp, vp, d_sm[:ns].view(n, l_new), page_size)
        e1.record()
        pa.pa_attention(q_flat[:n * H_q * l_new * D].view(n, H_q, l_new, D), kp, vp,
                        d_bt[:nb].view(n, max_pages), d_cl[:n], page_size,
                        max_context_len=int(cl.max()))
        e2.record()
        events.append((e0, e1, e2, is_decode))
    waiting = list(range(n_seqs))
    events = []
    append_ms = decode_ms = prefill_ms = 0.0
    active = {}                        # seq -> [prompt tokens done, output tokens done]
    steps = prefill_tokens = decode_tokens = 0
    host_s = 0.0
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    while waiting or active:
        while waiting and len(active) < batch:
            s_id = waiting.pop(0)
            cache.add(s_id)
            active[s_id] = [0, 0]
        dec = [s_id for s_id, (p_, o_) in active.items() if p_ >= prompts[s_id]]
        pre = [s_id for s_id, (p_, o_) in active.items() if p_ < prompts[s_id]]
        # decode group: one token each, one attention call
        run = step_native if native else step
        if dec:
            t0 = time.perf_counter()
            run(0, dec, [1] * len(dec), 1, True)
            host_s += time.perf_counter() - t0
            decode_tokens += len(dec)
            for s_id in dec:
                active[s_id][1] += 1
        # prefill: each request's next chunk in its own call
        for r, s_id in enumerate(pre, start=1):
            take = int(min(chunk, prompts[s_id] - active[s_id][0]))
            t0 = time.perf_counter()
            run(r, [s_id], [take], take, False)
            host_s += time.perf_counter() - t0
            prefill_tokens += take
            active[s_id][0] += take
        torch.cuda.synchronize()   # the pinned staging buffers are reused next step
        for e0, e1, e2, is_decode in events:
            append_ms += e0.elapsed_time(e1)
            if is_decode:
                decode_ms += e1.elapsed_time(e2)
            else:
                prefill_ms += e1.elapsed_time(e2)
        events.clear()
        for s_id in [s_id for s_id, (p_, o_) in active.items() if o_ >= outputs[s_id]]:
            cache.release(s_id)
            del active[s_id]
        steps += 1
    wall = time.perf_counter() - wall0
    st, flags = pa.pa_get_device_error()
    if st:
        raise RuntimeError(f"device error in the serving trace: {flags:#x}")
    leaked = num_pages - cache.free_pages
    cache.close()
    return {"requests": n_seqs, "max_active": batch, "steps": steps,
            "prefill_tokens": int(prefill_tokens), "decode_tokens": int(decode_tokens),
            "wall_s": round(wall, 4), "tokens_per_s": round((prefill_tokens + decode_tokens) / wall, 1),
            "us_per_step": round(1e6 * wall / steps, 2),
            "host_issue_us_per_step": round(1e6 * host_s / steps, 2),
            "device_us_per_step": {"append": round(1e3 * append_ms / steps, 2),
                                   "decode_attention": round(1e3 * decode_ms / steps, 2),
                                   "prefill_attention": round(1e3 * prefill_ms / steps, 2)},
            "pages_left_held": int(leaked),
            "shape": {"H_q": H_q, "H_kv": H_kv, "D": D, "page_size": page_size, "chunk": chunk,
                      "prompt": list(prompt), "output": list(output)},
            "issue": "native pa_kv_cache_step per call" if native else
                     "plan, table copies, append and attention issued from Python",
            "timing": "wall clock over the whole trace (one device sync per step); device "
                      "times from CUDA events around each append and attention call (native: "
                      "around each whole step call, reported under the attention kind; append 0)"}


PREFILL_SHAPES = [
    # (name, B, L, context_lens): H_q = 32, H_kv = 8, D = 128, page_size 16
    ("chunk512_b4", 4, 512, [1866, 2285, 710, 2052]),
    ("chunk512_b1_prefix16k", 1, 512, [16384 + 512]),
    ("chunk1024_b2_prefix8k", 2, 1024, [9216, 5000]),
    ("prompt2048_b1", 1, 2048, [2048]),
    ("chunk256_b8_mixed", 8, 256, [300, 4000, 800, 2500, 256, 6000, 1200, 3300]),
    ("chunk512_b16", 16, 512, [2347, 3567, 1221, 3885, 597, 1860, 2978, 3327,
                               2150, 802, 1462, 3739, 2811, 1028, 3300, 2444]),
]


def prefill_shapes(torch, device, only=None, steps=15, heads=(32, 8), page_size=16,
                   head_dim=128):
    """The tensor-core prefill paths (pa_attention with its workspace, as the
    product calls it; pa_prefill: whole request x head pair x query tile items
    on one block per SM; pa_prefill_split: K/V tiles spread over one block per
    SM; pa_prefill_fp8 on e4m3 pools) on chunked-prefill shapes with few and
    many query-tile items, L2 flushed before every call, CUDA events. Inputs:
    seeded N(0,1) K/V already in the pages (no append), random page
    permutation. With head_dim 64 or pages of fewer than 8 tokens (the pairs
    kernel only, no e4m3 pools) the split-KV kernel (pa_decode) is timed
    beside it instead."""
    import paged_kv_attention_06_gb300 as pa
    flush = torch.empty(int(2 * torch.cuda.get_device_properties(device).L2_cache_size),
                        dtype=torch.uint8, device=device)

    def to_dev(x):
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(np.ascontiguousarray(x)).to(device)

    def timeit(fn):
        evs = []
        for k in range(steps + 3):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            if k >= 3:
                evs.append((e0, e1))
        torch.cuda.synchronize()
        return float(np.median([x.elapsed_time(y) for x, y in evs])) * 1e3

    rows = []
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    for name, B, L, lens in PREFILL_SHAPES:
        if only and name != only:
            continue
        b = wl.build_batch(name, B=B, H_q=heads[0], H_kv=heads[1], D=head_dim,
                           page_size=page_size, L=L, context_lens=lens, seed=5, L_new=0,
                           placement="permutation")
        pairs_only = head_dim != 128 or page_size < 8
        q, kp, vp = to_dev(b.query), to_dev(b.key_pages), to_dev(b.value_pages)
        bt, cl = to_dev(b.block_table), to_dev(b.context_lens)
        out = torch.empty_like(q)
        t_pairs = timeit(lambda: pa.pa_prefill(q, kp, vp, bt, cl, b.page_size, scale=b.scale,
                                               causal=True, out=out))
        t_split = timeit(lambda: pa.pa_prefill_split(q, kp, vp, bt, cl, b.page_size,
                                                     scale=b.scale, causal=True, out=out))
        # the product path: pa_attention with its prefill workspace (split
        # kernel, pairs kernel with tail pieces, or whole items, by its rule)
        ws_att = torch.empty(max(1, pa.pa_prefill_workspace_bytes(
            pa.make_shape(q.shape, kp.shape, bt.shape[1]), b.page_size)), dtype=torch.uint8,
            device=device)
        mcl_att = int(b.context_lens.max())
        t_att = timeit(lambda: pa.pa_attention(q, kp, vp, bt, cl, b.page_size, scale=b.scale,
                                               causal=True, out=out, max_context_len=mcl_att,
                                               workspace=ws_att))
        del ws_att
        fl = prefill_flops(b)
        items = B * ((L + 127) // 128) * heads[1] * ((heads[0] // heads[1] + 1) // 2)
        if pairs_only:
            ws_dec, _ = pa.decode_workspace(pa.make_shape(q.shape, kp.shape, bt.shape[1]), device)
            t_dec = timeit(lambda: pa.pa_decode(q, kp, vp, bt, cl, b.page_size, scale=b.scale,
                                                causal=True, out=out, max_context_len=mcl_att,
                                                workspace=ws_dec))
            del ws_dec
            rows.append({"shape": name, "items": items, "items_per_sm": round(items / sms, 2),
                         "gflop": round(fl / 1e9, 2), "page_size": page_size,
                         "head_dim": head_dim, "attention_us": round(t_att, 2),
                         "attention_tflops": round(fl / t_att / 1e6, 1),
                         "split_kv_decode_us": round(t_dec, 2),
                         "attention_picks": "pairs"})
            continue
        rng = np.random.default_rng(6)
        kc = torch.from_numpy(wl.random_e4m3_codes(rng, b.key_pages.shape)).to(device)
        vc = torch.from_numpy(wl.random_e4m3_codes(rng, b.value_pages.shape)).to(device)
        mcl = int(b.context_lens.max())
        ws8 = torch.empty(pa.pa_prefill_fp8_workspace_bytes(
            pa.make_shape(q.shape, kc.shape, bt.shape[1]), mcl), dtype=torch.uint8, device=device)
        t_fp8 = timeit(lambda: pa.pa_prefill_fp8(q, kc, vc, bt, cl, b.page_size, 0.05, 0.05,
                                                 scale=b.scale, causal=True, out=out,
                                                 max_context_len=mcl, workspace=ws8))
        del ws8
        rows.append({"shape": name, "items": items, "items_per_sm": round(items / sms, 2),
                     "gflop": round(fl / 1e9, 2),
                     "attention_us": round(t_att, 2),
                     "attention_tflops": round(fl / t_att / 1e6, 1),
                     "pairs_us": round(t_pairs, 2), "split_us": round(t_split, 2),
                     "pairs_tflops": round(fl / t_pairs / 1e6, 1),
                     "split_tflops": round(fl / t_split / 1e6, 1),
                     "fp8_pages_us": round(t_fp8, 2), "fp8_pages_tflops": round(fl / t_fp8 / 1e6, 1),
                     "attention_picks": ("split" if 2 * items < 3 * sms else
                                         "pairs, tail pieces" if items <= 2 * sms else "pairs")})
    st, flags = pa.pa_get_device_error()
    if st:
        raise RuntimeError(f"device error in the prefill shapes: {flags:#x}")
    return rows


def bench_prefill(pa, binding, torch, device, stream, steps=20, cpu_budget=6.0):
    """Chunked causal prefill (512 new rows after a ragged prefix): append of
    the 512 rows, then pa_attention (prefill route), timed with events."""
    b = wl.make_workload("prefill_chunk512")

    def to_dev(x):
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(np.ascontiguousarray(x)).to(device)

    kp, vp = to_dev(b.key_pages), to_dev(b.value_pages)
    q, bt, cl = to_dev(b.query), to_dev(b.block_table), to_dev(b.context_lens)
    kn, vn, sm = to_dev(b.key_new), to_dev(b.value_new), to_dev(b.slot_mapping)
    out = torch.empty_like(q)
    flush = torch.empty(int(2 * torch.cuda.get_device_properties(device).L2_cache_size),
                        dtype=torch.uint8, device=device)
    pa.pa_append_kv(kn, vn, kp, vp, sm, b.page_size)
    mcl = int(b.context_lens.max())

    def timed(attend, append=None):
        evs = []
        for k in range(steps + 3):
            flush.zero_()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record(stream)
            if append is None:
                pa.pa_append_kv(kn, vn, kp, vp, sm, b.page_size)
            else:
                append()
            e[1].record(stream)
            attend()
            e[2].record(stream)
            if k >= 3:
                evs.append(e)
        torch.cuda.synchronize()
        st, flags = pa.pa_get_device_error()
        if st:
            raise RuntimeError(f"device error in prefill bench: {flags:#x}")
        return (float(np.median([e[1].elapsed_time(e[2]) for e in evs])),
                float(np.median([e[0].elapsed_time(e[1]) for e in evs])))

    # The product path: pa_attention routes L = 512 to prefill; with 256
    # (request, head pair, query tile) items on 152 SMs it takes the pairs
    # kernel. Beside it, the split kernel forced through pa_prefill_split.
    att_ms, app_ms = timed(lambda: pa.pa_attention(q, kp, vp, bt, cl, b.page_size, scale=b.scale,
                                                   causal=True, out=out, max_context_len=mcl))
    split_ms, _ = timed(lambda: pa.pa_prefill_split(q, kp, vp, bt, cl, b.page_size, scale=b.scale,
                                                    causal=True, out=out))
    # The same call back to back, as the decode call is timed: blocks of
    # PREFILL_BLOCK calls with no events between them (each call's launch
    # overlaps the one before through programmatic dependent launch), over 4
    # rotating copies of the pools and queries (4 x 42 MB > L2), so each call
    # reads K/V and Q last touched three calls before; median of the blocks.
    copies = 4
    sets = [(kp, vp, q)] + [(kp.clone(), vp.clone(), q.clone()) for _ in range(copies - 1)]

    def attend(c):
        k_, v_, q_ = sets[c % copies]
        pa.pa_attention(q_, k_, v_, bt, cl, b.page_size, scale=b.scale, causal=True, out=out,
                        max_context_len=mcl)
    for c in range(2 * copies):
        attend(c)
    blocks = []
    for _ in range(PREFILL_BLOCKS):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for c in range(PREFILL_BLOCK):
            attend(c)
        e1.record(stream)
        blocks.append((e0, e1))
    torch.cuda.synchronize()
    st, flags = pa.pa_get_device_error()
    if st:
        raise RuntimeError(f"device error in prefill bench: {flags:#x}")
    block_ms = [x.elapsed_time(y) / PREFILL_BLOCK for x, y in blocks]
    call_ms = float(np.median(block_ms))
    del sets
    items = b.B * ((b.L + 127) // 128) * (b.H_q // 2)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    kernel = "prefill_split_kernel" if 2 * items < 3 * sms else "prefill_pairs_kernel"
    flops = prefill_flops(b)
    _, app_bytes = step_bytes(b)
    # The same chunk over e4m3 pools (seeded random codes, per-tensor scales):
    # the quantising append, then pa_prefill_fp8 (bf16 copies of the visible
    # tokens, then the same tensor-core kernel choice).
    rng = np.random.default_rng(b.seed + 9)
    kc = torch.from_numpy(wl.random_e4m3_codes(rng, b.key_pages.shape)).to(device)
    vc = torch.from_numpy(wl.random_e4m3_codes(rng, b.value_pages.shape)).to(device)
    ks, vs = 0.05, 0.05
    shape = pa.make_shape(q.shape, kc.shape, bt.shape[1])
    ws8 = torch.empty(pa.pa_prefill_fp8_workspace_bytes(shape, mcl), dtype=torch.uint8,
                      device=device)
    fp8_ms, fp8_app_ms = timed(
        lambda: pa.pa_prefill_fp8(q, kc, vc, bt, cl, b.page_size, ks, vs, scale=b.scale,
                                  causal=True, out=out, max_context_len=mcl, workspace=ws8),
        append=lambda: pa.pa_append_kv_fp8(kn, vn, kc, vc, sm, b.page_size, ks, vs))
    visible = int(b.context_lens.astype(np.int64).sum())
    copy_bytes = visible * b.H_kv * b.D * 2 * 3           # e4m3 read + bf16 write, K and V
    cpu = prefill_cpu_baseline(b, cpu_budget) if cpu_budget > 0 else None
    return {"workload": b.name, "tflops": round(flops / (call_ms * 1e-3) / 1e12, 3),
            "cpu_baseline": cpu,
            "attention_ms": round(call_ms, 4), "kernel": kernel, "items": items,
            "call_timing": f"{PREFILL_BLOCKS} blocks of {PREFILL_BLOCK} back-to-back pa_attention "
                           f"calls over {copies} rotating copies of pools and queries, events "
                           "around each block, median of the blocks",
            "call_blocks_ms": [round(x, 4) for x in block_ms],
            "flushed_single_call": {"attention_ms": round(att_ms, 4),
                                    "tflops": round(flops / (att_ms * 1e-3) / 1e12, 3),
                                    "timing": "2x L2 buffer written before each call, events "
                                              "around the call, median of the steps"},
            "split_kernel": {"attention_ms": round(split_ms, 4),
                             "tflops": round(flops / (split_ms * 1e-3) / 1e12, 3)},
            "append_ms": round(app_ms, 4),
            "append_gbs": round(app_bytes / (app_ms * 1e-3) / 1e9, 2),
            "causal_useful_flops": flops, "steps": steps,
            "l2": "2x L2 buffer written before every step (outside the events)",
            "fp8_pages": {"call": "pa_prefill_fp8 (e4m3 to bf16 page copy + " + kernel + ")",
                          "attention_ms": round(fp8_ms, 4),
                          "tflops": round(flops / (fp8_ms * 1e-3) / 1e12, 3),
                          "append_ms": round(fp8_app_ms, 4),
                          "copy_bytes": copy_bytes,
                          "over_bf16_ms": round(fp8_ms - att_ms, 4)}}


if __name__ == "__main__":
    sys.exit(main())
