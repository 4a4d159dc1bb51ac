#!/usr/bin/env python
"""Benchmark of the HiSparse decode hot path on GB300.

One step = one decode step of the "attention" workload (32 requests x 2
sparse layers, ctx 65536, top-K 2048, B 4096, 128 heads; 70% step-to-step
selection reuse, the rest uniform): for each layer, RESOLVE (page table + LRU
hot buffer + miss copies from pinned host memory) then sparse MLA decode
attention over the K resolved rows, then the step counter advances.  The step
is one hs_decode_step call: the later layers' RESOLVE runs on a copy stream
("precise prefetch"; bf16 rows: beside layer 0's RESOLVE, FP8 rows: after it,
beside layer 0's attention).  Per-kernel rooflines come from a
second timed pass of the same workload with the calls made one after another
on one stream (CUDA events around each launch).  Inputs (top-K traces,
queries) are resident in HBM before the timed region.

Prints one JSON line (rank 0).  Metric: resolved top-K rows/s (value) and
sparse-MLA decode tokens/s, with the dominant kernel's roofline fraction and
the CPU oracle timed on the host as a baseline.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl ours|reference]
Multi-GPU: launched by torchrun, one process per GPU, each an independent
replica over its own requests (weak scaling; no collective on the data path).
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth import workloads as W  # noqa: E402

METRIC = "resolved top-K rows/s + sparse-MLA decode tok/s (1 GB300); % HBM & host-link peak"
Q_DISTINCT = 64  # distinct decode queries cycled through (query values do not steer the work)


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 2000; the mixed workload: 120; spec: 200)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="attention",
                    choices=("attention", "resolve", "gather", "mixed", "spec"))
    ap.add_argument("--kv-format", choices=("bf16", "fp8"), default="bf16",
                    help="KV row format of the attention / resolve / gather workloads: bf16 "
                         "[576] (1152 B) or FP8 (656 B: E4M3 latent + 4 scales + bf16 rope)")
    ap.add_argument("--e2e-steps", type=int, default=400)
    ap.add_argument("--kernel-steps", type=int, default=500,
                    help="steps of the sequential per-kernel timing pass")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--profile", action="store_true",
                    help="small run for profilers: no clocks, no e2e, no CPU baseline")
    ap.add_argument("--no-extra", action="store_true",
                    help="attention workload: skip the resolve / gather workload records")
    ap.add_argument("--extra-steps", type=int, default=40,
                    help="timed steps of each extra workload record (after 3 warm-up steps)")
    ap.add_argument("--replica-check", action="store_true",
                    help="no GPU work: every replica reports its request range and a timing "
                         "through the same launch, barrier and max-over-ranks path")
    ap.add_argument("--cpu-baseline-child", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-units", default="0:8", help=argparse.SUPPRESS)
    return ap.parse_args(argv)


# ----------------------------------------------------------------- helpers

def replica_request_base(rank: int, requests_per_replica: int) -> int:
    """Generator id of a replica's first request: replicas serve disjoint
    requests (units are independent, so the path shards with no exchange)."""
    return rank * requests_per_replica


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The slowest rank's time (every rank gets it)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_rate(units_per_rank_step: int, steps: int, world: int, elapsed_ms: float) -> float:
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    return world * steps * units_per_rank_step / (elapsed_ms * 1e-3)


def dist_context(force_gloo=False):
    """(dist module or None, world, rank, local rank) of this process; the
    process group is created once per process (NCCL on GPUs, gloo on CPU)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch
        import torch.distributed as dist
        if not dist.is_initialized():
            backend = "nccl" if (torch.cuda.is_available() and not force_gloo) else "gloo"
            dist.init_process_group(backend)
    return dist, world, rank, local


def spawn_replicas(args, argv):
    """`--gpus N` (N > 1) outside torchrun: relaunch this script under
    torch.distributed.run, one process per GPU on this node (each an
    independent replica); returns its exit status."""
    import socket
    if not args.replica_check:
        import torch
        n = torch.cuda.device_count()
        if args.gpus > n:
            print(json.dumps({"error": f"--gpus {args.gpus} but {n} GPU(s) visible"}))
            return 2
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
           "--master-port", str(port), os.path.abspath(__file__), *argv]
    return subprocess.run(cmd).returncode


def run_replica_check(args):
    """Every replica takes its own requests (req_base = rank x R) of the
    workload and times a CPU stand-in for a step (generating its requests'
    first selections); rank 0 prints the ranges, world size and the slowest
    rank's time, through the same barrier / max-over-ranks path as the GPU
    arm."""
    dist, world, rank, _ = dist_context(force_gloo=True)
    w = W.make(args.workload)
    base = replica_request_base(rank, w.R)
    if dist is not None:
        dist.barrier()
    t0 = time.perf_counter()
    w2 = W.Workload(**{**w.__dict__, "steps": 1})
    w2.req_base = base
    rows = sum(int((w2.trace(r) >= 0).sum()) for r in range(min(w.R, 2)))
    ms = max_over_ranks((time.perf_counter() - t0) * 1e3, dist)
    ranges = [[base, base + w.R]]
    if dist is not None:
        got = [None] * world
        dist.all_gather_object(got, ranges[0])
        ranges = got
    if rank == 0:
        print(json.dumps({"replica_check": True, "n_gpus": world, "scaling": "weak",
                          "workload": workload_name(w), "requests_per_replica": w.R,
                          "replica_requests": ranges, "max_rank_ms": ms, "rows": rows}))
    if dist is not None:
        dist.destroy_process_group()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def _lines(self):
        try:
            with open(self.path) as f:
                return sum(1 for line in f if line.count(",") >= 8)
        except OSError:
            return 0

    def wait_ready(self, timeout_s=20.0):
        """Return once nvidia-smi writes samples: its start-up can take a second
        or more, and while it initialises the CUDA launches of the first timed
        steps ran up to ~10x slower.  A timed region of a few milliseconds holds
        no 100-ms sample of its own, so the record keeps the samples from here
        on (the warm-up runs next) together with those taken during the timed
        region."""
        t0 = time.time()
        while self.proc is not None and self._lines() < 2 and time.time() - t0 < timeout_s:
            time.sleep(0.05)
        time.sleep(0.2)

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "samples": len(sm), "reasons": sorted(reasons)}


def build_inputs(w, steps, threads=16):
    """Top-K traces [steps][L][R][K] and Q_DISTINCT queries [q][L][R][H][576]."""
    w2 = W.Workload(**{**w.__dict__, "steps": steps})
    topk = np.empty((steps, w.L, w.R, w.K), dtype=np.int32)

    def one(r):
        topk[:, :, r, :] = w2.trace(r)

    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(one, range(w.R)))
    q = np.empty((Q_DISTINCT, w.L, w.R, w.heads, W.ROW_ELEMS), dtype=np.uint16)
    for t in range(Q_DISTINCT):
        for l in range(w.L):
            for r in range(w.R):
                q[t, l, r] = synth.q(w.seed, w.req_base + r, l, t, w.heads)
    return topk, q


def row_bytes(fp8):
    return synth.FP8_ROW_BYTES if fp8 else W.ROW_BYTES


def make_pool(hs, w, scen, threads=16, fp8=False):
    """libhs pool at the workload's step-0 state (host pool filled, tail loaded)."""
    import torch
    cap = w.ctx_capacity()
    max_pages = int((cap.max() + w.P - 1) // w.P)
    resident = max(1, scen.blocks_per_layer - w.R * w.hot_blocks_per_request())
    pool = hs.Pool(w.R, w.L, w.K, w.B, w.P, W.ROW_ELEMS, max_pages, w.host_tokens(), resident,
                   hs.HS_KV_FP8 if fp8 else hs.HS_KV_BF16)
    offs = w.host_offsets()
    for l in range(w.L):
        for r in range(w.R):
            n = int(w.ctx[r])
            base = pool.host_pool[l, int(offs[r]):int(offs[r]) + n]
            if fp8:
                synth.rows_fp8_into(w.seed, w.req_base + r, l, 0, n, base.ctypes.data, threads)
            else:
                synth.rows_into(w.seed, w.req_base + r, l, 0, n, W.ROW_ELEMS, base.ctypes.data,
                                threads)
    stream = torch.cuda.current_stream()
    for r in range(w.R):
        hs.hs_set_request(pool.handle, r, int(w.ctx[r]), int(offs[r]), stream)
    for (r, page, blk) in scen.initial:
        hs.hs_load_page(pool.handle, r, page, blk, stream)
    torch.cuda.synchronize()
    return pool


def measure_h2d_peak(torch, nbytes=1 << 30, reps=10):
    """Pinned host -> device cudaMemcpyAsync bandwidth, best of `reps` (GB/s)."""
    src = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    best = 0.0
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        b.synchronize()
        best = max(best, nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
    del src, dst
    return best


def measure_d2h_peak(torch, nbytes=1 << 30, reps=10):
    """Device -> pinned host cudaMemcpyAsync bandwidth, best of `reps` (GB/s)."""
    src = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    dst = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    best = 0.0
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        b.synchronize()
        best = max(best, nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
    del src, dst
    return best


def pretouch_host_pool(torch, hs, pool):
    """Setup, before the warm-up: the GPU reads the whole host pool once
    (hs_pool_touch_host).  On some boxes the GPU's first read of each host page
    is slow (the step-0 fill took 13-17 ms against ~1 ms on others, and the
    following steps ran ~10x slower until the pages had been seen); this keeps
    that one-time cost out of the warm-up and the timed steps.  Returns the
    time taken (ms)."""
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    hs.hs_pool_touch_host(pool.handle)
    b.record()
    b.synchronize()
    return a.elapsed_time(b)


def measure_host_read_peak(torch, hs, pool, nbytes=1 << 30, reps=10):
    """Kernel reads of mapped pinned host memory -> device (GB/s), best of reps.
    Reads the pool's own host pool through the device alias libhs returns."""
    nbytes = min(nbytes, int(pool.raw.host_pool_bytes)) // 16 * 16
    dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    best = 0.0
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        hs.hs_host_read(int(pool.raw.host_pool_device), nbytes, dst)
        b.record()
        b.synchronize()
        best = max(best, nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
    del dst
    return best


def kernel_source_hash(name):
    path = os.path.join(ROOT, "sparse_attention_kv_hs_gb300", "csrc", name)
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def ncu_traffic(kernel_file, workload, fp8=False):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}{'_fp8' if fp8 else ''}.json")
    try:
        with open(path) as f:
            d = json.load(f)
        k = d[kernel_file]
        if k.get("source_sha256_16") != kernel_source_hash(kernel_file):
            return None
        return float(k["dram_bytes_per_launch"])
    except Exception:
        return None


# ----------------------------------------------------------------- CPU oracle

def oracle_sample(w, seconds, units=2, steps_cap=None, skip=0, fp8=False, unit0=0):
    """Run the CPU oracle (resolve + gather from host full KV + fp64 attention)
    over the first `units` (request, layer) units of the workload, step after
    step, for about `seconds` after `skip` untimed warm-up steps.  With fp8 the
    host KV is FP8 rows, decoded to their values by the oracle as they are
    gathered.  Returns (rows resolved, elapsed s, steps) of the timed steps."""
    import oracle
    scen = W.Scenario.build(w)
    o = oracle.ResolveOracle(w.R, w.L, w.K, w.B, w.P, w.ctx_capacity(), scen.blocks_per_layer)
    for r in range(w.R):
        o.set_ctx(r, int(w.ctx[r]))
        for i in range(w.hot_blocks_per_request()):
            o.set_hot_block(r, i, r * w.hot_blocks_per_request() + i)
    for (r, page, blk) in scen.initial:
        o.set_page(r, page, blk)
    sel = [(u // w.L, u % w.L) for u in range(unit0, unit0 + units)]
    reqs = sorted({r for r, _ in sel})
    steps = steps_cap or w.steps
    w2 = W.Workload(**{**w.__dict__, "steps": steps})
    tr = {r: w2.trace(r) for r in reqs}
    gen = synth.rows_fp8 if fp8 else synth.rows
    full = {(r, l): gen(w.seed, w.req_base + r, l, 0, int(w.ctx[r]), threads=8)
            for (r, l) in sel}  # the host's full KV of the sampled units (not timed)
    qs = {(r, l): synth.q(w.seed, w.req_base + r, l, 0, w.heads) for (r, l) in sel}
    rows_done, t0, t = 0, time.perf_counter(), 0
    while t < steps:
        if t == skip:  # warm-up over: start the clock
            rows_done, t0 = 0, time.perf_counter()
        for (r, l) in sel:
            rows, _, _ = o.resolve(l, r, tr[r][t, l], t)
            gathered = full[(r, l)][tr[r][t, l]]          # rows at the selected positions
            if fp8:
                gathered = oracle.fp8_rows_to_f64(gathered)
            oracle.sparse_mla_decode(qs[(r, l)], gathered, rows >= 0, W.SCALE)
            rows_done += w.K
        t += 1
        if t > skip and time.perf_counter() - t0 >= seconds:
            break
    return rows_done, time.perf_counter() - t0, t - min(skip, t)


def cpu_baseline(w, seconds, fp8=False, units=8):
    """The oracle timed on the host: `units` (request, layer) units, one child
    process per unit, all at once (units are independent; each child's BLAS
    gets an equal share of the cores), for about `seconds`; value = all rows
    over the slowest child's time.  `value_1_thread`: one unit on one thread."""
    cores = os.cpu_count() or 1
    procs = min(units, cores)
    per = max(1, cores // procs)

    def launch(u0, n, threads, secs):
        env = dict(os.environ, OPENBLAS_NUM_THREADS=str(threads), OMP_NUM_THREADS=str(threads),
                   MKL_NUM_THREADS=str(threads))
        cmd = [sys.executable, os.path.abspath(__file__), "--cpu-baseline-child",
               "--workload", w.name, "--cpu-seconds", str(secs), "--cpu-units", f"{u0}:{u0 + n}",
               "--kv-format", "fp8" if fp8 else "bf16"]
        return subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True,
                                env=env)

    def collect(p):
        try:
            out, err = p.communicate(timeout=600)
            return json.loads(out.strip().splitlines()[-1]), None
        except Exception as e:
            return None, str(e)[-200:]

    spans = [(i * units // procs, (i + 1) * units // procs - i * units // procs)
             for i in range(procs)]
    children = [launch(u0, n, per, seconds) for u0, n in spans]
    res = [collect(p) for p in children]
    if any(d is None for d, _ in res):
        err = next(e for d, e in res if d is None)
        return {"value": None, "unit": "rows/s", "cores": cores, "kind": "oracle",
                "sample": f"failed: {err}"}
    rows = sum(d["rows"] for d, _ in res)
    secs = max(d["secs"] for d, _ in res)
    steps = min(d["steps"] for d, _ in res)
    d1, _ = collect(launch(0, 1, 1, max(seconds / 3, 1.0)))
    return {"value": rows / secs, "unit": "rows/s", "kind": "oracle", "cores": procs * per,
            "sample": f"{units} (request, layer) units in {procs} processes x {per} BLAS "
                      f"threads, >= {steps} steps each (resolve + gather + fp64 attention), "
                      f"{secs:.1f} s",
            "value_1_thread": d1["rows"] / d1["secs"] if d1 else None}


# ----------------------------------------------------------------- GPU arm

def run_ours(args):
    """Measure one workload; returns rank 0's JSON line (None on other ranks)."""
    import torch
    import sparse_attention_kv_hs_gb300 as hs

    dist, world, rank, local = dist_context()
    torch.cuda.set_device(local)
    lib = hs.load()

    w = W.make(args.workload)
    w.req_base = replica_request_base(rank, w.R)
    attention = args.workload == "attention"
    fp8 = args.kv_format == "fp8"
    rb = row_bytes(fp8)
    kern_steps = min(args.kernel_steps, args.steps) if attention else 0
    steps_total = args.warmup + args.steps + kern_steps
    topk_h, q_h = build_inputs(w, steps_total)
    scen = W.Scenario.build(w)
    pool = make_pool(hs, w, scen, fp8=fp8)
    R, L, K, H = w.R, w.L, w.K, w.heads
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream

    topk_d = torch.from_numpy(topk_h).to(dev)
    q_d = torch.from_numpy(q_h.view(np.int16)).to(dev)
    rows_d = torch.empty((L, R, K), dtype=torch.int32, device=dev)
    out_d = torch.empty((L, R, H, W.V_DIM), dtype=torch.bfloat16, device=dev)
    lse_d = torch.empty((L, R, H), dtype=torch.float32, device=dev)
    cnt_d = torch.zeros((steps_total, L, R), dtype=torch.int32, device=dev)
    copy_stream = torch.cuda.Stream(device=dev) if attention else None
    gather_d = None if attention else torch.empty((R * K, rb // 2), dtype=torch.int16, device=dev)
    ph = pool.handle
    step_ptr = pool.step.data_ptr()
    tk_base, tk_stride_t, tk_stride_l = topk_d.data_ptr(), L * R * K * 4, R * K * 4
    q_base, q_stride_t, q_stride_l = q_d.data_ptr(), L * R * H * W.ROW_ELEMS * 2, R * H * W.ROW_ELEMS * 2
    rows_ptr = [rows_d[l].data_ptr() for l in range(L)]
    out_ptr = [out_d[l].data_ptr() for l in range(L)]
    lse_ptr = [lse_d[l].data_ptr() for l in range(L)]
    cnt_base = cnt_d.data_ptr()
    splits = None

    def one_step(t, ev=None):
        for l in range(L):
            if ev is not None:
                ev[0][l].record(stream)
            st = lib.hs_resolve(ph, l, 1, tk_base + t * tk_stride_t + l * tk_stride_l, step_ptr,
                                rows_ptr[l], cnt_base + (t * L + l) * R * 4, None, sptr)
            if ev is not None:
                ev[1][l].record(stream)
            if attention:
                st |= lib.hs_sparse_mla_decode(ph, l, q_base + (t % Q_DISTINCT) * q_stride_t +
                                               l * q_stride_l, rows_ptr[l], H, W.V_DIM, W.SCALE,
                                               out_ptr[l], lse_ptr[l], sptr)
            else:
                st |= lib.hs_gather(ph, l, rows_ptr[l], R * K, gather_d.data_ptr(), sptr)
            if ev is not None:
                ev[2][l].record(stream)
            if st != 0:
                raise RuntimeError(f"libhs call failed at step {t}: {hs.status_string(st)}")
        lib.hs_step_advance(step_ptr, sptr)

    def fused_step(t, ev=None):
        """One hs_decode_step call (the later layers' RESOLVE on the copy stream)."""
        st = lib.hs_decode_step(ph, 0, L, tk_base + t * tk_stride_t,
                                q_base + (t % Q_DISTINCT) * q_stride_t, H, W.V_DIM, W.SCALE,
                                step_ptr, rows_d.data_ptr(), out_d.data_ptr(), lse_d.data_ptr(),
                                cnt_base + t * L * R * 4, sptr, copy_stream.cuda_stream)
        if st != 0:
            raise RuntimeError(f"hs_decode_step failed at step {t}: {hs.status_string(st)}")
        lib.hs_step_advance(step_ptr, sptr)

    step_fn = fused_step if attention else one_step

    peaks = load_peaks()
    h2d_peak = measure_h2d_peak(torch) if not args.profile else float("nan")
    host_read_peak = measure_host_read_peak(torch, hs, pool) if not args.profile else float("nan")

    # step 0 is the cold step (empty hot buffers): timed on its own, then warm-up.
    # First every kernel of the step is launched once without touching the
    # pool's state (attention over padding rows, a scratch step counter), so
    # that module loading is not counted.
    scratch_step = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.hs_step_advance(scratch_step.data_ptr(), sptr)
    if attention:
        pad = torch.full((R, K), -1, dtype=torch.int32, device=dev)
        for l in range(L):
            st = lib.hs_sparse_mla_decode(ph, l, q_base + l * q_stride_l, pad.data_ptr(), H,
                                          W.V_DIM, W.SCALE, out_ptr[l], lse_ptr[l], sptr)
            if st != 0:
                raise RuntimeError(f"pre-load attention failed: {hs.status_string(st)}")
    else:
        pad = torch.full((R * K,), -1, dtype=torch.int32, device=dev)
        if lib.hs_gather(ph, 0, pad.data_ptr(), R * K, gather_d.data_ptr(), sptr) != 0:
            raise RuntimeError("pre-load gather failed")
    pretouch_ms = pretouch_host_pool(torch, hs, pool)
    # The clock sampler starts, and the timing events are made, before the cold
    # step and the warm-up, so that the timed region follows the warm-up with
    # no more idle time than its synchronize: after an idle spell of a
    # millisecond or more, the first steps measured 0.5-1.0 ms (then 0.3-0.4)
    # against 0.27 ms in steady state.
    clocks = ClockSampler(local) if not args.profile else None
    if clocks:
        clocks.start()
        clocks.wait_ready()
    # sequential steps timed launch by launch: the main region itself for the
    # gather / resolve workloads, a second pass after it for the attention one
    n_ev = args.steps if not attention else kern_steps
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(L)] for _ in range(3)]
           for _ in range(n_ev)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    step_fn(0)
    c1.record(stream)
    for t in range(1, args.warmup):
        step_fn(t)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        step_fn(args.warmup + i, None if attention else evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    clock_info = clocks.stop() if clocks else None
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), dist, dev)
    cold_ms = c0.elapsed_time(c1) if args.warmup > 0 else None
    cold_misses = int(cnt_d[0].sum().item()) if args.warmup > 0 else None
    misses_main = int(cnt_d[args.warmup:args.warmup + args.steps].sum().item())
    k0 = args.warmup + args.steps if attention else args.warmup
    if attention:
        for i in range(kern_steps):
            one_step(k0 + i, evs[i])
        torch.cuda.synchronize()
    res_ms = sum(e[0][l].elapsed_time(e[1][l]) for e in evs for l in range(L))
    att_ms = sum(e[1][l].elapsed_time(e[2][l]) for e in evs for l in range(L))
    # the link again after the timed work: the host memory behind it is shared
    # with other jobs, so a congested spell shows as a drop here
    h2d_peak_after = measure_h2d_peak(torch) if not args.profile else float("nan")
    errs = hs.hs_check_errors(ph)
    if errs:
        raise RuntimeError(f"device error word set: {errs}")
    misses = int(cnt_d[k0:k0 + n_ev].sum().item())

    rows_per_step = L * R * K
    value = weak_scaling_rate(rows_per_step, args.steps, world, elapsed_ms)
    tok_s = weak_scaling_rate(R, args.steps, world, elapsed_ms)
    n_launch_res = max(n_ev, 1) * L
    res_avg_s = res_ms * 1e-3 / n_launch_res
    att_avg_s = att_ms * 1e-3 / n_launch_res
    miss_bytes_per_launch = misses * rb / n_launch_res
    # RESOLVE: the miss rows cross the host link (read) and land in HBM
    resolve_roof = {
        "kernel": "resolve_kernel", "bound": "host_link",
        "achieved": miss_bytes_per_launch / res_avg_s / 1e9, "peak": h2d_peak, "unit": "GB/s",
        "peak_source": "in-run pinned cudaMemcpyAsync H2D, 1 GiB, best of 10",
        "frac": miss_bytes_per_launch / res_avg_s / 1e9 / h2d_peak,
        "traffic": ncu_traffic("resolve.cu", args.workload, fp8),
        "avg_launch_us": res_avg_s * 1e6, "miss_rows_per_launch": misses / n_launch_res,
    }
    if attention:
        # rows read once + q read + bf16 out written + row ids, per request
        att_bytes = R * (K * rb + H * W.ROW_ELEMS * 2 + H * W.V_DIM * 2 + K * 4)
        att_flops = R * 2.0 * H * K * (W.ROW_ELEMS + W.V_DIM)
        att_roof = {
            "kernel": "mla_decode_kernel (+ split merge)", "bound": "hbm",
            "achieved": att_bytes / att_avg_s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": att_bytes / att_avg_s / 1e9 / peaks["hbm_gbs"],
            "traffic": ncu_traffic("mla_decode.cu", args.workload, fp8),
            "avg_launch_us": att_avg_s * 1e6,
            "tensor_tflops": att_flops / att_avg_s / 1e12,
            "tensor_frac_of_burst_peak": att_flops / att_avg_s / 1e12 / peaks["bf16_tflops"],
        }
    else:
        g_bytes = R * K * (2 * rb + 4)
        att_roof = {
            "kernel": "gather_rows_kernel", "bound": "hbm",
            "achieved": g_bytes / att_avg_s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": g_bytes / att_avg_s / 1e9 / peaks["hbm_gbs"],
            "traffic": ncu_traffic("gather.cu", args.workload, fp8),
            "avg_launch_us": att_avg_s * 1e6,
        }
    dominant = resolve_roof if res_ms >= att_ms else att_roof
    gpu_launches = args.steps * (2 * L + 1)  # RESOLVE + attention (or gather) per layer, step
    if attention:  # + the split merge of each attention launch with more than one K split
        gpu_launches += args.steps * sum(1 for s in decode_step_splits(pool, R, K, L) if s > 1)

    # ---- end to end: host buffers, H2D of the step's inputs, D2H of its outputs
    e2e = None
    if not args.no_e2e and not args.profile:
        e2e = run_e2e(torch, hs, lib, pool, w, topk_h, q_h, args, stream, dev, dist, world)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "fp8-e4m3 rows, fp16 MMA operands" if fp8 else "bf16",
            "data": "synthetic (seeded generator; no dataset)",
            "config": {"workload": workload_name(w), "requests_per_gpu": R, "sparse_layers": L,
                       "kv_rows": kv_rows_name(fp8),
                       "context": int(w.ctx[0]), "top_k": K, "hot_slots": B_of(w),
                       "heads": H if attention else None, "selection": "70% reuse + 30% uniform"
                       if attention else "70/20/10 drift, layers share 80%",
                       "l2": "inputs larger than L2 (per-step unique KV > 129 MB; host pool "
                             f"{w.host_bytes() / 1e9:.1f} GB), no flush",
                       "parallelism": f"replicas x{world}"},
            "decode_tok_s": tok_s if attention else None,
            "miss_rows_per_step": misses_main / args.steps,
            "cold_step": {"ms": cold_ms, "miss_rows": cold_misses,
                          "note": "step 0 (empty hot buffers), before the warm-up; not in value"},
            "host_pool_pretouch_ms": pretouch_ms,
            "schedule": ("hs_decode_step: the later layers' RESOLVE on a copy stream "
                         + ("after layer 0's RESOLVE, beside its attention" if fp8 else
                            "beside layer 0's RESOLVE")
                         + f"; per-kernel rooflines from a sequential pass of {n_ev} steps")
            if attention else "sequential, one stream",
            "roofline": dominant,
            "kernels": [resolve_roof, att_roof],
            "host_link_peak_gbs": h2d_peak,
            "host_link_peak_after_gbs": h2d_peak_after,
            "host_kernel_read_peak_gbs": host_read_peak,
            "peaks": peaks,
            "e2e": e2e,
            "gpu_launches": gpu_launches,
            "clocks": clock_info,
        }
        if not args.no_cpu_baseline and not args.profile and world == 1:
            line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds, fp8)
    pool.close()
    return line if rank == 0 else None


def extra_workloads(args):
    """The resolve and gather workloads at full size, measured in the same run
    after the attention workload: their rows/s and per-launch rooflines
    (RESOLVE against the in-run host link peak, the standalone gather against
    HBM), so the hit/gather-path and miss-path targets are in the same line."""
    import copy
    out = {}
    for name in ("resolve", "gather"):
        a2 = copy.copy(args)
        a2.workload, a2.steps, a2.warmup = name, args.extra_steps, 3
        a2.no_e2e, a2.no_cpu_baseline = True, True
        rec = run_ours(a2)
        if rec is not None:
            out[name] = {k: rec[k] for k in ("value", "unit", "ms_per_step", "steps",
                                                "miss_rows_per_step", "cold_step", "kernels",
                                                "host_link_peak_gbs", "clocks", "gpu_launches")}
            out[name]["workload"] = rec["config"]["workload"]
    return out


def pool_splits(pool, R, K):
    sms = __import__("torch").cuda.get_device_properties(0).multi_processor_count
    tiles = (K + 63) // 64
    return max(1, min(tiles, sms // (2 * R)))


def decode_step_splits(pool, R, K, L, T=1):
    """K splits of each attention launch of one hs_decode_step(_tokens) (the
    library's rule: a launch beside a RESOLVE gets the SMs RESOLVE's clusters
    leave; R x T decode rows per launch)."""
    sms = __import__("torch").cuda.get_device_properties(0).multi_processor_count
    full = pool_splits(pool, R * T, K)
    c_side = 2 if 3 * R <= sms else 1
    s_side = max(1, (sms - c_side * R) // (2 * R * T))
    return [min(full, s_side) if l + 1 < L else full for l in range(L)]


def B_of(w):
    return w.B


def kv_rows_name(fp8):
    return ("FP8: 512 E4M3 + 4 fp32 scales + 64 bf16 rope (656 B)" if fp8
            else "bf16 [576] (1152 B)")


def workload_name(w):
    return (f"{w.name}: {w.R} requests x {w.L} sparse layers, ctx {int(w.ctx[0])}, "
            f"top-K {w.K}, B {w.B}" + (f", {w.heads} heads" if w.name == "attention" else ""))


def run_mixed(args):
    """The mixed-residency workload (128 requests x 1 sparse layer, contexts
    log-uniform in [16384, 1048576], a quarter zero-residency and a quarter
    fully resident, the rest with a 4096-token tail; K 2048, B 4096).  One step:
    the page-table flips due at its boundary (committing the host copies queued
    a step earlier), RESOLVE, the step counter, then ~6 requests each append a
    finished 256-token page -- its rows are written into a resident block (the
    stand-in for the model writing KV), mapped, queued for host offload on a
    side stream, and the context grows.  Metric: resolved rows/s over the whole
    step; the offload copies are timed on the side stream."""
    import torch
    import sparse_attention_kv_hs_gb300 as hs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    lib = hs.load()
    steps_total = args.warmup + args.steps
    w = W.make("mixed", steps=steps_total)
    w.req_base = replica_request_base(rank, w.R)
    scen = W.Scenario.build(w)
    R, L, K, P = w.R, w.L, w.K, w.P
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream(device=dev)
    sptr = stream.cuda_stream
    topk = np.empty((steps_total, L, R, K), dtype=np.int32)
    with cf.ThreadPoolExecutor(max_workers=16) as ex:
        def one(r):
            topk[:, :, r, :] = w.trace(r)
        list(ex.map(one, range(R)))
    fp8 = args.kv_format == "fp8"
    rb = row_bytes(fp8)
    pool = make_pool(hs, w, scen, fp8=fp8)
    # rows of every page appended during the run, generated up front (device)
    app = [(t, r, page, blk) for t in range(steps_total) for (r, page, blk) in scen.appends[t]]
    app_rows = torch.empty((len(app), L, P, rb // 2), dtype=torch.int16, device=dev)
    gen = synth.rows_fp8 if fp8 else synth.rows
    for i, (t, r, page, blk) in enumerate(app):
        rows = np.stack([gen(w.seed, w.req_base + r, l, page * P, P, threads=8)
                         for l in range(L)])
        app_rows[i].copy_(torch.from_numpy(rows.view(np.int16)))
    topk_d = torch.from_numpy(topk).to(dev)
    rows_d = torch.empty((R, K), dtype=torch.int32, device=dev)
    cnt_d = torch.zeros((steps_total, R), dtype=torch.int32, device=dev)
    offs = w.host_offsets()
    ctx = w.ctx.astype(np.int64).copy()
    ph = pool.handle
    step_ptr = pool.step.data_ptr()
    # one offload launch per step (all of the step's completed pages)
    ev_go = [torch.cuda.Event() for _ in range(steps_total)]
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(steps_total)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(steps_total)]
    for e in ev_b:  # torch creates events lazily; the library is handed raw handles
        e.record(side)
    torch.cuda.synchronize()
    pending = {}
    launches = [0]

    def call(st, what):
        if st != 0:
            raise RuntimeError(f"{what} failed: {hs.status_string(st)}")

    def one_step(t, ev_res=None):
        for (r, page, blk) in scen.flips[t]:
            i = pending.pop((r, page), None)
            if i is not None:
                call(lib.hs_commit_offload(ph, r, page, sptr, ev_b[i].cuda_event), "commit")
            else:
                call(lib.hs_map_page(ph, r, page, -1, sptr), "map_page")
            launches[0] += 1
        if ev_res is not None:
            ev_res[0].record(stream)
        call(lib.hs_resolve(ph, 0, 1, topk_d[t].data_ptr(), step_ptr, rows_d.data_ptr(),
                            cnt_d[t].data_ptr(), None, sptr), "resolve")
        if ev_res is not None:
            ev_res[1].record(stream)
        lib.hs_step_advance(step_ptr, sptr)
        launches[0] += 2
        apps = scen.appends[t]
        for (r, page, blk) in apps:
            i = app_index[(t, r, page)]
            pool.kv_pool[0:L, blk * P:(blk + 1) * P].copy_(app_rows[i])  # model writes the page
            call(lib.hs_map_page(ph, r, page, blk, sptr), "map_page")
            pending[(r, page)] = t
            ctx[r] += P
            call(lib.hs_set_request(ph, r, int(ctx[r]), int(offs[r]), sptr), "set_request")
            launches[0] += 2  # map, set_request (the page copy is a memcpy)
        if apps:  # the step's completed pages -> host, one launch on the side stream
            ev_go[t].record(stream)
            side.wait_event(ev_go[t])
            ev_a[t].record(side)
            reqs = (ctypes.c_int32 * len(apps))(*[a[0] for a in apps])
            pages = (ctypes.c_int32 * len(apps))(*[a[1] for a in apps])
            call(lib.hs_offload_pages(ph, len(apps), ctypes.addressof(reqs), ctypes.addressof(pages),
                                      sptr, side.cuda_stream, ev_b[t].cuda_event), "offload")
            launches[0] += 1

    app_index = {(t, r, page): i for i, (t, r, page, blk) in enumerate(app)}
    h2d_peak = measure_h2d_peak(torch) if not args.profile else float("nan")
    d2h_peak = measure_d2h_peak(torch) if not args.profile else float("nan")
    pretouch_ms = pretouch_host_pool(torch, hs, pool)
    # sampler and events before the warm-up: the timed region follows it with
    # no idle time beyond its synchronize (see run_ours)
    clocks = ClockSampler(local) if not args.profile else None
    if clocks:
        clocks.start()
        clocks.wait_ready()
    evr = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for t in range(args.warmup):
        one_step(t)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    launches[0] = 0
    off_steps = [t for t in range(args.warmup, steps_total) if scen.appends[t]]
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        one_step(args.warmup + i, evr[i])
    stream.wait_stream(side)  # the step's offload copies are part of the work
    t_end.record(stream)
    torch.cuda.synchronize()
    clock_info = clocks.stop() if clocks else None
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), dist, dev)
    if hs.hs_check_errors(ph):
        raise RuntimeError("device error word set in the mixed run")
    res_ms = sum(e[0].elapsed_time(e[1]) for e in evr)
    off_ms = [ev_a[t].elapsed_time(ev_b[t]) for t in off_steps]
    misses = int(cnt_d[args.warmup:].sum().item())
    res_avg_s = res_ms * 1e-3 / args.steps
    miss_bytes = misses * rb / args.steps
    page_bytes = L * P * rb
    off_bytes = page_bytes * sum(len(scen.appends[t]) for t in off_steps) / max(len(off_steps), 1)
    off_avg_s = (sum(off_ms) / max(len(off_ms), 1)) * 1e-3
    resolve_roof = {
        "kernel": "resolve_kernel", "bound": "host_link",
        "achieved": miss_bytes / res_avg_s / 1e9, "peak": h2d_peak, "unit": "GB/s",
        "peak_source": "in-run pinned cudaMemcpyAsync H2D, 1 GiB, best of 10",
        "frac": miss_bytes / res_avg_s / 1e9 / h2d_peak,
        "traffic": ncu_traffic("resolve.cu", "mixed", fp8), "avg_launch_us": res_avg_s * 1e6,
        "miss_rows_per_launch": misses / args.steps,
    }
    off_roof = {
        "kernel": "offload_pages_kernel", "bound": "host_link",
        "achieved": off_bytes / off_avg_s / 1e9 if off_ms else None, "peak": d2h_peak,
        "unit": "GB/s", "peak_source": "in-run pinned cudaMemcpyAsync D2H, 1 GiB, best of 10",
        "frac": off_bytes / off_avg_s / 1e9 / d2h_peak if off_ms else None,
        "traffic": None, "avg_launch_us": off_avg_s * 1e6, "launches": len(off_ms),
        "bytes_per_launch": off_bytes, "pages_per_launch": off_bytes / page_bytes,
    }
    if rank == 0:
        line = {
            "metric": METRIC, "value": weak_scaling_rate(R * K * L, args.steps, world, elapsed_ms),
            "unit": "rows/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "host_pool_pretouch_ms": pretouch_ms,
            "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp8-e4m3 rows (moved as bytes)" if fp8 else "bf16",
            "data": "synthetic (seeded generator; no dataset)",
            "config": {"kv_rows": kv_rows_name(fp8), "workload": (f"mixed: {R} requests x {L} sparse layer, ctx log-uniform "
                                    f"16384..1048576, top-K {K}, B {w.B}, tail 4096; a quarter "
                                    "zero-residency, a quarter fully resident; "
                                    f"{w.appends_per_step} page appends + offloads per step"),
                       "host_pool_gb": round(w.host_bytes() / 1e9, 1),
                       "l2": "inputs larger than L2 (host pool and per-step misses), no flush",
                       "parallelism": f"replicas x{world}"},
            "miss_rows_per_step": misses / args.steps,
            "roofline": resolve_roof,
            "kernels": [resolve_roof, off_roof],
            "host_link_peak_gbs": h2d_peak, "host_link_d2h_peak_gbs": d2h_peak,
            "e2e": None, "gpu_launches": launches[0], "clocks": clock_info,
        }
        print(json.dumps(line))
    pool.close()
    if dist is not None:
        dist.destroy_process_group()


def run_spec(args):
    """The speculative-decoding workload: the attention workload's 32 requests
    x 2 layers (ctx 65536, K 2048) with T = 2 verify tokens per request and
    step and B = (T + 2) K = 8192.  One step is one hs_decode_step_tokens call
    (per layer: RESOLVE of the request's T lists as one, then one decode per
    verify token; the later layers' RESOLVE on a copy stream), then the step
    counter.  Per-kernel rooflines come from a second pass in which
    hs_resolve_tokens and hs_sparse_mla_decode_tokens run one after another on
    one stream.  Metric: resolved rows/s (R x L x T x K per step); verify
    tokens/s alongside."""
    import torch
    import sparse_attention_kv_hs_gb300 as hs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    lib = hs.load()
    kern_steps = min(args.kernel_steps, args.steps)
    steps_total = args.warmup + args.steps + kern_steps
    w = W.make("spec", steps=steps_total)
    w.req_base = replica_request_base(rank, w.R)
    R, L, K, T, H = w.R, w.L, w.K, w.tokens, w.heads
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    topk = np.empty((steps_total, L, R, T, K), dtype=np.int32)
    with cf.ThreadPoolExecutor(max_workers=16) as ex:
        def one(r):
            topk[:, :, r] = w.trace_tokens(r)
        list(ex.map(one, range(R)))
    q = np.empty((Q_DISTINCT, L, R, T, H, W.ROW_ELEMS), dtype=np.uint16)
    for t in range(Q_DISTINCT):
        for l in range(L):
            for r in range(R):
                for k in range(T):
                    q[t, l, r, k] = synth.q(w.seed, w.req_base + r, l, t * T + k, H)
    scen = W.Scenario.build(w)
    fp8 = args.kv_format == "fp8"
    rb = row_bytes(fp8)
    pool = make_pool(hs, w, scen, fp8=fp8)
    topk_d = torch.from_numpy(topk).to(dev)
    q_d = torch.from_numpy(q.view(np.int16)).to(dev)
    rows_d = torch.empty((L, R, T, K), dtype=torch.int32, device=dev)
    out_d = torch.empty((L, R, T, H, W.V_DIM), dtype=torch.bfloat16, device=dev)
    lse_d = torch.empty((L, R, T, H), dtype=torch.float32, device=dev)
    cnt_d = torch.zeros((steps_total, L, R), dtype=torch.int32, device=dev)
    ph, step_ptr = pool.handle, pool.step.data_ptr()
    copy_stream = torch.cuda.Stream(device=dev)

    def fused_step(t):
        st = lib.hs_decode_step_tokens(ph, 0, L, T, topk_d[t].data_ptr(),
                                       q_d[t % Q_DISTINCT].data_ptr(), H, W.V_DIM, W.SCALE,
                                       step_ptr, rows_d.data_ptr(), out_d.data_ptr(),
                                       lse_d.data_ptr(), cnt_d[t].data_ptr(), sptr,
                                       copy_stream.cuda_stream)
        if st != 0:
            raise RuntimeError(f"hs_decode_step_tokens failed at step {t}: {hs.status_string(st)}")
        lib.hs_step_advance(step_ptr, sptr)

    def one_step(t, ev=None):
        for l in range(L):
            if ev is not None:
                ev[0][l].record(stream)
            st = lib.hs_resolve_tokens(ph, l, 1, T, topk_d[t, l].data_ptr(), step_ptr,
                                       rows_d[l].data_ptr(), cnt_d[t, l].data_ptr(), None, sptr)
            if ev is not None:
                ev[1][l].record(stream)
            st |= lib.hs_sparse_mla_decode_tokens(ph, l, T, q_d[t % Q_DISTINCT, l].data_ptr(),
                                                  rows_d[l].data_ptr(), H, W.V_DIM, W.SCALE,
                                                  out_d[l].data_ptr(), lse_d[l].data_ptr(), sptr)
            if ev is not None:
                ev[2][l].record(stream)
            if st != 0:
                raise RuntimeError(f"libhs call failed at step {t}: {hs.status_string(st)}")
        lib.hs_step_advance(step_ptr, sptr)

    peaks = load_peaks()
    h2d_peak = measure_h2d_peak(torch) if not args.profile else float("nan")
    pretouch_ms = pretouch_host_pool(torch, hs, pool)
    # sampler and events before the warm-up: the timed region follows it with
    # no idle time beyond its synchronize (see run_ours)
    clocks = ClockSampler(local) if not args.profile else None
    if clocks:
        clocks.start()
        clocks.wait_ready()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for t in range(args.warmup):
        fused_step(t)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        fused_step(args.warmup + i)
    t_end.record(stream)
    torch.cuda.synchronize()
    clock_info = clocks.stop() if clocks else None
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), dist, dev)
    misses_main = int(cnt_d[args.warmup:args.warmup + args.steps].sum().item())
    # per-kernel pass: the two calls one after another on one stream
    k0 = args.warmup + args.steps
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(L)] for _ in range(3)]
           for _ in range(kern_steps)]
    for i in range(kern_steps):
        one_step(k0 + i, evs[i])
    torch.cuda.synchronize()
    if hs.hs_check_errors(ph):
        raise RuntimeError("device error word set in the spec run")
    n_launch = kern_steps * L
    res_s = sum(e[0][l].elapsed_time(e[1][l]) for e in evs for l in range(L)) * 1e-3 / n_launch
    att_s = sum(e[1][l].elapsed_time(e[2][l]) for e in evs for l in range(L)) * 1e-3 / n_launch
    misses = int(cnt_d[k0:].sum().item())
    miss_bytes = misses * rb / n_launch
    n_rows = R * T  # decode rows of one attention launch
    att_bytes = n_rows * (K * rb + H * W.ROW_ELEMS * 2 + H * W.V_DIM * 2 + K * 4)
    resolve_roof = {
        "kernel": "resolve_kernel (T = 2 verify tokens)", "bound": "host_link",
        "achieved": miss_bytes / res_s / 1e9, "peak": h2d_peak, "unit": "GB/s",
        "peak_source": "in-run pinned cudaMemcpyAsync H2D, 1 GiB, best of 10",
        "frac": miss_bytes / res_s / 1e9 / h2d_peak, "traffic": None,
        "avg_launch_us": res_s * 1e6, "miss_rows_per_launch": misses / n_launch,
    }
    att_roof = {
        "kernel": "mla_decode_kernel (64 decode rows)", "bound": "hbm",
        "achieved": att_bytes / att_s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
        "frac": att_bytes / att_s / 1e9 / peaks["hbm_gbs"], "traffic": None,
        "avg_launch_us": att_s * 1e6,
    }
    if rank == 0:
        line = {
            "metric": METRIC, "value": weak_scaling_rate(R * L * T * K, args.steps, world, elapsed_ms),
            "unit": "rows/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "host_pool_pretouch_ms": pretouch_ms,
            "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp8-e4m3 rows, fp16 MMA operands" if fp8 else "bf16",
            "data": "synthetic (seeded generator; no dataset)",
            "config": {"kv_rows": kv_rows_name(fp8), "workload": (f"spec: {R} requests x {L} sparse layers, ctx {int(w.ctx[0])}, "
                                    f"top-K {K}, {T} verify tokens, B {w.B}, {H} heads"),
                       "l2": "inputs larger than L2, no flush", "parallelism": f"replicas x{world}"},
            "verify_tok_s": weak_scaling_rate(R * T, args.steps, world, elapsed_ms),
            "miss_rows_per_step": misses_main / args.steps,
            "schedule": ("hs_decode_step_tokens: the later layers' RESOLVE on a copy stream; "
                         "per-kernel rooflines from a sequential pass of "
                         f"{kern_steps} steps"),
            "roofline": resolve_roof if res_s >= att_s else att_roof,
            "kernels": [resolve_roof, att_roof], "host_link_peak_gbs": h2d_peak, "peaks": peaks,
            "e2e": None, "clocks": clock_info,
            "gpu_launches": args.steps * (2 * L + 1 + sum(
                1 for sp in decode_step_splits(pool, R, K, L, T) if sp > 1)),
        }
        print(json.dumps(line))
    pool.close()
    if dist is not None:
        dist.destroy_process_group()


def run_e2e(torch, hs, lib, pool, w, topk_h, q_h, args, stream, dev, dist, world):
    """Same step through the C ABI with HOST inputs/outputs: each step copies its
    top-K rows and queries from pinned host memory and reads the attention
    output (and lse) back; copies are inside the timed region.  A step's inputs
    are copied after the previous step (a decode step's inputs come from the
    one before); its output read-back runs on a second stream and overlaps the
    next step (outputs are double-buffered)."""
    R, L, K, H = w.R, w.L, w.K, w.heads
    attention = w.name == "attention"
    rb = row_bytes(args.kv_format == "fp8")
    steps = min(args.e2e_steps, topk_h.shape[0] - args.warmup)
    hs.hs_pool_reset(pool.handle, stream)
    tk_pin = torch.from_numpy(topk_h).pin_memory()
    q_pin = torch.from_numpy(q_h.view(np.int16)).pin_memory()
    tk_d = torch.empty((L, R, K), dtype=torch.int32, device=dev)
    q_d = torch.empty((L, R, H, W.ROW_ELEMS), dtype=torch.int16, device=dev)
    rows_d = torch.empty((L, R, K), dtype=torch.int32, device=dev)
    if attention:
        res_d = [(torch.empty((L, R, H, W.V_DIM), dtype=torch.bfloat16, device=dev),
                  torch.empty((L, R, H), dtype=torch.float32, device=dev)) for _ in range(2)]
        res_h = [(torch.empty((L, R, H, W.V_DIM), dtype=torch.bfloat16).pin_memory(),
                  torch.empty((L, R, H), dtype=torch.float32).pin_memory()) for _ in range(2)]
    else:
        res_d = [(torch.empty((R * K, rb // 2), dtype=torch.int16, device=dev),) for _ in range(2)]
        res_h = [(torch.empty((R * K, rb // 2), dtype=torch.int16).pin_memory(),)
                 for _ in range(2)]
    sptr = stream.cuda_stream
    copy_stream = torch.cuda.Stream(device=dev) if attention else None
    d2h_stream = torch.cuda.Stream(device=dev)
    done = [torch.cuda.Event() for _ in range(2)]    # step wrote result buffer i
    read = [torch.cuda.Event() for _ in range(2)]    # host copy of buffer i finished

    def step(t):
        i = t % 2
        tk_d.copy_(tk_pin[t], non_blocking=True)
        if attention:
            q_d.copy_(q_pin[t % Q_DISTINCT], non_blocking=True)
        if t >= 2:
            stream.wait_event(read[i])  # buffer i's previous result has been read back
        if attention:  # the library's step call, as in the device-resident run
            st = lib.hs_decode_step(pool.handle, 0, L, tk_d.data_ptr(), q_d.data_ptr(), H, W.V_DIM,
                                    W.SCALE, pool.step.data_ptr(), rows_d.data_ptr(),
                                    res_d[i][0].data_ptr(), res_d[i][1].data_ptr(), None, sptr,
                                    copy_stream.cuda_stream)
            if st != 0:
                raise RuntimeError(f"hs_decode_step failed: {hs.status_string(st)}")
        else:
            for l in range(L):
                lib.hs_resolve(pool.handle, l, 1, tk_d[l].data_ptr(), pool.step.data_ptr(),
                               rows_d[l].data_ptr(), None, None, sptr)
            lib.hs_gather(pool.handle, L - 1, rows_d[L - 1].data_ptr(), R * K,
                          res_d[i][0].data_ptr(), sptr)
        lib.hs_step_advance(pool.step.data_ptr(), sptr)
        done[i].record(stream)
        d2h_stream.wait_event(done[i])
        with torch.cuda.stream(d2h_stream):
            for hb, db in zip(res_h[i], res_d[i]):
                hb.copy_(db, non_blocking=True)
        read[i].record(d2h_stream)

    for t in range(args.warmup):
        step(t)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(steps):
        step(args.warmup + i)
    stream.wait_stream(d2h_stream)  # the last read-back is inside the timed region
    b.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), dist, dev)
    if hs.hs_check_errors(pool.handle):
        raise RuntimeError("device error word set in the e2e run")
    h2d = L * R * K * 4 + (L * R * H * W.ROW_ELEMS * 2 if attention else 0)
    d2h = (L * R * H * (W.V_DIM * 2 + 4)) if attention else R * K * rb
    return {"value": weak_scaling_rate(L * R * K, steps, world, ms), "unit": "rows/s",
            "steps": steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": "read-back of step t on a second stream beside step t+1"}


# ----------------------------------------------------------------- reference arm

def run_reference(args):
    """The CPU oracle as the reference arm: each step runs the oracle on a
    bounded sample of the workload (2 units: resolve + gather from the host's
    full KV + fp64 attention), on the host cores."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = W.make(args.workload)
    total = args.warmup + args.steps
    units = 2
    # the warm-up steps run untimed, then `steps` timed steps
    rows, secs, done = oracle_sample(w, seconds=1e9, units=units, steps_cap=total,
                                     skip=args.warmup, fp8=args.kv_format == "fp8")
    per_step = secs / max(done, 1)
    value = units * w.K / per_step
    cores = os.cpu_count() or 1
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generator; no dataset)", "impl": "reference",
        "config": {"workload": workload_name(w), "sample": f"{units} units per step",
                   "kv_rows": kv_rows_name(args.kv_format == "fp8")},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                         "sample": f"{units} (request, layer) units per step, {done} steps"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main(argv=None):
    raw = sys.argv[1:] if argv is None else list(argv)
    args = parse_args(raw)
    if args.cpu_baseline_child:
        w = W.make(args.workload)
        u0, u1 = (int(x) for x in args.cpu_units.split(":"))
        rows, secs, steps = oracle_sample(w, args.cpu_seconds, units=u1 - u0, steps_cap=512,
                                          fp8=args.kv_format == "fp8", unit0=u0)
        print(json.dumps({"rows": rows, "secs": secs, "steps": steps}))
        return 0
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return spawn_replicas(args, raw)
    if args.replica_check:
        run_replica_check(args)
        return 0
    if args.steps is None:
        args.steps = {"mixed": 120, "spec": 200}.get(args.workload, 2000)
    if args.impl == "reference":
        run_reference(args)
        return 0
    if args.workload == "mixed":
        run_mixed(args)
        return 0
    if args.workload == "spec":
        run_spec(args)
        return 0
    line = run_ours(args)
    if args.workload == "attention" and not args.no_extra and not args.profile:
        extra = extra_workloads(args)
        if line is not None:
            line["workloads"] = extra
    if line is not None:
        print(json.dumps(line))
    dist, _, _, _ = dist_context()
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
