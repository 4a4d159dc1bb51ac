"""Test harness: replay one synthetic workload scenario through the CUDA path
(via the C ABI binding) and through the CPU oracle, step by step.

Inputs for both sides come only from ``synth`` (seeded rows, queries, traces,
scenario); no expected value is ever read back from the GPU into the oracle.
"""
from __future__ import annotations

import os

import numpy as np

import oracle
import synth
from synth import workloads as W

HOST_THREADS = max(1, min(32, os.cpu_count() or 1))


def make_pool(w: W.Workload, scen: W.Scenario, kv_format: int = 0):
    """Create the libhs pool for a workload and bring it to its step-0 state:
    every request's full KV in the pinned host pool, resident pages loaded."""
    import torch
    import sparse_attention_kv_hs_gb300 as hs

    cap = w.ctx_capacity()
    max_pages = int((cap.max() + w.P - 1) // w.P)
    resident_blocks = scen.blocks_per_layer - w.R * w.hot_blocks_per_request()
    pool = hs.Pool(w.R, w.L, w.K, w.B, w.P, W.ROW_ELEMS, max_pages, w.host_tokens(),
                   max(resident_blocks, 1), kv_format)
    offs = w.host_offsets()
    hp = pool.host_pool
    # Host rows for positions < ctx at step 0; rows of pages appended later are
    # left zero: only the offload path may fill them.
    for l in range(w.L):
        for r in range(w.R):
            n = int(w.ctx[r])
            base = hp[l, int(offs[r]):int(offs[r]) + n]
            if kv_format == 1:  # FP8 rows (656 bytes each)
                synth.rows_fp8_into(w.seed, r, l, 0, n, base.ctypes.data, HOST_THREADS)
            else:
                synth.rows_into(w.seed, r, l, 0, n, W.ROW_ELEMS, base.ctypes.data, HOST_THREADS)
            extra = int(cap[r]) - n
            if extra > 0:
                hp[l, int(offs[r]) + n:int(offs[r]) + int(cap[r])] = 0
    stream = torch.cuda.current_stream()
    for r in range(w.R):
        hs.hs_set_request(pool.handle, r, int(w.ctx[r]), int(offs[r]), stream)
    for (r, page, blk) in scen.initial:
        hs.hs_load_page(pool.handle, r, page, blk, stream)
    torch.cuda.synchronize()
    return pool


def rows_for_oracle(w: W.Workload, r: int, l: int, pos, kv_format: int = 0) -> np.ndarray:
    """The KV rows at token positions `pos` of (request r, layer l) as the
    oracle's attention takes them: bf16 bits, or for FP8 pools the values the
    656-byte rows stand for (fp64)."""
    if kv_format == 1:
        return oracle.fp8_rows_to_f64(synth.rows_fp8_at(w.seed, r, l, pos))
    return synth.rows_at(w.seed, r, l, pos)


def make_oracle(w: W.Workload, scen: W.Scenario) -> oracle.ResolveOracle:
    o = oracle.ResolveOracle(w.R, w.L, w.K, w.B, w.P, w.ctx_capacity(), scen.blocks_per_layer)
    for r in range(w.R):
        o.set_ctx(r, int(w.ctx[r]))
        for i in range(w.hot_blocks_per_request()):
            o.set_hot_block(r, i, r * w.hot_blocks_per_request() + i)
    for (r, page, blk) in scen.initial:
        o.set_page(r, page, blk)
    return o


def traces(w: W.Workload) -> np.ndarray:
    """[steps, L, R, K] int32 selections for the whole workload."""
    out = np.empty((w.steps, w.L, w.R, w.K), dtype=np.int32)
    for r in range(w.R):
        out[:, :, r, :] = w.trace(r)
    return out


def lru_order_reference(stamp: np.ndarray) -> np.ndarray:
    """Slots sorted by (stamp, slot) -- what lru_order must hold."""
    return np.lexsort((np.arange(stamp.size), stamp)).astype(np.int32)


def write_append_gpu(pool, w, r, page, blk, stream):
    """A finished page: its rows are produced on the GPU (copied in from the
    generator, standing in for the model writing KV) and mapped resident."""
    import torch
    import sparse_attention_kv_hs_gb300 as hs

    rows = np.stack([synth.rows(w.seed, r, l, page * w.P, w.P) for l in range(w.L)])
    dev = torch.from_numpy(rows.view(np.int16)).to("cuda", non_blocking=False)
    for l in range(w.L):
        pool.kv_pool[l, blk * w.P:(blk + 1) * w.P].copy_(dev[l])
    hs.hs_map_page(pool.handle, r, page, blk, stream)


def apply_append_gpu(pool, w, r, page, blk, stream, side, events):
    """write_append_gpu, then a host copy of the page queued on the side stream."""
    import torch
    import sparse_attention_kv_hs_gb300 as hs

    write_append_gpu(pool, w, r, page, blk, stream)
    ev = torch.cuda.Event()
    hs.hs_offload_prefix(pool.handle, r, page, stream, side, ev)
    events[(r, page)] = ev
    return ev
