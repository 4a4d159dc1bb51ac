"""Replacement-policy study on the synthetic selection traces -- test
infrastructure, CPU only.

Page "59188saintaubert.com ... HiSparse", section 04, compares hot-buffer
replacement policies on real selection traces (GLM-5.1, LongBenchV2): at
B = 4096 the miss rate is 13.4% for LRU, 17.2% for FIFO, 16.1% for random and
8.2% for the offline optimum (Belady); at B = 8192 LRU misses 6.7%.  Those
traces are not available; this script runs the same comparison on the seeded
synthetic traces of the resolve and attention workloads, for B = 2048, 4096,
8192 (top-K 2048), with RESOLVE's step structure (oracle/policy_sim.c).
Miss rate = misses / selected non-resident positions over steps >= 1 (step 0
fills an empty buffer).

    python oracle/policy_study.py [--requests N] [--steps S]
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

import oracle  # noqa: E402
from synth import workloads as W  # noqa: E402

POLICIES = ("lru", "fifo", "random", "belady")
SLOTS = (2048, 4096, 8192)


def unit_traces(name: str, requests: int, steps: int):
    """Layer-0 selections of the first `requests` requests, resident positions
    (the tail) masked to -1, with each request's context length."""
    w = W.make(name, steps=steps)
    out = []
    for r in range(min(requests, w.R)):
        tr = w.trace(r)[:, 0, :].astype(np.int32)  # [steps][K]
        ctx = int(w.ctx[r])
        resident = set(w.resident_pages(r, ctx))
        if resident:
            pages = tr // w.P
            mask = np.isin(pages, np.array(sorted(resident)))
            tr = np.where(mask, -1, tr).astype(np.int32)
        out.append((tr, ctx))
    return w, out


def study(name: str, requests: int, steps: int):
    w, traces = unit_traces(name, requests, steps)
    rows = {}
    for B in SLOTS:
        for pol in POLICIES:
            miss = sel = 0
            for u, (tr, ctx) in enumerate(traces):
                m = oracle.policy_misses(pol, tr, B, ctx, seed=1000 + u)
                miss += int(m[1:].sum())
                sel += int((tr[1:] >= 0).sum())
            rows[(B, pol)] = miss / max(sel, 1)
    return w, rows


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--requests", type=int, default=16)
    ap.add_argument("--steps", type=int, default=128)
    args = ap.parse_args(argv)
    print("| workload | B | LRU | FIFO | random | Belady |")
    print("|---|---|---|---|---|---|")
    for name in ("resolve", "attention"):
        w, rows = study(name, args.requests, args.steps)
        for B in SLOTS:
            cells = " | ".join(f"{100 * rows[(B, p)]:.1f}%" for p in POLICIES)
            print(f"| {name} ({args.requests} requests x {args.steps} steps, K {w.K}) | {B} | {cells} |")


if __name__ == "__main__":
    main()
