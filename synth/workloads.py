"""The five synthetic decode workloads and their residency scenarios.

Input structure only (sizes, context lengths, residency classes, append
schedule, block numbering); no step of the method is computed here.  Both the
CUDA path's tests/bench and the oracle replay the same scenario object, so the
two sides see identical page tables, block ids and selections.

Workloads (sizes as stated for the HiSparse decode path):
  tiny      1 request x 1 layer, ctx 8192, top-K 256, B 512, no resident tail,
            64 steps, 70% reuse + 30% uniform, 16 heads
  resolve   16 x 4, ctx 32768, K 2048, B 4096, tail 4096, 256 steps,
            70% reuse / 20% Zipf(1.1) / 10% uniform, adjacent layers share 80%
  gather    64 x 4, ctx 131072, K 2048, B 4096, tail 4096, 128 steps, same
            drift; cold start at step 0
  attention 32 x 2, ctx 65536, K 2048, B 4096, 128 heads, 64 steps,
            70% reuse + 30% uniform (no resident tail)
  mixed     128 x 1, ctx log-uniform in [16384, 1048576] (host <= 64 GB),
            K 2048, B 4096, tail 4096; 1/4 zero residency, 1/4 fully resident,
            1/2 resident tail; 5% of requests append a 256-token page per step
            (queued for host offload); 128 steps, 70/20/10 drift
  spec      the attention workload with speculative decoding: T = 2 verify
            tokens per request and step (one speculative token), B = (T + 2) K
            = 8192; token 0 drifts as in "attention", token t > 0 keeps 85% of
            token t-1's selection and draws the rest uniformly
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

from . import key as _key, draw as _draw, trace as _trace

ROW_ELEMS = 576
ROW_BYTES = ROW_ELEMS * 2
PAGE_TOKENS = 256
V_DIM = 512
SCALE = 1.0 / math.sqrt(192.0)

TAG_SCEN = 0x5343454E  # "SCEN"
TAG_SPEC = 0x53504543  # "SPEC"


@dataclasses.dataclass
class Workload:
    name: str
    R: int
    L: int
    K: int
    B: int
    steps: int
    ctx: np.ndarray                 # [R] context length at step 0
    tail: int                       # resident tail tokens for "mixed" requests
    residency: list                 # [R] "mixed" | "full" | "zero"
    reuse: float
    zipf_frac: float
    layer_share: float
    heads: int
    seed: int
    appends_per_step: int = 0
    P: int = PAGE_TOKENS
    zipf_s: float = 1.1
    req_base: int = 0               # generator id of request 0 (replicas use disjoint ids)
    tokens: int = 1                 # verify tokens per step (speculative decoding)
    token_share: float = 0.0        # share of token t-1's selection token t keeps

    # ---- derived scenario -------------------------------------------------
    def append_schedule(self) -> list:
        """Requests that append a finished page at the end of each step."""
        sched = []
        if self.appends_per_step <= 0:
            return [[] for _ in range(self.steps)]
        for t in range(self.steps):
            k = _key(self.seed, TAG_SCEN, 1, t)
            order = list(range(self.R))
            for i in range(self.R - 1, 0, -1):  # seeded Fisher-Yates
                j = _draw(k, i) % (i + 1)
                order[i], order[j] = order[j], order[i]
            sched.append(sorted(order[: self.appends_per_step]))
        return sched

    def ctx_per_step(self) -> np.ndarray:
        """[steps, R] context length seen by the resolve of each step."""
        out = np.empty((self.steps, self.R), dtype=np.int64)
        cur = self.ctx.astype(np.int64).copy()
        for t, reqs in enumerate(self.append_schedule()):
            out[t] = cur
            for r in reqs:
                cur[r] += self.P
        return out

    def ctx_capacity(self) -> np.ndarray:
        cps = self.ctx_per_step()
        last = cps[-1].copy()
        for r in self.append_schedule()[-1]:
            last[r] += self.P
        return np.maximum(last, self.ctx).astype(np.int64)

    def host_offsets(self) -> np.ndarray:
        cap = self.ctx_capacity()
        return np.concatenate([[0], np.cumsum(cap)[:-1]]).astype(np.int64)

    def host_tokens(self) -> int:
        return int(self.ctx_capacity().sum())

    def hot_blocks_per_request(self) -> int:
        return self.B // self.P

    def resident_pages(self, r: int, ctx: int) -> list:
        """Pages of request r that are GPU-resident at context length ctx."""
        n_pages = ctx // self.P
        kind = self.residency[r]
        if kind == "full":
            return list(range(n_pages))
        if kind == "zero":
            return []
        first = max(0, (ctx - self.tail) // self.P)
        return list(range(first, n_pages))

    def max_resident_blocks(self) -> int:
        """Upper bound on resident blocks live at once (+ transient appends)."""
        cap = self.ctx_capacity()
        total = 0
        for r in range(self.R):
            if self.residency[r] == "full":
                total += int(cap[r]) // self.P
            elif self.residency[r] == "mixed":
                total += min(int(cap[r]) // self.P, self.tail // self.P + 1)
            else:
                total += 1
        return total + self.appends_per_step

    def trace(self, r: int) -> np.ndarray:
        """[steps, L, K] top-K positions of request r."""
        return _trace(self.seed, self.req_base + r, self.K, self.L, self.steps,
                      self.ctx_per_step()[:, r].astype(np.int32), self.reuse,
                      self.zipf_frac, self.zipf_s, self.layer_share)

    def trace_tokens(self, r: int) -> np.ndarray:
        """[steps, L, T, K] selections of request r's T verify tokens: token 0
        is trace(r); token t > 0 keeps floor(token_share * K) positions of
        token t-1's selection (a seeded choice) and draws the rest uniformly
        over the context, never repeating a position within the token."""
        base = self.trace(r)
        steps, L, K = base.shape
        out = np.empty((steps, L, self.tokens, K), dtype=np.int32)
        out[:, :, 0, :] = base
        keep = int(self.token_share * K)
        ctx = self.ctx_per_step()[:, r]
        for t in range(steps):
            n = int(ctx[t])
            for l in range(L):
                for tok in range(1, self.tokens):
                    g = np.random.Generator(np.random.PCG64(
                        _key(self.seed, TAG_SPEC, self.req_base + r, t * L + l, tok)))
                    prev = out[t, l, tok - 1]
                    kept = g.choice(prev, keep, replace=False)
                    taken = np.zeros(n, dtype=bool)
                    taken[kept] = True
                    fresh = []
                    while len(fresh) < K - keep:
                        cand = g.integers(0, n, size=2 * (K - keep))
                        for c in cand:
                            if not taken[c]:
                                taken[c] = True
                                fresh.append(c)
                                if len(fresh) == K - keep:
                                    break
                    row = np.concatenate([kept, np.array(fresh, dtype=np.int64)])
                    out[t, l, tok] = g.permutation(row)
        return out

    def host_bytes(self) -> int:
        return self.host_tokens() * self.L * ROW_BYTES


def _residency(kind: str, R: int, seed: int) -> list:
    if kind != "mixed-stress":
        return [kind] * R
    k = _key(seed, TAG_SCEN, 2)
    order = list(range(R))
    for i in range(R - 1, 0, -1):
        j = _draw(k, i) % (i + 1)
        order[i], order[j] = order[j], order[i]
    res = ["mixed"] * R
    q = R // 4
    for r in order[:q]:
        res[r] = "zero"
    for r in order[q:2 * q]:
        res[r] = "full"
    return res


def _log_uniform_ctx(R: int, lo: int, hi: int, seed: int, budget_bytes: int, L: int,
                     P: int, extra_tokens: int) -> np.ndarray:
    attempt = 0
    while True:
        k = _key(seed, TAG_SCEN, 3, attempt)
        u = np.array([(_draw(k, i) >> 11) * 2.0**-53 for i in range(R)])
        ctx = np.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
        ctx = (np.floor(ctx / P) * P).astype(np.int64)
        ctx = np.clip(ctx, lo, hi)
        if (ctx.sum() + extra_tokens) * ROW_BYTES * L <= budget_bytes:
            return ctx
        attempt += 1


def make(name: str, *, R: int | None = None, steps: int | None = None,
         ctx: int | None = None, ctx_hi: int | None = None, L: int | None = None,
         tokens: int | None = None) -> Workload:
    """One of the workloads; keyword overrides give scaled-down copies (tokens:
    the spec workload's verify tokens T, with B = (T + 2) K)."""
    if name == "tiny":
        R_ = R or 1
        w = Workload("tiny", R_, L or 1, 256, 512, steps or 64,
                     np.full(R_, ctx or 8192, dtype=np.int64), 0, ["zero"] * R_,
                     0.7, 0.0, 0.0, 16, 1001)
    elif name == "resolve":
        R_ = R or 16
        w = Workload("resolve", R_, L or 4, 2048, 4096, steps or 256,
                     np.full(R_, ctx or 32768, dtype=np.int64), 4096, ["mixed"] * R_,
                     0.7, 0.2, 0.8, 128, 1002)
    elif name == "gather":
        R_ = R or 64
        w = Workload("gather", R_, L or 4, 2048, 4096, steps or 128,
                     np.full(R_, ctx or 131072, dtype=np.int64), 4096, ["mixed"] * R_,
                     0.7, 0.2, 0.8, 128, 1003)
    elif name == "attention":
        R_ = R or 32
        w = Workload("attention", R_, L or 2, 2048, 4096, steps or 64,
                     np.full(R_, ctx or 65536, dtype=np.int64), 0, ["zero"] * R_,
                     0.7, 0.0, 0.0, 128, 1004)
    elif name == "spec":
        R_ = R or 32
        T = tokens or 2
        w = Workload("spec", R_, L or 2, 2048, (T + 2) * 2048, steps or 64,
                     np.full(R_, ctx or 65536, dtype=np.int64), 0, ["zero"] * R_,
                     0.7, 0.0, 0.0, 128, 1006, tokens=T, token_share=0.85)
    elif name == "mixed":
        R_ = R or 128
        steps_ = steps or 128
        appends = max(1, round(0.05 * R_))
        hi = ctx_hi or 1048576
        c = _log_uniform_ctx(R_, 16384, hi, 1005, 64 << 30, L or 1, PAGE_TOKENS,
                             steps_ * appends * PAGE_TOKENS)
        w = Workload("mixed", R_, L or 1, 2048, 4096, steps_, c, 4096,
                     _residency("mixed-stress", R_, 1005), 0.7, 0.2, 0.0, 128, 1005,
                     appends_per_step=appends)
    else:
        raise KeyError(name)
    return w


NAMES = ("tiny", "resolve", "gather", "attention", "mixed", "spec")


@dataclasses.dataclass
class Scenario:
    """Block numbering and page-table events of one workload, step by step.

    * hot blocks: request r owns blocks r*(B/P) .. r*(B/P)+B/P-1 (leased once);
    * resident pages get blocks from a free list (lowest id first);
    * appends[t]: (req, page, block) appended after the step-t decode and
      queued for host offload;
    * flips[t]: (req, page, block) that turn host-only at the boundary before
      step t (their host copy exists by then); their block is freed.
    """
    initial: list          # [(req, page, block)] resident at step 0
    appends: list          # per step: [(req, page, block)]
    flips: list            # per step: [(req, page, block)]
    blocks_per_layer: int
    hot_block_base: int = 0

    @staticmethod
    def build(w: Workload) -> "Scenario":
        hot = w.R * w.hot_blocks_per_request()
        free: list = []
        next_block = hot
        import heapq

        def alloc():
            nonlocal next_block
            if free:
                return heapq.heappop(free)
            b = next_block
            next_block += 1
            return b

        initial = []
        where = {}  # (r, page) -> block
        for r in range(w.R):
            for page in w.resident_pages(r, int(w.ctx[r])):
                b = alloc()
                initial.append((r, page, b))
                where[(r, page)] = b
        ctx = w.ctx.astype(np.int64).copy()
        appends, flips = [], [[] for _ in range(w.steps)]
        for t, reqs in enumerate(w.append_schedule()):
            # boundary before step t: pending flips were decided at step t-1
            for (r, page, b) in flips[t]:
                del where[(r, page)]
                heapq.heappush(free, b)
            step_app = []
            for r in reqs:
                page = int(ctx[r]) // w.P
                b = alloc()
                where[(r, page)] = b
                step_app.append((r, page, b))
                ctx[r] += w.P
                keep = set(w.resident_pages(r, int(ctx[r])))
                if w.residency[r] == "zero":
                    keep = set()
                if t + 1 < w.steps:
                    for (rr, pg), bb in sorted(where.items()):
                        if rr == r and pg not in keep:
                            flips[t + 1].append((rr, pg, bb))
            appends.append(step_app)
        return Scenario(initial, appends, flips, next_block)
