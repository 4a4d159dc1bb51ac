"""Pins for the CPU oracle: checks against things fixed outside the oracle's
own code (a hand-worked example, an independently written LRU model, closed
forms from the pages, the Belady bound, textbook special cases of softmax
attention).  No GPU needed."""
import itertools
import math
import os
import random

import numpy as np
import pytest

import oracle
import synth
from synth import workloads as W
from tests import lru_alt

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "resolve_worked_example.txt")


def _parse_golden():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("setup"):
            kv = dict(tok.split("=") for tok in line.split()[1:])
            res = {}
            if kv["resident"]:
                for item in kv["resident"].split(","):
                    pg, blk = item.split(":")
                    res[int(pg)] = int(blk)
            cur = dict(ctx=int(kv["ctx"]), P=int(kv["P"]), K=int(kv["K"]), B=int(kv["B"]),
                       hot=int(kv["hot_blocks"]), resident=res, steps=[])
            cases.append(cur)
        elif line.startswith("step"):
            f = [x.strip() for x in line[len("step"):].split("|")]
            cur["steps"].append(dict(t=int(f[0]), topk=[int(x) for x in f[1].split()],
                                     rows=[int(x) for x in f[2].split()],
                                     pos=[int(x) for x in f[3].split()],
                                     stamp=[int(x) for x in f[4].split()], err=int(f[5])))
    return cases


def _oracle_for(ctx, P, K, B, hot_blocks, resident, blocks_per_layer=64):
    o = oracle.ResolveOracle(1, 1, K, B, P, [ctx], blocks_per_layer)
    o.set_ctx(0, ctx)
    for i, blk in enumerate(hot_blocks):
        o.set_hot_block(0, i, blk)
    for page, blk in resident.items():
        o.set_page(0, page, blk)
    return o


def test_worked_example_golden():
    cases = _parse_golden()
    assert len(cases) == 2
    for c in cases:
        o = _oracle_for(c["ctx"], c["P"], c["K"], c["B"], [c["hot"]], c["resident"])
        for st in c["steps"]:
            rows, log, err = o.resolve(0, 0, np.array(st["topk"]), st["t"])
            pos, stamp = o.unit_state(0, 0)
            assert rows.tolist() == st["rows"], st
            assert pos.tolist() == st["pos"], st
            assert stamp.tolist() == st["stamp"], st
            assert err == st["err"], st
            # the miss log lists served misses in selection order
            assert [r[0] for r in log] == sorted(r[0] for r in log)


def _random_case(rng):
    P = rng.choice([1, 2])
    ctx = rng.randint(2, 8)
    K = rng.randint(1, 3)
    B = P * rng.randint(max(1, (K + P - 1) // P) if rng.random() < 0.8 else 1, 6 // P if P > 1 else 6)
    n_pages = (ctx + P - 1) // P
    resident = {pg: 10 + pg for pg in range(n_pages) if rng.random() < 0.25}
    hot = [20 + i for i in range(B // P)]
    steps = []
    for _ in range(rng.randint(1, 4)):
        sel = rng.sample(range(ctx), min(K, ctx))
        sel += [-1] * (K - len(sel))
        if rng.random() < 0.1:
            sel[rng.randrange(K)] = rng.choice([ctx, ctx + 3, -2])  # invalid
        if K > 1 and rng.random() < 0.1:
            sel[1] = sel[0]                                        # repeat
        steps.append(sel)
    return ctx, P, K, B, hot, resident, steps


def test_bruteforce_against_independent_lru():
    """Thousands of tiny traces (ctx <= 8, K <= 3, B <= 6, <= 4 steps):
    the oracle and the recency-list model agree on every row id, every slot's
    position and every error bit."""
    rng = random.Random(7)
    for _ in range(3000):
        ctx, P, K, B, hot, resident, steps = _random_case(rng)
        o = _oracle_for(ctx, P, K, B, hot, resident)
        ref = lru_alt.replay(ctx, P, B, hot, resident, steps)
        for t, (sel, (rows_ref, holder_ref, err_ref)) in enumerate(zip(steps, ref)):
            rows, _, err = o.resolve(0, 0, np.array(sel), t)
            pos, _ = o.unit_state(0, 0)
            assert rows.tolist() == rows_ref, (ctx, P, K, B, resident, steps, t)
            assert pos.tolist() == holder_ref, (ctx, P, K, B, resident, steps, t)
            assert err == err_ref


def test_exhaustive_small_two_step():
    """Every pair of 2-selections over ctx=5 with B=2 (no resident pages)."""
    sels = [list(c) for c in itertools.permutations(range(5), 2)]
    for a in sels:
        for b in sels:
            o = _oracle_for(5, 1, 2, 2, [30, 31], {})
            ref = lru_alt.replay(5, 1, 2, [30, 31], {}, [a, b])
            for t, sel in enumerate((a, b)):
                rows, _, err = o.resolve(0, 0, np.array(sel), t)
                assert rows.tolist() == ref[t][0] and err == ref[t][2] == 0


def _replay_oracle(w, r=0, layer=0, scen=None):
    """Run the oracle over all steps of one unit of a workload (no appends)."""
    scen = scen or W.Scenario.build(w)
    o = oracle.ResolveOracle(w.R, w.L, w.K, w.B, w.P, w.ctx_capacity(), scen.blocks_per_layer)
    for rr in range(w.R):
        o.set_ctx(rr, int(w.ctx[rr]))
        for i in range(w.hot_blocks_per_request()):
            o.set_hot_block(rr, i, rr * w.hot_blocks_per_request() + i)
    for (rr, page, blk) in scen.initial:
        o.set_page(rr, page, blk)
    tr = w.trace(r)
    per_step = []
    for t in range(w.steps):
        rows, log, err = o.resolve(layer, r, tr[t, layer], t)
        assert err == 0
        per_step.append((rows, log))
    return o, tr, per_step


def test_closed_form_b_equals_k():
    """B = K, nothing resident: after every step the buffer holds exactly that
    step's selection, so step t misses exactly |S_t minus S_(t-1)| (page
    "59188saintaubert.com ... HiSparse", section 02: staging only the current
    top-k misses about 30% of each step's selections)."""
    w = W.make("tiny")
    w.B = w.K
    o, tr, per_step = _replay_oracle(w)
    rates = []
    for t in range(w.steps):
        expect = w.K if t == 0 else len(set(tr[t, 0]) - set(tr[t - 1, 0]))
        assert len(per_step[t][1]) == expect
        if t:
            rates.append(expect / w.K)
    pos, _ = o.unit_state(0, 0)
    assert set(pos.tolist()) == set(tr[-1, 0].tolist())
    assert 0.25 <= np.mean(rates) <= 0.31   # "about 30%"


def test_cold_buffer_misses_are_new_selections():
    """While the buffer has never been full, a miss is exactly a first-time
    selection of a host-only position."""
    w = W.make("tiny", steps=8)
    w.B = 4096  # 8 steps x <= 256 new positions never fill it
    o, tr, per_step = _replay_oracle(w)
    seen = set()
    for t in range(w.steps):
        new = set(tr[t, 0].tolist()) - seen
        assert {int(p) for _, p, _ in per_step[t][1]} == new
        seen |= set(tr[t, 0].tolist())


def test_buffer_at_least_context_every_position_misses_once():
    """B >= ctx: each position misses at most once; after first touch every
    selection hits (hit rate 100%)."""
    w = W.make("tiny", ctx=1024, steps=32)
    w.B = 1024
    o, tr, per_step = _replay_oracle(w)
    loaded = [int(p) for step in per_step for _, p, _ in step[1]]
    assert len(loaded) == len(set(loaded)) == len(set(tr.reshape(-1).tolist()))


def _belady_misses(stream, capacity):
    """Offline optimal (furthest next use) miss count on an access stream."""
    nxt = [0] * len(stream)
    last = {}
    for i in range(len(stream) - 1, -1, -1):
        nxt[i] = last.get(stream[i], math.inf)
        last[stream[i]] = i
    cache, misses = {}, 0      # position -> next use index
    for i, p in enumerate(stream):
        if p in cache:
            cache[p] = nxt[i]
            continue
        misses += 1
        if len(cache) >= capacity:
            victim = max(cache, key=lambda x: cache[x])
            del cache[victim]
        cache[p] = nxt[i]
    return misses


def test_lru_never_beats_belady():
    """Two-phase LRU is a demand-paging policy on the selection stream, so its
    misses are >= the offline optimum with the same capacity (page
    "59188saintaubert.com ... HiSparse", section 04 compares LRU with Belady)."""
    w = W.make("tiny", ctx=2048, steps=24)
    w.K, w.B, w.P = 64, 96, 32
    o, tr, per_step = _replay_oracle(w)
    lru = sum(len(s[1]) for s in per_step)
    opt = _belady_misses([int(p) for t in range(w.steps) for p in tr[t, 0]], w.B)
    assert lru >= opt
    assert opt > 0


def test_exactness_rows_hold_the_selected_positions():
    """Only placement changes (page "59188saintaubert.com ... HiSparse", end of
    section 02): every row id handed out holds the selected position, whether
    it is read in place (resident tail) or from the hot buffer."""
    w = W.make("resolve", R=2, steps=12, ctx=8192)
    scen = W.Scenario.build(w)
    o = oracle.ResolveOracle(w.R, w.L, w.K, w.B, w.P, w.ctx_capacity(), scen.blocks_per_layer)
    for r in range(w.R):
        o.set_ctx(r, int(w.ctx[r]))
        for i in range(w.hot_blocks_per_request()):
            o.set_hot_block(r, i, r * w.hot_blocks_per_request() + i)
    for (r, page, blk) in scen.initial:
        o.set_page(r, page, blk)
    traces = [w.trace(r) for r in range(w.R)]
    resident_seen = 0
    for t in range(w.steps):
        for l in range(w.L):
            for r in range(w.R):
                rows, log, err = o.resolve(l, r, traces[r][t, l], t)
                assert err == 0
                for j in range(0, w.K, 7):
                    assert o.row_content(l, r, int(rows[j])) == traces[r][t, l, j]
                tail0 = int(w.ctx[r]) - w.tail
                resident_seen += int((traces[r][t, l] >= tail0).sum())
                # resident positions never enter the miss log
                assert all(p < tail0 for _, p, _ in log)
    assert resident_seen > 0


def test_capacity_ratio_matches_pages():
    """Per-request decode KV scales with B, not context: at 128K context and
    B = 4096 the hot buffer is ctx/B = 32x smaller than full KV; the pages
    quote 13.09 GB -> about 0.4 GB, "about 30x" (page "59188saintaubert.com
    ... HiSparse", section 03)."""
    ratio = 131072 / 4096
    assert ratio == 32
    assert abs(13.09 / ratio - 0.4) < 0.01


# --------------------------------------------------------------- attention

def _bf16(x):
    """Round float64 values to bf16 bits (RNE) for test inputs."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def test_attention_single_row_is_that_row():
    rng = np.random.default_rng(0)
    q = _bf16(rng.standard_normal((4, 576)))
    k = _bf16(rng.standard_normal((1, 576)))
    out, lse = oracle.sparse_mla_decode(q, k, None, W.SCALE)
    v = oracle.bf16_bits_to_f64(k)[0, :512]
    assert np.array_equal(out, np.broadcast_to(v, out.shape))
    s = W.SCALE * (oracle.bf16_bits_to_f64(q) @ oracle.bf16_bits_to_f64(k)[0])
    assert np.allclose(lse, s, rtol=0, atol=1e-12)


def test_attention_zero_query_is_mean():
    rng = np.random.default_rng(1)
    k = _bf16(rng.standard_normal((37, 576)))
    q = np.zeros((3, 576), dtype=np.uint16)
    out, lse = oracle.sparse_mla_decode(q, k, None, W.SCALE)
    kf = oracle.bf16_bits_to_f64(k)
    assert np.allclose(out, kf[:, :512].mean(axis=0), rtol=0, atol=1e-12)
    assert np.allclose(lse, math.log(37), atol=1e-12)


def test_attention_identical_rows():
    rng = np.random.default_rng(2)
    row = _bf16(rng.standard_normal(576))
    k = np.tile(row, (9, 1))
    q = _bf16(rng.standard_normal((5, 576)))
    out, _ = oracle.sparse_mla_decode(q, k, None, W.SCALE)
    assert np.allclose(out, oracle.bf16_bits_to_f64(row)[:512], rtol=0, atol=1e-12)


def test_attention_two_rows_logistic():
    """Two rows: the weights are logistic in the score difference."""
    rng = np.random.default_rng(3)
    q = _bf16(rng.standard_normal((1, 576)))
    k = _bf16(rng.standard_normal((2, 576)))
    qf, kf = oracle.bf16_bits_to_f64(q)[0], oracle.bf16_bits_to_f64(k)
    s = [W.SCALE * math.fsum(float(a) * float(b) for a, b in zip(qf, kf[j])) for j in range(2)]
    w0 = 1.0 / (1.0 + math.exp(s[1] - s[0]))
    expect = w0 * kf[0, :512] + (1.0 - w0) * kf[1, :512]
    out, lse = oracle.sparse_mla_decode(q, k, None, W.SCALE)
    assert np.allclose(out[0], expect, rtol=0, atol=1e-12)
    assert abs(lse[0] - (max(s) + math.log1p(math.exp(min(s) - max(s))))) < 1e-12


def test_attention_bruteforce_loops_and_padding():
    """Pure-Python loops on a small case; padding rows are excluded."""
    rng = np.random.default_rng(4)
    H, K, D, V = 3, 6, 8, 5
    q = rng.standard_normal((H, D))
    k = rng.standard_normal((K, D))
    valid = np.array([1, 0, 1, 1, 0, 1], dtype=bool)
    out, lse = oracle.sparse_mla_decode(q, k, valid, 0.37, v_dim=V)
    for h in range(H):
        sc = {j: 0.37 * math.fsum(q[h, d] * k[j, d] for d in range(D)) for j in range(K) if valid[j]}
        m = max(sc.values())
        den = math.fsum(math.exp(x - m) for x in sc.values())
        for e in range(V):
            num = math.fsum(math.exp(sc[j] - m) * k[j, e] for j in sc)
            assert abs(out[h, e] - num / den) < 1e-12
        assert abs(lse[h] - (m + math.log(den))) < 1e-12


def test_attention_no_valid_rows():
    q = np.zeros((2, 576), dtype=np.uint16)
    k = np.zeros((3, 576), dtype=np.uint16)
    out, lse = oracle.sparse_mla_decode(q, k, np.zeros(3, bool), W.SCALE)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_attention_through_cache_equals_full_kv():
    """Exactness end to end on the tiny workload: attention over the rows the
    oracle's resolve hands out (looked up by the position each row holds)
    equals attention over rows read straight from full KV."""
    w = W.make("tiny", steps=6)
    o, tr, per_step = _replay_oracle(w)
    for t in (0, 5):
        rows = per_step[t][0]
        held = np.array([o.row_content(0, 0, int(x)) for x in rows]) if t == 5 else None
        q = synth.q(w.seed, 0, 0, t, w.heads)
        full = synth.rows_at(w.seed, 0, 0, tr[t, 0])
        a, la = oracle.sparse_mla_decode(q, full, None, W.SCALE)
        if held is not None:
            via = synth.rows_at(w.seed, 0, 0, held)
            b, lb = oracle.sparse_mla_decode(q, via, None, W.SCALE)
            assert np.array_equal(a, b) and np.array_equal(la, lb)


# ------------------------------------------------ speculative decoding (T verify tokens)

def test_tokens_hand_worked_example():
    """B = 3 one-row slots (rows 20, 21, 22), K = 2, T = 2 verify tokens,
    positions a=0, b=1, c=2, d=3.
    Step 0, tokens [a b] [b c]: a, b, c miss and fill slots 0, 1, 2; token 1's
    b shares token 0's row 21.
    Step 1, tokens [c d] [a d]: c (slot 2) and a (slot 0) are hits, pinned for
    the whole step; d misses and takes the only unpinned slot, 1 (b's);
    token 1's d shares that row.  Resolving the tokens one call at a time
    instead would let token 0's d evict a (slot 0, the lowest of the two
    oldest), which token 1 then misses."""
    o = _oracle_for(4, 1, 2, 3, [20, 21, 22], {})
    rows, log, err = o.resolve_tokens(0, 0, np.array([[0, 1], [1, 2]]), 0)
    assert err == 0 and rows.tolist() == [[20, 21], [21, 22]] and len(log) == 3
    rows, log, err = o.resolve_tokens(0, 0, np.array([[2, 3], [0, 3]]), 1)
    assert err == 0 and rows.tolist() == [[22, 21], [20, 21]]
    assert log.tolist() == [[1, 3, 1]]  # (list index j, position, slot)
    assert o.unit_state(0, 0)[0].tolist() == [0, 3, 2]
    # the same two steps token by token give a different (worse) result
    o2 = _oracle_for(4, 1, 2, 3, [20, 21, 22], {})
    o2.resolve(0, 0, np.array([0, 1]), 0)
    o2.resolve(0, 0, np.array([1, 2]), 0)
    r0, l0, _ = o2.resolve(0, 0, np.array([2, 3]), 1)
    r1, l1, _ = o2.resolve(0, 0, np.array([0, 3]), 1)
    assert r0.tolist() == [22, 20] and r1.tolist() == [21, 20] and len(l0) + len(l1) == 2


def _random_tokens_case(rng):
    P = rng.choice([1, 2])
    ctx = rng.randint(2, 8)
    K = rng.randint(1, 3)
    T = rng.randint(1, 3)
    lo = max(1, (T * K + P - 1) // P) if rng.random() < 0.8 else 1
    B = P * rng.randint(lo, max(lo, 9 // P))
    n_pages = (ctx + P - 1) // P
    resident = {pg: 10 + pg for pg in range(n_pages) if rng.random() < 0.25}
    hot = [20 + i for i in range(B // P)]
    steps = []
    for _ in range(rng.randint(1, 4)):
        toks = []
        for _t in range(T):
            sel = rng.sample(range(ctx), min(K, ctx))
            sel += [-1] * (K - len(sel))
            if rng.random() < 0.08:
                sel[rng.randrange(K)] = rng.choice([ctx, ctx + 3, -2])  # invalid
            if K > 1 and rng.random() < 0.08:
                sel[1] = sel[0]                                        # repeat in a token
            toks.append(sel)
        steps.append(toks)
    return ctx, P, K, T, B, hot, resident, steps


def test_tokens_bruteforce_against_independent_lru():
    """Thousands of tiny multi-token traces (ctx <= 8, K <= 3, T <= 3, B <= 9):
    the oracle and the recency-list model agree on every row id, every slot's
    position and every error bit."""
    rng = random.Random(17)
    for _ in range(3000):
        ctx, P, K, T, B, hot, resident, steps = _random_tokens_case(rng)
        o = _oracle_for(ctx, P, K, B, hot, resident)
        ref = lru_alt.replay_tokens(ctx, P, B, hot, resident, steps)
        for t, (toks, (rows_ref, holder_ref, err_ref)) in enumerate(zip(steps, ref)):
            rows, _, err = o.resolve_tokens(0, 0, np.array(toks), t)
            pos, _ = o.unit_state(0, 0)
            assert rows.tolist() == rows_ref, (ctx, P, K, T, B, resident, steps, t)
            assert pos.tolist() == holder_ref, (ctx, P, K, T, B, resident, steps, t)
            assert err == err_ref


def test_tokens_one_token_is_the_plain_call():
    rng = random.Random(23)
    for _ in range(500):
        ctx, P, K, B, hot, resident, steps = _random_case(rng)
        a = _oracle_for(ctx, P, K, B, hot, resident)
        b = _oracle_for(ctx, P, K, B, hot, resident)
        for t, sel in enumerate(steps):
            ra, la, ea = a.resolve(0, 0, np.array(sel), t)
            rb, lb, eb = b.resolve_tokens(0, 0, np.array([sel]), t)
            assert rb[0].tolist() == ra.tolist() and lb.tolist() == la.tolist() and ea == eb


def test_tokens_exactness_and_shared_rows():
    """K 64, T 3 overlapping verify tokens, B = (T + 2) K: every entry's row
    holds its position, a position shared by tokens has one row, and the misses
    of a step are exactly the union's positions not yet in the buffer."""
    rng = np.random.default_rng(29)
    ctx, K, T, P = 2048, 64, 3, 64
    B = (T + 2) * K
    o = oracle.ResolveOracle(1, 1, K, B, P, [ctx], B // P)
    o.set_ctx(0, ctx)
    for i in range(B // P):
        o.set_hot_block(0, i, i)
    held = set()
    prev = rng.choice(ctx, K, replace=False)
    for t in range(20):
        toks = []
        for _ in range(T):
            keep = rng.choice(prev, int(0.7 * K), replace=False)
            rest = rng.choice(np.setdiff1d(np.arange(ctx), keep), K - len(keep), replace=False)
            toks.append(rng.permutation(np.concatenate([keep, rest])))
        rows, log, err = o.resolve_tokens(0, 0, np.array(toks), t)
        assert err == 0
        union = set(int(p) for tok in toks for p in tok)
        assert len(log) == len(union - held)
        seen = {}
        for ti in range(T):
            for j in range(K):
                p, row = int(toks[ti][j]), int(rows[ti, j])
                assert o.row_content(0, 0, row) == p
                assert seen.setdefault(p, row) == row
        pos, _ = o.unit_state(0, 0)
        held = set(int(x) for x in pos if x >= 0)
        prev = toks[-1]
