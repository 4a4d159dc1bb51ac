"""Pins of the replacement-policy simulator (oracle/policy_sim.c), the CPU
extension behind the LRU / FIFO / random / Belady comparison of page
"59188saintaubert.com ... HiSparse", section 04.

* its LRU reproduces the RESOLVE oracle's miss counts (two separate codes);
* B = K: every policy coincides (the only candidates are the slots the new
  selection dropped);
* B >= context: every policy has compulsory misses only;
* Belady equals the optimum found by exhaustive search on tiny traces, and no
  policy beats it;
* a hand-worked trace that separates LRU from FIFO.
"""
import itertools

import numpy as np
import pytest

import oracle

POLICIES = ("lru", "fifo", "random", "belady")


def _random_trace(rng, steps, K, ctx, reuse=0.6):
    rows, prev = [], None
    for _ in range(steps):
        if prev is None:
            cur = list(rng.choice(ctx, K, replace=False))
        else:
            keep = list(rng.choice(prev, int(reuse * K), replace=False))
            rest = [p for p in rng.permutation(ctx) if p not in keep][:K - len(keep)]
            cur = keep + rest
            rng.shuffle(cur)
        rows.append(cur)
        prev = cur
    return np.array(rows, dtype=np.int32)


def test_lru_matches_the_resolve_oracle():
    rng = np.random.default_rng(11)
    for K, B, ctx, steps in [(8, 16, 64, 30), (16, 16, 40, 20), (5, 12, 25, 40), (32, 64, 512, 25)]:
        tr = _random_trace(rng, steps, K, ctx)
        o = oracle.ResolveOracle(1, 1, K, B, B, [ctx], 1)  # page = B tokens: one hot block
        o.set_ctx(0, ctx)
        o.set_hot_block(0, 0, 0)
        ref = np.array([len(o.resolve(0, 0, tr[t], t)[1]) for t in range(steps)])
        np.testing.assert_array_equal(oracle.policy_misses("lru", tr, B, ctx), ref)


def test_b_equal_k_every_policy_coincides():
    rng = np.random.default_rng(3)
    tr = _random_trace(rng, 40, 12, 100)
    want = [12] + [len(set(tr[t]) - set(tr[t - 1])) for t in range(1, 40)]
    for pol in POLICIES:
        np.testing.assert_array_equal(oracle.policy_misses(pol, tr, 12, 100, seed=5), want, pol)


def test_b_at_least_context_only_compulsory_misses():
    rng = np.random.default_rng(4)
    tr = _random_trace(rng, 30, 6, 20)
    seen, want = set(), []
    for row in tr:
        new = set(row) - seen
        want.append(len(new))
        seen |= new
    for pol in POLICIES:
        np.testing.assert_array_equal(oracle.policy_misses(pol, tr, 20, 20, seed=9), want, pol)


def _optimum(trace, B):
    """Fewest total misses over every choice of victims (resident sets only;
    filling an empty slot before evicting is never worse)."""
    best = [None]

    def go(t, resident, total):
        if best[0] is not None and total >= best[0]:
            return
        if t == len(trace):
            best[0] = total
            return
        sel = list(dict.fromkeys(int(p) for p in trace[t] if p >= 0))
        miss = [p for p in sel if p not in resident]
        free = B - len(resident)
        evictable = sorted(resident - set(sel))
        need = max(0, len(miss) - free)
        for out in itertools.combinations(evictable, need):
            go(t + 1, (resident - set(out)) | set(miss), total + len(miss))

    go(0, frozenset(), 0)
    return best[0]


def test_belady_is_optimal_on_tiny_traces():
    rng = np.random.default_rng(8)
    for _ in range(300):
        ctx = int(rng.integers(3, 7))
        K = int(rng.integers(1, 3))
        B = int(rng.integers(K, 5))
        steps = int(rng.integers(2, 6))
        tr = np.array([rng.choice(ctx, K, replace=False) for _ in range(steps)], dtype=np.int32)
        opt = _optimum(tr, B)
        got = {pol: int(oracle.policy_misses(pol, tr, B, ctx, seed=1).sum()) for pol in POLICIES}
        assert got["belady"] == opt, (tr.tolist(), B, got, opt)
        assert all(v >= opt for v in got.values()), (tr.tolist(), B, got, opt)


def test_hand_worked_lru_and_fifo_differ():
    # B = 2, K = 1, selections a, b, a, c, a (a=0, b=1, c=2).  At step 3, c
    # misses and both slots are candidates: LRU evicts b (last used at step 1,
    # a at step 2), so step 4's a hits; FIFO evicts a (loaded at step 0, b at
    # step 1), so step 4's a misses; Belady evicts b (never used again).
    tr = np.array([[0], [1], [0], [2], [0]], dtype=np.int32)
    assert oracle.policy_misses("lru", tr, 2, 3).tolist() == [1, 1, 0, 1, 0]
    assert oracle.policy_misses("fifo", tr, 2, 3).tolist() == [1, 1, 0, 1, 1]
    assert oracle.policy_misses("belady", tr, 2, 3).tolist() == [1, 1, 0, 1, 0]


def test_random_is_seeded_and_valid():
    rng = np.random.default_rng(6)
    tr = _random_trace(rng, 30, 8, 60)
    a = oracle.policy_misses("random", tr, 16, 60, seed=123)
    b = oracle.policy_misses("random", tr, 16, 60, seed=123)
    np.testing.assert_array_equal(a, b)
    assert a.sum() >= oracle.policy_misses("belady", tr, 16, 60).sum()


def test_bad_arguments_are_rejected():
    with pytest.raises(ValueError):
        oracle.policy_misses("lru", np.zeros((2, 2), dtype=np.int32), 0, 4)
