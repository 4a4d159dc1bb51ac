"""The seeded input generator: determinism, value encoding and the structure
of the selection traces (drift, layer sharing, no repeats)."""
import numpy as np

import synth
from synth import workloads as W


def test_rows_are_deterministic_and_position_addressed():
    a = synth.rows(11, 2, 1, 100, 50)
    b = synth.rows(11, 2, 1, 0, 200, threads=4)[100:150]
    c = synth.rows_at(11, 2, 1, np.arange(100, 150))
    assert np.array_equal(a, b) and np.array_equal(a, c)
    assert not np.array_equal(a, synth.rows(11, 2, 0, 100, 50))
    assert np.all(synth.rows_at(11, 2, 1, [-1]) == 0)


def test_normal_encoding_by_hand():
    # A draw whose four 16-bit fields sum to the mean gives +0.0.
    d = (0x7FFF << 48) | (0x8000 << 32) | (0x7FFF << 16) | 0x8000
    assert synth.normal_bf16(d) == 0x0000
    # All fields at 0xFFFF: s = 131070 -> 131070 / 37837.227 = 3.4640...,
    # bf16 of 3.4640 is 0x405e (3.46875).
    assert synth.normal_bf16(2**64 - 1) == 0x405E
    # All zero: the negative of the above.
    assert synth.normal_bf16(0) == 0xC05E


def test_row_statistics():
    x = synth.bf16_to_f32(synth.rows(5, 0, 0, 0, 4000))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01


def test_permutation_is_a_bijection():
    for n in (1, 7, 64, 1000, 4097):
        got = sorted(synth.permute(9, 3, i, n) for i in range(n))
        assert got == list(range(n))


def test_trace_structure_resolve_workload():
    w = W.make("resolve", R=1, steps=40)
    tr = w.trace(0)
    K = w.K
    for t in range(w.steps):
        for l in range(w.L):
            assert len(set(tr[t, l].tolist())) == K
            assert tr[t, l].min() >= 0 and tr[t, l].max() < w.ctx[0]
    # layer l > 0 shares >= 80% with layer l-1 at the same step
    share = [len(set(tr[t, l]) & set(tr[t, l - 1])) / K
             for t in range(w.steps) for l in range(1, w.L)]
    assert min(share) >= 0.8
    # layer 0 keeps >= 70% of its previous step
    keep = [len(set(tr[t, 0]) & set(tr[t - 1, 0])) / K for t in range(1, w.steps)]
    assert min(keep) >= 0.7 and np.mean(keep) < 0.8
    # Zipf share: some positions recur far more often than uniform draws would
    counts = np.bincount(tr[:, 0].reshape(-1), minlength=int(w.ctx[0]))
    assert counts.max() >= w.steps  # the head of the Zipf law is selected every step


def test_mixed_workload_scenario_is_consistent():
    w = W.make("mixed", R=16, steps=12, ctx_hi=65536)
    s = W.Scenario.build(w)
    assert w.appends_per_step == 1
    assert sorted(set(w.residency)) == ["full", "mixed", "zero"]
    live = {(r, p): b for (r, p, b) in s.initial}
    for t in range(w.steps):
        for (r, p, b) in s.flips[t]:
            assert live.pop((r, p)) == b
        for (r, p, b) in s.appends[t]:
            assert (r, p) not in live and b not in live.values()
            live[(r, p)] = b
        assert len(set(live.values())) == len(live)
        assert all(b < s.blocks_per_layer for b in live.values())
        assert all(b >= w.R * w.hot_blocks_per_request() for b in live.values())


def test_spec_token_traces():
    """Verify-token traces: token 0 is the plain trace; token t > 0 keeps
    floor(0.85 K) of token t-1's positions, never repeats one within a token,
    stays inside the context, and is reproducible."""
    w = W.make("spec", R=2, steps=5)
    for r in range(2):
        tt = w.trace_tokens(r)
        assert tt.shape == (5, w.L, w.tokens, w.K)
        np.testing.assert_array_equal(tt[:, :, 0], w.trace(r))
        keep = int(w.token_share * w.K)
        for t in range(5):
            for l in range(w.L):
                for k in range(1, w.tokens):
                    row, prev = tt[t, l, k], tt[t, l, k - 1]
                    assert len(set(row.tolist())) == w.K
                    assert row.min() >= 0 and row.max() < int(w.ctx[r])
                    assert len(set(row.tolist()) & set(prev.tolist())) >= keep
        np.testing.assert_array_equal(tt, w.trace_tokens(r))
