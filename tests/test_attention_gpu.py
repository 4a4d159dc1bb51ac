"""Sparse MLA decode attention on the GPU against the fp64 oracle.

Tolerance (stated for this path): max-abs <= 1e-2 and mean-rel <= 2e-3, where
mean-rel = sum|o_gpu - o_ref| / sum|o_ref| over all outputs of a call.  The
output is bf16, whose rounding alone costs ~1.4e-3 mean-rel on these inputs.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from synth import workloads as W
from tests import harness

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import sparse_attention_kv_hs_gb300 as hs  # noqa: E402

MAX_ABS, MEAN_REL = 1e-2, 2e-3


def _check(got, ref, what=""):
    err = np.abs(got.astype(np.float64) - ref)
    max_abs = float(err.max()) if err.size else 0.0
    denom = float(np.abs(ref).sum())
    mean_rel = float(err.sum() / denom) if denom > 0 else float(err.sum())
    assert max_abs <= MAX_ABS and mean_rel <= MEAN_REL, (what, max_abs, mean_rel)
    return max_abs, mean_rel


def _decode(pool, layer, q_bits, row_ids, heads):
    R = q_bits.shape[0]
    d_q = torch.from_numpy(q_bits.view(np.int16)).cuda()
    d_rows = row_ids if torch.is_tensor(row_ids) else torch.from_numpy(row_ids).cuda()
    out = torch.empty((R, heads, W.V_DIM), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((R, heads), dtype=torch.float32, device="cuda")
    hs.hs_sparse_mla_decode(pool.handle, layer, d_q, d_rows, heads, W.V_DIM, W.SCALE, out, lse)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def replay_with_attention(w, check_steps):
    scen = W.Scenario.build(w)
    pool = harness.make_pool(w, scen)
    o = harness.make_oracle(w, scen)
    tr = harness.traces(w)
    R, K, L, H = w.R, w.K, w.L, w.heads
    d_topk = torch.empty((R, K), dtype=torch.int32, device="cuda")
    d_out = [torch.empty((R, K), dtype=torch.int32, device="cuda") for _ in range(L)]
    worst = (0.0, 0.0)
    for t in range(w.steps):
        for l in range(L):
            d_topk.copy_(torch.from_numpy(tr[t, l]))
            hs.hs_resolve(pool.handle, l, 1, d_topk, pool.step, d_out[l])
            refs = []
            for r in range(R):
                ref_rows, _, err = o.resolve(l, r, tr[t, l, r], t)
                assert err == 0
                refs.append(ref_rows)
            np.testing.assert_array_equal(d_out[l].cpu().numpy(), np.stack(refs))
            if t in check_steps:
                q = np.stack([synth.q(w.seed, r, l, t, H) for r in range(R)])
                got, lse = _decode(pool, l, q, d_out[l], H)
                for r in range(R):
                    rows = synth.rows_at(w.seed, r, l, tr[t, l, r])
                    ref, ref_lse = oracle.sparse_mla_decode(q[r], rows, None, W.SCALE)
                    m = _check(got[r], ref, (t, l, r))
                    worst = (max(worst[0], m[0]), max(worst[1], m[1]))
                    assert np.allclose(lse[r], ref_lse, rtol=0, atol=2e-3)
        hs.hs_step_advance(pool.step)
    assert hs.hs_check_errors(pool.handle) == 0
    pool.close()
    return worst


def test_tiny_workload_attention_every_step():
    """1 request, 16 heads, K 256: several K splits and the merge path."""
    w = W.make("tiny")
    replay_with_attention(w, check_steps=set(range(w.steps)))


def test_attention_workload_scaled_down():
    w = W.make("attention", R=4, steps=6)
    replay_with_attention(w, check_steps={0, 1, 5})


def test_attention_workload_full_size():
    """32 requests x 2 layers, ctx 65536, K 2048, B 4096, 128 heads, 64 steps;
    attention checked on steps 0, 1 and 63 for every (request, layer)."""
    w = W.make("attention")
    worst = replay_with_attention(w, check_steps={0, 1, 63})
    print("worst max_abs %.3g mean_rel %.3g" % worst)


# ------------------------------------------------------------------ edge cases

def _pool_with_rows(K, R=1, blocks=8, P=256):
    """A pool whose resident blocks hold seeded rows; returns (pool, kv rows)."""
    pool = hs.Pool(R, 1, K, P, P, W.ROW_ELEMS, 1, P * R, blocks)
    rows = synth.rows(4242, 0, 0, 0, pool.blocks_per_layer * P)
    pool.kv_pool[0].copy_(torch.from_numpy(rows.view(np.int16)).cuda())
    torch.cuda.synchronize()
    return pool, rows


@pytest.mark.parametrize("K,H", [(100, 128), (64, 16), (1000, 1), (65, 100), (2048, 128)])
def test_ragged_k_and_head_counts_with_padding(K, H):
    R = 3
    pool, rows = _pool_with_rows(K, R=R, blocks=16)
    n = rows.shape[0]
    rng = np.random.default_rng(K * 7 + H)
    ids = np.stack([rng.choice(n, K, replace=False) for _ in range(R)]).astype(np.int32)
    ids[0, rng.choice(K, K // 5, replace=False)] = -1     # padding rows are excluded
    q = np.stack([synth.q(9, r, 0, 0, H) for r in range(R)])
    got, lse = _decode(pool, 0, q, ids, H)
    for r in range(R):
        valid = ids[r] >= 0
        ref, ref_lse = oracle.sparse_mla_decode(q[r], rows[np.maximum(ids[r], 0)], valid, W.SCALE)
        _check(got[r], ref, (K, H, r))
        assert np.allclose(lse[r], ref_lse, rtol=0, atol=2e-3)
    assert hs.hs_check_errors(pool.handle) == 0
    pool.close()


def test_single_row_returns_that_row_exactly():
    pool, rows = _pool_with_rows(1, R=2)
    ids = np.array([[5], [77]], dtype=np.int32)
    q = np.stack([synth.q(3, r, 0, 0, 128) for r in range(2)])
    got, _ = _decode(pool, 0, q, ids, 128)
    for r in range(2):
        v = synth.bf16_to_f32(rows[ids[r, 0], :512])
        assert np.array_equal(got[r], np.broadcast_to(v, got[r].shape))
    pool.close()


def test_identical_rows_and_zero_query():
    pool, rows = _pool_with_rows(256)
    ids = np.full((1, 256), 9, dtype=np.int32)             # the same row 256 times
    q = synth.q(4, 0, 0, 0, 128)[None]
    got, lse = _decode(pool, 0, q, ids, 128)
    v = synth.bf16_to_f32(rows[9, :512])
    assert np.array_equal(got[0], np.broadcast_to(v, got[0].shape))
    ids2 = np.arange(256, dtype=np.int32)[None]
    q0 = np.zeros((1, 128, W.ROW_ELEMS), dtype=np.uint16)  # q = 0: mean of the rows
    got2, lse2 = _decode(pool, 0, q0, ids2, 128)
    mean = synth.bf16_to_f32(rows[:256, :512]).astype(np.float64).mean(axis=0)
    _check(got2[0], np.broadcast_to(mean, got2[0].shape))
    assert np.allclose(lse2, math.log(256), atol=1e-4)
    pool.close()


def test_no_valid_row_gives_zero_and_minus_inf():
    pool, rows = _pool_with_rows(128, R=2)
    ids = np.full((2, 128), -1, dtype=np.int32)
    ids[1, :3] = [1, 2, 3]
    q = np.stack([synth.q(5, r, 0, 0, 128) for r in range(2)])
    got, lse = _decode(pool, 0, q, ids, 128)
    assert np.all(got[0] == 0) and np.all(np.isneginf(lse[0]))
    ref, _ = oracle.sparse_mla_decode(q[1], rows[[1, 2, 3]], None, W.SCALE)
    _check(got[1], ref)
    pool.close()


def test_out_of_pool_row_ids_are_excluded_and_flagged():
    pool, rows = _pool_with_rows(64)
    n = pool.blocks_per_layer * 256
    ids = np.arange(64, dtype=np.int32)[None].copy()
    ids[0, 10] = n + 5
    q = synth.q(6, 0, 0, 0, 128)[None]
    got, _ = _decode(pool, 0, q, ids, 128)
    valid = np.ones(64, bool)
    valid[10] = False
    ref, _ = oracle.sparse_mla_decode(q[0], rows[np.minimum(ids[0], n - 1)], valid, W.SCALE)
    _check(got[0], ref)
    assert hs.hs_check_errors(pool.handle) == hs.DEV_ERR_BLOCK
    pool.close()


def _bf16_bits(x):
    """float values -> bf16 bit patterns (round to nearest even)."""
    f = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((f + 0x7FFF + ((f >> 16) & 1)) >> 16).astype(np.uint16)


def _zero_query_mean(pool, n):
    """q = 0: every score is 0, so the output is the mean of the n rows' value columns."""
    ids = np.arange(n, dtype=np.int32)[None]
    q0 = np.zeros((1, 128, W.ROW_ELEMS), dtype=np.uint16)
    got, _ = _decode(pool, 0, q0, ids, 128)
    return got[0]


def test_value_columns_at_the_fp16_range_edges():
    """P.V runs in fp16: bf16 values up to 65280 in magnitude and down to 2^-24
    (fp16 subnormals) are carried exactly; the mean over the rows comes out
    within bf16 rounding of the fp64 mean (plus fp32 accumulation for the large
    values)."""
    rng = np.random.default_rng(11)
    cases = [
        (rng.choice([-65280.0, 65280.0, -40000.0, 32768.0, 1.5], size=(32, 512)), 65280.0 * 2.0 ** -20),
        (rng.choice([-2.0 ** -20, 2.0 ** -20, 3 * 2.0 ** -18, 2.0 ** -24], size=(32, 512)), 0.0),
    ]
    for vals, slack in cases:
        pool, rows = _pool_with_rows(32)
        rows = rows[:32].copy()
        rows[:, :512] = _bf16_bits(vals)
        pool.kv_pool[0][:32].copy_(torch.from_numpy(rows.view(np.int16)).cuda())
        got = _zero_query_mean(pool, 32)
        ref = synth.bf16_to_f32(rows[:, :512]).astype(np.float64).mean(axis=0)
        err = np.abs(got - ref)
        assert np.all(err <= np.abs(ref) * 2.0 ** -8 + slack), float(err.max())
        assert hs.hs_check_errors(pool.handle) == 0
        pool.close()


@pytest.mark.parametrize("bits", [0x4780, 0xC780, 0x7F80, 0xFF80, 0x7FC0])
def test_value_outside_fp16_range_is_flagged(bits):
    """A value element of magnitude >= 65536 (or inf / NaN) sets error bit VALUE."""
    pool, rows = _pool_with_rows(64)
    rows = rows[:64].copy()
    rows[7, 100] = bits
    pool.kv_pool[0][:64].copy_(torch.from_numpy(rows.view(np.int16)).cuda())
    _zero_query_mean(pool, 64)
    assert hs.hs_check_errors(pool.handle) == hs.DEV_ERR_VALUE
    pool.close()


def test_rope_columns_are_not_range_checked():
    """Columns 512..575 only enter the scores (bf16 x bf16 -> fp32), not P.V."""
    pool, rows = _pool_with_rows(64)
    rows = rows[:64].copy()
    rows[7, 520] = 0x4780  # 65536 in a rope column
    pool.kv_pool[0][:64].copy_(torch.from_numpy(rows.view(np.int16)).cuda())
    got = _zero_query_mean(pool, 64)
    ref = synth.bf16_to_f32(rows[:, :512]).astype(np.float64).mean(axis=0)
    _check(np.broadcast_to(got, (128, 512)), np.broadcast_to(ref, (128, 512)))
    assert hs.hs_check_errors(pool.handle) == 0
    pool.close()


def test_graph_captured_decode_step():
    """RESOLVE + attention of one layer captured once and replayed per step."""
    w = W.make("attention", R=2, L=1, steps=5)
    scen = W.Scenario.build(w)
    pool = harness.make_pool(w, scen)
    o = harness.make_oracle(w, scen)
    tr = harness.traces(w)
    H = w.heads
    d_topk = torch.empty((w.R, w.K), dtype=torch.int32, device="cuda")
    d_rows = torch.empty((w.R, w.K), dtype=torch.int32, device="cuda")
    d_q = torch.empty((w.R, H, W.ROW_ELEMS), dtype=torch.int16, device="cuda")
    d_o = torch.empty((w.R, H, W.V_DIM), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            hs.hs_resolve(pool.handle, 0, 1, d_topk, pool.step, d_rows, None, None, s)
            hs.hs_sparse_mla_decode(pool.handle, 0, d_q, d_rows, H, W.V_DIM, W.SCALE, d_o, None, s)
            hs.hs_step_advance(pool.step, s)
    for t in range(w.steps):
        q = np.stack([synth.q(w.seed, r, 0, t, H) for r in range(w.R)])
        d_topk.copy_(torch.from_numpy(tr[t, 0]))
        d_q.copy_(torch.from_numpy(q.view(np.int16)))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        got = d_o.float().cpu().numpy()
        for r in range(w.R):
            ref_rows, _, _ = o.resolve(0, r, tr[t, 0, r], t)
            np.testing.assert_array_equal(d_rows[r].cpu().numpy(), ref_rows)
            ref, _ = oracle.sparse_mla_decode(q[r], synth.rows_at(w.seed, r, 0, tr[t, 0, r]), None,
                                              W.SCALE)
            _check(got[r], ref, (t, r))
    pool.close()
