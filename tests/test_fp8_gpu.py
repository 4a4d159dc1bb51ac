"""FP8 KV rows (656 bytes, HS_KV_FP8) on the GPU against the CPU oracle.

RESOLVE, the row gather, page loads and prefix offload move rows as opaque
bytes, so with an FP8 pool the row ids are still bit-exact against the oracle
and every gathered or offloaded row is byte-identical to the generator's FP8
row at that position.

Attention on FP8 rows is checked against the fp64 oracle over the values the
rows stand for (E4M3 code x group scale; rope bf16), with the bf16 path's
tolerance: max-abs <= 1e-2, mean-rel <= 2e-3.  The kernel rounds each latent
value (the group scale rounded to fp16, then E4M3 x scale in fp16: at most
2 x 2^-11 relative) and Q (2^-11) to fp16 before the MMAs; averaged over the
rows that is well below the bf16 output rounding (~1.4e-3 mean-rel) the bound
is set by."""
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

FP8 = 1
UNITS = synth.FP8_ROW_BYTES // 2  # a row in 2-byte units
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


def _fp8_page(w, r, l, page):
    return torch.from_numpy(synth.rows_fp8(w.seed, r, l, page * w.P, w.P).view(np.int16))


def replay_fp8(w, gather_every=1, attn_steps=()):
    scen = W.Scenario.build(w)
    pool = harness.make_pool(w, scen, kv_format=FP8)
    o = harness.make_oracle(w, scen)
    tr = harness.traces(w)
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    R, K, L = w.R, w.K, w.L
    d_topk = torch.empty((R, K), dtype=torch.int32, device="cuda")
    d_out = torch.empty((R, K), dtype=torch.int32, device="cuda")
    d_rows = torch.empty((R * K, UNITS), dtype=torch.int16, device="cuda")
    offs = w.host_offsets()
    ctx = w.ctx.astype(np.int64).copy()
    events, appended = {}, []
    for t in range(w.steps):
        for (r, page, blk) in scen.flips[t]:
            ev = events.pop((r, page), None)
            if ev is not None:
                hs.hs_commit_offload(pool.handle, r, page, stream, ev)
            else:
                hs.hs_map_page(pool.handle, r, page, -1, stream)
            o.set_page(r, page, -1)
        for l in range(L):
            d_topk.copy_(torch.from_numpy(tr[t, l]))
            hs.hs_resolve(pool.handle, l, 1, d_topk, pool.step, d_out)
            out = d_out.cpu().numpy()
            for r in range(R):
                ref_rows, _, err = o.resolve(l, r, tr[t, l, r], t)
                assert err == 0
                np.testing.assert_array_equal(out[r], ref_rows, err_msg=f"t={t} l={l} r={r}")
            if t % gather_every == 0:
                hs.hs_gather(pool.handle, l, d_out, R * K, d_rows, stream)
                got = d_rows.view(R, K, UNITS).cpu().numpy().view(np.uint8)
                for r in range(R):
                    want = synth.rows_fp8_at(w.seed, r, l, tr[t, l, r])
                    np.testing.assert_array_equal(got[r], want, err_msg=f"t={t} l={l} r={r}")
            if t in attn_steps:
                q = np.stack([synth.q(w.seed, r, l, t, w.heads) for r in range(R)])
                o_gpu, lse = _decode(pool, l, q, d_out, w.heads)
                for r in range(R):
                    kv = harness.rows_for_oracle(w, r, l, tr[t, l, r], FP8)
                    ref, ref_lse = oracle.sparse_mla_decode(q[r], kv, None, W.SCALE)
                    _check(o_gpu[r], ref, (t, l, r))
                    assert np.allclose(lse[r], ref_lse, rtol=0, atol=2e-3)
        hs.hs_step_advance(pool.step, stream)
        for (r, page, blk) in scen.appends[t]:
            for l in range(L):
                pool.kv_pool[l, blk * w.P:(blk + 1) * w.P].copy_(_fp8_page(w, r, l, page))
            hs.hs_map_page(pool.handle, r, page, blk, stream)
            ev = torch.cuda.Event()
            hs.hs_offload_prefix(pool.handle, r, page, stream, side, ev)
            events[(r, page)] = ev
            ctx[r] += w.P
            hs.hs_set_request(pool.handle, r, int(ctx[r]), int(offs[r]), stream)
            o.set_page(r, page, blk)
            o.set_ctx(r, int(ctx[r]))
            appended.append((r, page))
    torch.cuda.synchronize()
    assert hs.hs_check_errors(pool.handle) == 0
    for (r, page) in appended:  # the offload wrote the FP8 bytes to the host pool
        for l in range(L):
            base = int(offs[r]) + page * w.P
            got = pool.host_pool[l, base:base + w.P].view(np.uint8)
            np.testing.assert_array_equal(got, synth.rows_fp8(w.seed, r, l, page * w.P, w.P))
    pool.close()


def test_fp8_attention_workload_scaled_down():
    replay_fp8(W.make("attention", R=4, steps=6), attn_steps={0, 5})


def test_fp8_attention_workload_full_size():
    """32 requests x 2 layers, ctx 65536, K 2048, B 4096, 128 heads; attention
    on steps 0 and 3 for every (request, layer)."""
    replay_fp8(W.make("attention", steps=4), gather_every=4, attn_steps={0, 3})


def test_fp8_resolve_workload_with_resident_tail():
    replay_fp8(W.make("resolve", R=4, steps=8), gather_every=2)


def test_fp8_mixed_residency_with_offload():
    replay_fp8(W.make("mixed", R=16, steps=12, ctx_hi=131072), gather_every=3, attn_steps={11})


def test_fp8_pool_needs_576_wide_rows():
    with pytest.raises(hs.HsError):
        hs.Pool(1, 1, 64, 256, 256, 512, 4, 1024, 1, FP8)


# ------------------------------------------------------------------ attention edge cases

def _fp8_pool_with_rows(K, R=1, blocks=8, P=256):
    """An FP8 pool whose resident blocks hold seeded rows; returns (pool, raw rows)."""
    pool = hs.Pool(R, 1, K, P, P, W.ROW_ELEMS, 1, P * R, blocks, FP8)
    raw = synth.rows_fp8(4242, 0, 0, 0, pool.blocks_per_layer * P)
    pool.kv_pool[0].copy_(torch.from_numpy(raw.view(np.int16)).cuda())
    torch.cuda.synchronize()
    return pool, raw


@pytest.mark.parametrize("K,H", [(100, 128), (64, 16), (1000, 1), (65, 100), (2048, 128)])
def test_fp8_ragged_k_and_head_counts_with_padding(K, H):
    R = 3
    pool, raw = _fp8_pool_with_rows(K, R=R, blocks=16)
    rows = oracle.fp8_rows_to_f64(raw)
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


def test_fp8_single_row_returns_its_latent_values():
    """One row: the output is that row's first 512 values (E4M3 x scale), to
    the rounding of the fp16 operand (the scale rounded to fp16, then the
    product: 2 x 2^-11 relative) and of the bf16 output (2^-8 relative)."""
    pool, raw = _fp8_pool_with_rows(1, R=2)
    ids = np.array([[5], [77]], dtype=np.int32)
    q = np.stack([synth.q(3, r, 0, 0, 128) for r in range(2)])
    got, _ = _decode(pool, 0, q, ids, 128)
    rows = oracle.fp8_rows_to_f64(raw)
    for r in range(2):
        want = np.broadcast_to(rows[ids[r, 0], :512], (128, 512))
        assert np.all(np.abs(got[r] - want) <= np.abs(want) * (2.0 ** -8 + 2.0 ** -9) + 2.0 ** -24)
    assert hs.hs_check_errors(pool.handle) == 0
    pool.close()


def test_fp8_scale_past_the_fp16_range_is_flagged():
    """A group scale that takes code x scale past fp16's range raises the
    VALUE error bit (the operand cannot be represented)."""
    pool, raw = _fp8_pool_with_rows(64)
    raw = raw.copy()
    raw[10, 512:516] = np.array([1000.0], dtype=np.float32).view(np.uint8)  # 448 x 1000
    pool.kv_pool[0].copy_(torch.from_numpy(raw.view(np.int16)).cuda())
    ids = np.arange(64, dtype=np.int32)[None]
    q = synth.q(3, 0, 0, 0, 128)[None]
    _decode(pool, 0, q, ids, 128)
    assert hs.hs_check_errors(pool.handle) == hs.DEV_ERR_VALUE
    pool.close()


def test_fp8_query_past_the_fp16_range_is_flagged():
    pool, _ = _fp8_pool_with_rows(64)
    ids = np.arange(64, dtype=np.int32)[None]
    q = synth.q(3, 0, 0, 0, 128)[None].copy()
    q[0, 7, 100] = 0x4790                                 # bf16 73728
    _decode(pool, 0, q, ids, 128)
    assert hs.hs_check_errors(pool.handle) == hs.DEV_ERR_VALUE
    pool.close()


def test_fp8_small_scales_take_the_fp32_products():
    """Group scales below fp16's normal range (2^-14) are formed as fp32
    products; rows of both kinds in one call match the oracle."""
    pool, raw = _fp8_pool_with_rows(200, R=2)
    raw = raw.copy()
    sc = raw[:, 512:528].copy().view(np.float32)
    sc[::3] *= np.float32(2.0 ** -12)                    # every third row: scales ~1e-6
    raw[:, 512:528] = sc.view(np.uint8)
    pool.kv_pool[0].copy_(torch.from_numpy(raw.view(np.int16)).cuda())
    rows = oracle.fp8_rows_to_f64(raw)
    rng = np.random.default_rng(11)
    ids = np.stack([rng.choice(rows.shape[0], 200, replace=False) for _ in range(2)])
    ids = ids.astype(np.int32)
    q = np.stack([synth.q(5, r, 0, 0, 128) for r in range(2)])
    got, lse = _decode(pool, 0, q, ids, 128)
    for r in range(2):
        ref, ref_lse = oracle.sparse_mla_decode(q[r], rows[ids[r]], None, W.SCALE)
        _check(got[r], ref, r)
        assert np.allclose(lse[r], ref_lse, rtol=0, atol=2e-3)
    assert hs.hs_check_errors(pool.handle) == 0
    pool.close()
