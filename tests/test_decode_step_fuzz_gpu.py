"""Randomised decode steps (hs_decode_step_tokens on two streams) against the
oracle.

Each case draws bf16 or FP8 rows, 1-4 requests, 1-4 sparse layers, one or
two verify tokens, K 64..1024, B of two to three K, random contexts and
resident pages (loaded from the host pool).  Every step, all layers' row ids
and miss counts must equal the oracle's, and the attention output of one
sampled (layer, request, token) must be within the stated tolerance of fp64
attention over the rows at the selected positions.  Both stream schedules
(bf16: the later layers' RESOLVE starts with layer 0's; FP8: after it) run
with their launches racing as they do in the benchmark."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import sparse_attention_kv_hs_gb300 as hs  # noqa: E402

ROW_ELEMS, V_DIM, SCALE, P = 576, 512, 192 ** -0.5, 256


def one_case(seed):
    rng = np.random.default_rng(7000 + seed)
    fp8 = bool(rng.random() < 0.5)
    R, L, T = int(rng.integers(1, 5)), int(rng.integers(1, 5)), int(rng.choice([1, 2]))
    K = int(rng.integers(64, 1025))
    H = int(rng.choice([16, 128]))
    B = P * -(-int(rng.integers(2 * K, 3 * K + 1)) // P)
    ctx = rng.integers(2 * T * K, 2 * T * K + 2048, size=R)
    max_pages = int(-(-int(ctx.max()) // P))
    host_off = np.concatenate([[0], np.cumsum(ctx)[:-1]]).astype(np.int64)
    resident = int(rng.integers(1, 5))
    seedrows = 8000 + seed
    pool = hs.Pool(R, L, K, B, P, ROW_ELEMS, max_pages, int(ctx.sum()), resident,
                   1 if fp8 else 0)
    for l in range(L):
        for r in range(R):
            n = int(ctx[r])
            dst = pool.host_pool[l, int(host_off[r]):int(host_off[r]) + n]
            if fp8:
                synth.rows_fp8_into(seedrows, r, l, 0, n, dst.ctypes.data, 8)
            else:
                synth.rows_into(seedrows, r, l, 0, n, ROW_ELEMS, dst.ctypes.data, 8)
    o = oracle.ResolveOracle(R, L, K, B, P, ctx, pool.blocks_per_layer)
    s = torch.cuda.current_stream()
    hot = B // P
    for r in range(R):
        hs.hs_set_request(pool.handle, r, int(ctx[r]), int(host_off[r]), s)
        o.set_ctx(r, int(ctx[r]))
        for i in range(hot):
            o.set_hot_block(r, i, r * hot + i)
    for blk in range(R * hot, pool.blocks_per_layer):
        r = int(rng.integers(R))
        if rng.random() < 0.7 and int(ctx[r]) >= P:
            page = int(rng.integers(int(ctx[r]) // P))                  # a whole page
            hs.hs_load_page(pool.handle, r, page, blk, s)
            o.set_page(r, page, blk)
    d_topk = torch.empty((L, R, T, K), dtype=torch.int32, device="cuda")
    d_q = torch.empty((L, R, T, H, ROW_ELEMS), dtype=torch.int16, device="cuda")
    d_rows = torch.empty((L, R, T, K), dtype=torch.int32, device="cuda")
    d_cnt = torch.empty((L, R), dtype=torch.int32, device="cuda")
    d_o = torch.empty((L, R, T, H, V_DIM), dtype=torch.bfloat16, device="cuda")
    d_lse = torch.empty((L, R, T, H), dtype=torch.float32, device="cuda")
    main, copy = torch.cuda.Stream(), torch.cuda.Stream()
    what = f"seed={seed} fp8={fp8} R={R} L={L} T={T} K={K} H={H} B={B}"
    for t in range(3):
        topk = np.empty((L, R, T, K), dtype=np.int32)
        for l in range(L):
            for r in range(R):
                sel = rng.choice(int(ctx[r]), T * K, replace=False).astype(np.int32)
                topk[l, r] = sel.reshape(T, K)
                if T == 2:                                   # token 1 repeats part of token 0
                    share = rng.random(K) < 0.6
                    topk[l, r, 1][share] = topk[l, r, 0][share]
        q = np.stack([np.stack([np.stack([synth.q(9000 + seed, r, l, t * T + k, H)
                                          for k in range(T)]) for r in range(R)])
                      for l in range(L)])
        d_topk.copy_(torch.from_numpy(topk))
        d_q.copy_(torch.from_numpy(q.view(np.int16)))
        torch.cuda.synchronize()
        with torch.cuda.stream(main):
            hs.hs_decode_step_tokens(pool.handle, 0, L, T, d_topk, d_q, H, V_DIM, SCALE,
                                     pool.step, d_rows, d_o, d_lse, d_cnt, main, copy)
            hs.hs_step_advance(pool.step, main)
        torch.cuda.synchronize()
        rows, cnt = d_rows.cpu().numpy(), d_cnt.cpu().numpy()
        for l in range(L):
            for r in range(R):
                ref_rows, ref_log, err = o.resolve_tokens(l, r, topk[l, r], t)
                assert err == 0, what
                np.testing.assert_array_equal(rows[l, r], np.asarray(ref_rows).reshape(T, K),
                                              err_msg=f"{what} t={t} l={l} r={r}")
                assert cnt[l, r] == len(ref_log), (what, t, l, r)
        l, r, k = int(rng.integers(L)), int(rng.integers(R)), int(rng.integers(T))
        pos = topk[l, r, k]
        kv = (oracle.fp8_rows_to_f64(synth.rows_fp8_at(seedrows, r, l, pos)) if fp8
              else synth.rows_at(seedrows, r, l, pos))
        ref, ref_lse = oracle.sparse_mla_decode(q[l, r, k], kv, None, SCALE)
        got = d_o[l, r, k].float().cpu().numpy()
        err = np.abs(got.astype(np.float64) - ref)
        mean_rel = err.sum() / np.abs(ref).sum()
        assert err.max() <= 1e-2 and mean_rel <= 2e-3, (what, t, l, r, k, err.max(), mean_rel)
        assert np.allclose(d_lse[l, r, k].cpu().numpy(), ref_lse, rtol=0, atol=2e-3), what
    assert hs.hs_check_errors(pool.handle) == 0, what
    pool.close()
    o.close()


@pytest.mark.parametrize("seed", range(24))
def test_random_decode_steps(seed):
    one_case(seed)
