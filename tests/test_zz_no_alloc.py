"""The allocation-free decode entry point, for callers that cannot allocate
device memory while they decode (all HBM pre-reserved, an allocator that
forbids new allocations, a plug-in given only raw pointers).

Each call is checked against the fp64 oracle within the attention tolerance
of the other tests (max-abs 1e-2, mean-rel 2e-3; lse 2e-3) and against the
pool-based call, on consecutive calls that reuse its fixed scratch; the shapes
reach every branch of its split choice (its usual split count, a count cut
down to fit the scratch, one split when even two do not fit, and one split
with no scratch at all).  Its device errors are read through its own error
word.  This file is collected last so that a stop-at-first-failure run has
already run every other test."""
import numpy as np
import pytest

import oracle
import synth
from synth import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import sparse_attention_kv_hs_gb300 as hs  # noqa: E402

MAX_ABS, MEAN_REL = 1e-2, 2e-3


def _close(a, b, what=""):
    a = a.astype(np.float64)
    b = b.astype(np.float64)
    err = np.abs(a - b)
    assert err.max() <= MAX_ABS, (what, err.max())
    assert err.sum() <= MEAN_REL * np.abs(b).sum(), (what, err.sum() / np.abs(b).sum())


def _pool_rows(R, K, seed=777):
    P = 256
    pool = hs.Pool(R, 1, K, P, P, W.ROW_ELEMS, 1, P * R, -(-R * K // P) + 16)
    n = pool.blocks_per_layer * P
    rows = synth.rows(seed, 0, 0, 0, n)
    pool.kv_pool[0].copy_(torch.from_numpy(rows.view(np.int16)).cuda())
    return pool, rows, n


# (R, K, H): 2 splits as the pool call; 3 wanted, cut to 2 (24 x 3 > 64);
# 2 wanted, cut to 1 (33 x 2 > 64); 1 split, no scratch; small and ragged
@pytest.mark.parametrize("R,K,H", [(32, 2048, 128), (24, 4096, 128), (33, 2048, 128),
                                   (65, 512, 64), (1, 256, 16), (3, 1000, 100)])
def test_noalloc_matches_oracle_and_pool_call_on_consecutive_calls(R, K, H):
    pool, rows, n = _pool_rows(R, K)
    kv = pool.kv_pool[0]
    rng = np.random.default_rng(R * 131 + K)
    assert hs.hs_noalloc_check_errors() == 0  # starts clean (or a previous test left it so)
    for call in range(2):  # two calls in a row share the fixed scratch
        ids = np.stack([rng.choice(n, K, replace=False) for _ in range(R)]).astype(np.int32)
        ids[0, : K // 7] = -1
        q = np.stack([synth.q(5 + call, r, 0, 0, H) for r in range(R)])
        d_ids = torch.from_numpy(ids).cuda()
        d_q = torch.from_numpy(q.view(np.int16)).cuda()
        ref = torch.empty((R, H, W.V_DIM), dtype=torch.bfloat16, device="cuda")
        got = torch.empty_like(ref)
        lse_ref = torch.empty((R, H), dtype=torch.float32, device="cuda")
        lse_got = torch.empty_like(lse_ref)
        hs.hs_sparse_mla_decode(pool.handle, 0, d_q, d_ids, H, W.V_DIM, W.SCALE, ref, lse_ref)
        hs.hs_sparse_mla_decode_noalloc(kv, n, d_q, d_ids, R, K, H, W.V_DIM, W.SCALE, got, lse_got)
        torch.cuda.synchronize()
        g, gl = got.float().cpu().numpy(), lse_got.cpu().numpy()
        for r in range(R):
            valid = ids[r] >= 0
            o, o_lse = oracle.sparse_mla_decode(q[r], rows[np.maximum(ids[r], 0)], valid, W.SCALE)
            _close(g[r], o, (R, K, H, call, r))
            assert np.allclose(gl[r], o_lse, rtol=0, atol=2e-3), (R, K, H, call, r)
        _close(g, ref.float().cpu().numpy(), "against the pool call")
        assert np.allclose(gl, lse_ref.cpu().numpy(), atol=1e-4)
        assert hs.hs_noalloc_check_errors() == 0
    assert hs.hs_check_errors(pool.handle) == 0
    pool.close()


def test_noalloc_reports_device_errors_through_its_own_word():
    """A value column holding 65536 (outside what the fp16 P.V product takes)
    sets VALUE, a row id past the rows sets BLOCK; reading clears the word."""
    R, K, H = 2, 300, 128
    pool, rows, n = _pool_rows(R, K, seed=31)
    bad = rows[:R * K].copy()
    bad[5, 17] = 0x4780  # bf16 65536 in row 5, a value column
    pool.kv_pool[0][:R * K].copy_(torch.from_numpy(bad.view(np.int16)).cuda())
    kv = pool.kv_pool[0]
    ids = np.arange(R * K, dtype=np.int32).reshape(R, K)
    q = np.stack([synth.q(8, r, 0, 0, H) for r in range(R)])
    d_q = torch.from_numpy(q.view(np.int16)).cuda()
    out = torch.empty((R, H, W.V_DIM), dtype=torch.bfloat16, device="cuda")
    hs.hs_noalloc_check_errors()
    hs.hs_sparse_mla_decode_noalloc(kv, n, d_q, torch.from_numpy(ids).cuda(), R, K, H, W.V_DIM,
                                    W.SCALE, out)
    assert hs.hs_noalloc_check_errors() & hs.DEV_ERR_VALUE
    assert hs.hs_noalloc_check_errors() == 0  # cleared by the read
    ids2 = ids.copy()
    ids2[:, 5] = 6  # drop the bad row (a repeat is fine for attention)
    ids2[1, 9] = n + 3
    hs.hs_sparse_mla_decode_noalloc(kv, n, d_q, torch.from_numpy(ids2).cuda(), R, K, H, W.V_DIM,
                                    W.SCALE, out)
    assert hs.hs_noalloc_check_errors() == hs.DEV_ERR_BLOCK
    got = out.float().cpu().numpy()
    valid = ids2[1] < n
    o, _ = oracle.sparse_mla_decode(q[1], bad[np.minimum(ids2[1], R * K - 1)], valid, W.SCALE)
    _close(got[1], o, "bad id excluded")
    assert hs.hs_check_errors(pool.handle) == 0  # the pool's own word is untouched
    pool.close()


def test_noalloc_rejects_more_partials_than_its_scratch_holds():
    # K = 8192 needs at least 4 splits; 20 requests x 4 > 64 partials
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    with pytest.raises(hs.HsError) as e:
        hs.hs_sparse_mla_decode_noalloc(dummy, 16, dummy, dummy, 20, 8192, 128, W.V_DIM, W.SCALE,
                                        dummy)
    assert e.value.status == hs.HS_ERR_INVALID
