"""The allocation-free decode entry point, for callers that cannot allocate
device memory while they decode (all HBM pre-reserved, an allocator that
forbids new allocations, a plug-in given only raw pointers).

It must give the same result as the pool-based call, within the attention
tolerance of the other tests, on consecutive calls that reuse its fixed
scratch.  This file is collected last so that a stop-at-first-failure run has
already run every other test."""
import numpy as np
import pytest

import synth
from synth import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import sparse_attention_kv_hs_gb300 as hs  # noqa: E402

MAX_ABS, MEAN_REL = 1e-2, 2e-3


def _close(a, b):
    a = a.astype(np.float64)
    b = b.astype(np.float64)
    err = np.abs(a - b)
    assert err.max() <= MAX_ABS, err.max()
    assert err.sum() <= MEAN_REL * np.abs(b).sum(), err.sum() / np.abs(b).sum()


@pytest.mark.parametrize("R,K,H", [(32, 2048, 128), (1, 256, 16), (3, 1000, 100)])
def test_noalloc_matches_pool_call_on_consecutive_calls(R, K, H):
    P = 256
    pool = hs.Pool(R, 1, K, P, P, W.ROW_ELEMS, 1, P * R, 16)
    n = pool.blocks_per_layer * P
    rows = synth.rows(777, 0, 0, 0, n)
    pool.kv_pool[0].copy_(torch.from_numpy(rows.view(np.int16)).cuda())
    kv = pool.kv_pool[0]
    rng = np.random.default_rng(R * 131 + K)
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
        _close(got.float().cpu().numpy(), ref.float().cpu().numpy())
        assert np.allclose(lse_got.cpu().numpy(), lse_ref.cpu().numpy(), atol=1e-4)
    assert hs.hs_check_errors(pool.handle) == 0
    pool.close()


def test_noalloc_rejects_more_partials_than_its_scratch_holds():
    # K = 8192 needs at least 4 splits; 20 requests x 4 > 64 partials
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    with pytest.raises(hs.HsError) as e:
        hs.hs_sparse_mla_decode_noalloc(dummy, 16, dummy, dummy, 20, 8192, 128, W.V_DIM, W.SCALE,
                                        dummy)
    assert e.value.status == hs.HS_ERR_INVALID
