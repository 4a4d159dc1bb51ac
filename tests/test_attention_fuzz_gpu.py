"""Randomised sparse MLA decode cases on the GPU against the fp64 oracle.

Each case draws bf16 or FP8 rows, 1-4 requests, one or two verify tokens,
K in 1..2100 (one split to many, and more than 2048 rows), 1-128 heads, and
row ids with padding; the outputs and log-sum-exps must be within the stated
tolerance of the oracle (max-abs 1e-2, mean-rel 2e-3; lse 2e-3)."""
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
    rng = np.random.default_rng(1000 + seed)
    fp8 = bool(rng.random() < 0.4)
    R, T = int(rng.integers(1, 5)), int(rng.choice([1, 1, 2]))
    K = int(rng.integers(1, 2101))
    H = int(rng.choice([1, 7, 64, 100, 128]))
    blocks = -(-2 * K // P) + 1
    pool = hs.Pool(R, 1, K, P, P, ROW_ELEMS, 1, P * R, blocks, 1 if fp8 else 0)
    n = pool.blocks_per_layer * P
    raw = synth.rows_fp8(5000 + seed, 0, 0, 0, n) if fp8 else synth.rows(5000 + seed, 0, 0, 0, n)
    pool.kv_pool[0].copy_(torch.from_numpy(raw.view(np.int16)).cuda())
    rows = oracle.fp8_rows_to_f64(raw) if fp8 else raw
    ids = np.stack([np.stack([rng.choice(n, K, replace=False) for _ in range(T)])
                    for _ in range(R)]).astype(np.int32)                  # [R][T][K]
    pad = rng.random((R, T, K)) < rng.choice([0.0, 0.05, 0.5])
    ids[pad] = -1
    q = np.stack([np.stack([synth.q(6000 + seed, r, 0, k, H) for k in range(T)])
                  for r in range(R)])                                      # [R][T][H][576]
    out = torch.empty((R, T, H, V_DIM), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((R, T, H), dtype=torch.float32, device="cuda")
    d_q = torch.from_numpy(q.view(np.int16)).cuda()
    d_ids = torch.from_numpy(ids).cuda()
    if T == 1:
        hs.hs_sparse_mla_decode(pool.handle, 0, d_q, d_ids, H, V_DIM, SCALE, out, lse)
    else:
        hs.hs_sparse_mla_decode_tokens(pool.handle, 0, T, d_q, d_ids, H, V_DIM, SCALE, out, lse)
    torch.cuda.synchronize()
    got, got_lse = out.float().cpu().numpy(), lse.cpu().numpy()
    what = f"seed={seed} fp8={fp8} R={R} T={T} K={K} H={H}"
    for r in range(R):
        for k in range(T):
            valid = ids[r, k] >= 0
            ref, ref_lse = oracle.sparse_mla_decode(q[r, k], rows[np.maximum(ids[r, k], 0)],
                                                    valid, SCALE)
            if not valid.any():
                assert np.all(got[r, k] == 0) and np.all(np.isneginf(got_lse[r, k])), what
                continue
            err = np.abs(got[r, k].astype(np.float64) - ref)
            mean_rel = err.sum() / max(np.abs(ref).sum(), 1e-30)
            assert err.max() <= 1e-2 and mean_rel <= 2e-3, (what, r, k, err.max(), mean_rel)
            assert np.allclose(got_lse[r, k], ref_lse, rtol=0, atol=2e-3), (what, r, k)
    assert hs.hs_check_errors(pool.handle) == 0, what
    pool.close()


@pytest.mark.parametrize("seed", range(80))
def test_random_attention_cases(seed):
    one_case(seed)
