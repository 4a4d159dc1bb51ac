"""Randomised RESOLVE cases on the GPU against the CPU oracle.

Each case draws a small pool of random shape: 1-3 requests, 1-2 layers, K in
1..699 (so one unit's launch may use clusters of 1, 2, 4 or 8 CTAs), B from
about K to about 2K in whole pages (sometimes below K), P of 64 or 256,
random contexts, random resident pages, and one or two verify tokens.  The
lists are mostly distinct positions, with padding, repeats and out-of-range
entries mixed in now and then.  Every step, every unit's row ids, miss count
and slot positions, and the error bits, must equal the oracle's."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import sparse_attention_kv_hs_gb300 as hs  # noqa: E402

ROW_ELEMS = 576
SEEN = {"units": 0, "misses": 0, "errors": 0}   # what the random cases exercised


def _lists(rng, R, T, K, ctx):
    """[R][T][K] selections: distinct positions per token, token 1 sharing
    about half of token 0's, with rare padding, repeats and bad positions."""
    out = np.empty((R, T, K), dtype=np.int32)
    for r in range(R):
        for t in range(T):
            sel = rng.choice(int(ctx[r]), K, replace=False).astype(np.int32)
            if t > 0:
                keep = rng.random(K) < 0.5
                sel[keep] = out[r, 0][keep]
                # keep the token's own entries distinct: redraw collisions
                _, first = np.unique(sel, return_index=True)
                dup = np.ones(K, dtype=bool)
                dup[first] = False
                pool = np.setdiff1d(np.arange(int(ctx[r])), sel)
                sel[dup] = rng.choice(pool, int(dup.sum()), replace=False)
            u = rng.random()
            if u < 0.10:
                sel[rng.choice(K, max(1, K // 10), replace=False)] = -1      # padding
            elif u < 0.14 and K > 1:
                sel[K - 1] = sel[0]                                          # repeat
            elif u < 0.17:
                sel[rng.integers(K)] = int(ctx[r]) + int(rng.integers(1, 50))  # out of range
            out[r, t] = sel
    return out


def one_case(seed):
    rng = np.random.default_rng(seed)
    P = int(rng.choice([64, 256]))
    R, L = int(rng.integers(1, 4)), int(rng.integers(1, 3))
    K = int(rng.integers(1, 700))
    T = int(rng.choice([1, 1, 2]))
    nb = -(-K // P)
    hot = nb + int(rng.integers(0, nb + 1))
    if rng.random() < 0.1 and nb > 1:
        hot = nb - 1                                                         # B < K
    B = hot * P
    lo = max(2 * K, P)                         # room to redraw a token's repeats
    ctx = rng.integers(lo, lo + 5 * P + 1, size=R)
    max_pages = int(-(-int(ctx.max()) // P))
    host_off = np.concatenate([[0], np.cumsum(ctx)[:-1]]).astype(np.int64)
    resident = int(rng.integers(1, 4))
    pool = hs.Pool(R, L, K, B, P, ROW_ELEMS, max_pages, int(ctx.sum()), resident)
    o = oracle.ResolveOracle(R, L, K, B, P, ctx, pool.blocks_per_layer)
    s = torch.cuda.current_stream()
    for r in range(R):
        hs.hs_set_request(pool.handle, r, int(ctx[r]), int(host_off[r]), s)
        o.set_ctx(r, int(ctx[r]))
        for i in range(hot):
            o.set_hot_block(r, i, r * hot + i)
    for blk in range(R * hot, pool.blocks_per_layer):          # some resident pages
        if rng.random() < 0.7:
            r = int(rng.integers(R))
            page = int(rng.integers(-(-int(ctx[r]) // P)))
            hs.hs_map_page(pool.handle, r, page, blk, s)
            o.set_page(r, page, blk)
    d_list = torch.empty((R, T, K), dtype=torch.int32, device="cuda")
    d_rows = torch.empty((R, T, K), dtype=torch.int32, device="cuda")
    d_cnt = torch.empty((R,), dtype=torch.int32, device="cuda")
    what = f"seed={seed} P={P} R={R} L={L} K={K} T={T} B={B}"
    for t in range(4):
        for l in range(L):
            lists = _lists(rng, R, T, K, ctx)
            d_list.copy_(torch.from_numpy(lists))
            if T == 1:
                hs.hs_resolve(pool.handle, l, 1, d_list.view(R, K), pool.step,
                              d_rows.view(R, K), d_cnt, None, s)
            else:
                hs.hs_resolve_tokens(pool.handle, l, 1, T, d_list, pool.step, d_rows, d_cnt,
                                     None, s)
            rows, cnt = d_rows.cpu().numpy(), d_cnt.cpu().numpy()
            err_all = 0
            for r in range(R):
                if T == 1:
                    ref_rows, ref_log, err = o.resolve(l, r, lists[r, 0], t)
                    ref_rows = np.asarray(ref_rows).reshape(1, K)
                else:
                    ref_rows, ref_log, err = o.resolve_tokens(l, r, lists[r], t)
                    ref_rows = np.asarray(ref_rows).reshape(T, K)
                err_all |= err
                np.testing.assert_array_equal(rows[r], ref_rows, err_msg=f"{what} t={t} l={l} r={r}")
                assert cnt[r] == len(ref_log), (what, t, l, r)
                SEEN["units"] += 1
                SEEN["misses"] += int(cnt[r])
                SEEN["errors"] |= err
            assert hs.hs_check_errors(pool.handle) == err_all, (what, t, l)
            sp = pool.slot_pos.cpu().numpy()
            for r in range(R):
                np.testing.assert_array_equal(sp[l, r], o.unit_state(l, r)[0],
                                              err_msg=f"{what} t={t} l={l} r={r}")
        hs.hs_step_advance(pool.step, s)
    torch.cuda.synchronize()
    pool.close()
    o.close()


@pytest.mark.parametrize("seed", range(160))
def test_random_resolve_cases(seed):
    one_case(seed)


def test_the_random_cases_covered_every_error_kind():
    """Runs after the cases above: they checked many units and misses, and hit
    out-of-range positions (1), repeats (2) and a full hot buffer (4)."""
    if SEEN["units"] == 0:
        pytest.skip("the random cases did not run in this session")
    assert SEEN["units"] > 1000 and SEEN["misses"] > 100000, SEEN
    assert SEEN["errors"] & 7 == 7, SEEN
