"""RESOLVE + gather + prefix offload on the GPU against the CPU oracle.

Indexing parity is bit-exact: every row id, miss count, miss-log entry, slot
position, LRU stamp and the LRU order of every unit; every gathered row is
byte-identical to the generator's row at the selected position (the pages'
exactness statement: only placement changes)."""
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


def replay(w, *, state_every=1, gather_requests=None, check_offload=True, use_graph=False,
           batch_offload=False):
    scen = W.Scenario.build(w)
    pool = harness.make_pool(w, scen)
    o = harness.make_oracle(w, scen)
    tr = harness.traces(w)
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    R, K, L = w.R, w.K, w.L
    d_topk = torch.empty((R, K), dtype=torch.int32, device="cuda")
    d_out = torch.empty((R, K), dtype=torch.int32, device="cuda")
    d_cnt = torch.empty((R,), dtype=torch.int32, device="cuda")
    d_log = torch.empty((R, K, 3), dtype=torch.int32, device="cuda")
    d_rows = torch.empty((R * K, W.ROW_ELEMS), dtype=torch.int16, device="cuda")
    events = {}
    appended = []
    offs = w.host_offsets()
    ctx = w.ctx.astype(np.int64).copy()
    total_misses = 0
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
            hs.hs_resolve(pool.handle, l, 1, d_topk, pool.step, d_out, d_cnt, d_log, stream)
            out = d_out.cpu().numpy()
            cnt = d_cnt.cpu().numpy()
            log = d_log.cpu().numpy()
            for r in range(R):
                rows_ref, log_ref, err = o.resolve(l, r, tr[t, l, r], t)
                assert err == 0
                np.testing.assert_array_equal(out[r], rows_ref, err_msg=f"rows t={t} l={l} r={r}")
                assert cnt[r] == len(log_ref), (t, l, r)
                np.testing.assert_array_equal(log[r, :cnt[r]], log_ref)
                total_misses += int(cnt[r])
            if gather_requests is not None:
                hs.hs_gather(pool.handle, l, d_out, R * K, d_rows, stream)
                got = d_rows.view(R, K, W.ROW_ELEMS)
                for r in gather_requests(t, l):
                    expect = synth.rows_at(w.seed, r, l, tr[t, l, r])
                    assert np.array_equal(got[r].cpu().numpy().view(np.uint16), expect), (t, l, r)
        if state_every and (t % state_every == 0 or t == w.steps - 1):
            sp = pool.slot_pos.cpu().numpy()
            ss = pool.slot_stamp.cpu().numpy()
            so = pool.lru_order.cpu().numpy()
            for l in range(L):
                for r in range(R):
                    pos_ref, stamp_ref = o.unit_state(l, r)
                    np.testing.assert_array_equal(sp[l, r], pos_ref)
                    np.testing.assert_array_equal(ss[l, r], stamp_ref)
                    np.testing.assert_array_equal(so[l, r], harness.lru_order_reference(stamp_ref))
        hs.hs_step_advance(pool.step, stream)
        if batch_offload and scen.appends[t]:  # the step's pages in one offload launch
            for (r, page, blk) in scen.appends[t]:
                harness.write_append_gpu(pool, w, r, page, blk, stream)
            ev = torch.cuda.Event()
            hs.hs_offload_pages(pool.handle, [a[0] for a in scen.appends[t]],
                                [a[1] for a in scen.appends[t]], stream, side, ev)
            for (r, page, blk) in scen.appends[t]:
                events[(r, page)] = ev
        for (r, page, blk) in scen.appends[t]:
            if not batch_offload:
                harness.apply_append_gpu(pool, w, r, page, blk, stream, side, events)
            ctx[r] += w.P
            hs.hs_set_request(pool.handle, r, int(ctx[r]), int(offs[r]), stream)
            o.set_page(r, page, blk)
            o.set_ctx(r, int(ctx[r]))
            appended.append((r, page))
    torch.cuda.synchronize()
    assert hs.hs_check_errors(pool.handle) == 0
    if check_offload:
        for (r, page) in appended:
            for l in range(L):
                base = int(offs[r]) + page * w.P
                got = pool.host_pool[l, base:base + w.P]
                assert np.array_equal(got, synth.rows(w.seed, r, l, page * w.P, w.P)), (r, page, l)
    pool.close()
    return total_misses


def test_tiny_workload_every_step():
    w = W.make("tiny")
    misses = replay(w, gather_requests=lambda t, l: [0])
    assert misses > 0


def test_resolve_workload_scaled_down_with_tail():
    w = W.make("resolve", R=4, steps=24)
    replay(w, gather_requests=lambda t, l: range(4))


def test_resolve_workload_full_size():
    """16 requests x 4 layers, ctx 32768, K 2048, B 4096, tail 4096, 256 steps."""
    w = W.make("resolve")
    replay(w, state_every=8, gather_requests=lambda t, l: [(t + l) % w.R] if t % 8 == 0 else [])


def test_gather_workload_full_size():
    """64 x 4, ctx 131072 (host pool 38.7 GB), cold start then steady state."""
    w = W.make("gather")
    replay(w, state_every=32, gather_requests=lambda t, l: [(3 * t + l) % w.R] if t % 16 == 0 else [])


def test_mixed_residency_scaled_down_with_offload():
    w = W.make("mixed", R=16, steps=24, ctx_hi=131072)
    replay(w, state_every=4, gather_requests=lambda t, l: range(w.R) if t % 4 == 0 else [])


def test_mixed_residency_scaled_down_with_batched_offload():
    """The step's appended pages offloaded by one hs_offload_pages launch."""
    w = W.make("mixed", R=16, steps=24, ctx_hi=131072)
    replay(w, state_every=4, gather_requests=lambda t, l: range(w.R) if t % 4 == 0 else [],
           batch_offload=True)


def test_offload_pages_arguments_and_unmapped_page():
    """Out-of-range pairs and counts are rejected with nothing launched; an
    unmapped page is skipped with error bit BLOCK while the others copy."""
    w = W.make("tiny")
    scen = W.Scenario.build(w)
    pool = harness.make_pool(w, scen)
    stream, side = torch.cuda.current_stream(), torch.cuda.Stream()
    ev = torch.cuda.Event()
    for reqs, pages in ([w.R], [0]), ([0], [-1]), ([0], [10 ** 6]), ([], []), \
            ([0] * (hs.HS_OFFLOAD_MAX_PAGES + 1), [0] * (hs.HS_OFFLOAD_MAX_PAGES + 1)):
        with pytest.raises(hs.HsError):
            hs.hs_offload_pages(pool.handle, reqs, pages, stream, side, ev)
    blk = pool.blocks_per_layer - 1                        # the resident block
    last = int(w.ctx_capacity()[0]) // w.P - 1
    harness.write_append_gpu(pool, w, 0, last, blk, stream)
    hs.hs_map_page(pool.handle, 0, last - 1, -1, stream)   # unmapped: skipped
    pool.host_pool[:, int(w.host_offsets()[0]) + last * w.P:][:, :w.P] = 0
    hs.hs_offload_pages(pool.handle, [0, 0], [last - 1, last], stream, side, ev)
    torch.cuda.synchronize()
    assert hs.hs_check_errors(pool.handle) == hs.DEV_ERR_BLOCK
    base = int(w.host_offsets()[0]) + last * w.P
    for l in range(w.L):
        assert np.array_equal(pool.host_pool[l, base:base + w.P],
                              synth.rows(w.seed, 0, l, last * w.P, w.P))
    pool.close()


def test_mixed_residency_full_size():
    """128 requests, ctx log-uniform 16K..1M, zero/full/tail residency, page
    appends queued for async host offload every step."""
    w = W.make("mixed")
    replay(w, state_every=16, gather_requests=lambda t, l: [t % w.R, (7 * t + 3) % w.R])


# ------------------------------------------------------------------ edge cases

def _small_pool(K, B, P, ctx, R=1, L=1, resident=None, host_rows=True):
    max_pages = (ctx + P - 1) // P
    resident = resident or {}
    pool = hs.Pool(R, L, K, B, P, W.ROW_ELEMS, max_pages, R * ctx, max(1, len(resident) * R))
    o = oracle.ResolveOracle(R, L, K, B, P, [ctx] * R, pool.blocks_per_layer)
    s = torch.cuda.current_stream()
    for r in range(R):
        if host_rows:
            for l in range(L):
                synth.rows_into(77, r, l, 0, ctx, W.ROW_ELEMS,
                                pool.host_pool[l, r * ctx:].ctypes.data, harness.HOST_THREADS)
        hs.hs_set_request(pool.handle, r, ctx, r * ctx, s)
        o.set_ctx(r, ctx)
        for i in range(B // P):
            o.set_hot_block(r, i, r * (B // P) + i)
    nb = R * (B // P)
    for r in range(R):
        for k, page in enumerate(sorted(resident)):
            blk = nb + r * len(resident) + k
            hs.hs_load_page(pool.handle, r, page, blk, s)
            o.set_page(r, page, blk)
    torch.cuda.synchronize()
    return pool, o


def _run_steps(pool, o, sels, R=1, L=1, expect_err=0):
    K = pool.K
    d_topk = torch.empty((R, K), dtype=torch.int32, device="cuda")
    d_out = torch.empty((R, K), dtype=torch.int32, device="cuda")
    d_cnt = torch.empty((R,), dtype=torch.int32, device="cuda")
    d_log = torch.empty((R, K, 3), dtype=torch.int32, device="cuda")
    errs = 0
    for t, sel in enumerate(sels):
        sel = np.asarray(sel, dtype=np.int32).reshape(R, K)
        d_topk.copy_(torch.from_numpy(sel))
        hs.hs_resolve(pool.handle, 0, 1, d_topk, pool.step, d_out, d_cnt, d_log)
        out, cnt, log = d_out.cpu().numpy(), d_cnt.cpu().numpy(), d_log.cpu().numpy()
        for r in range(R):
            ref, log_ref, err = o.resolve(0, r, sel[r], t)
            errs |= err
            np.testing.assert_array_equal(out[r], ref, err_msg=f"t={t}")
            assert cnt[r] == len(log_ref)
            np.testing.assert_array_equal(log[r, :cnt[r]], log_ref)
            pos_ref, stamp_ref = o.unit_state(0, r)
            np.testing.assert_array_equal(pool.slot_pos[0, r].cpu().numpy(), pos_ref)
            np.testing.assert_array_equal(pool.slot_stamp[0, r].cpu().numpy(), stamp_ref)
            np.testing.assert_array_equal(pool.lru_order[0, r].cpu().numpy(),
                                          harness.lru_order_reference(stamp_ref))
        hs.hs_step_advance(pool.step)
    code = hs.hs_check_errors(pool.handle)
    assert code == errs == expect_err
    return errs


def test_padding_range_and_repeats():
    K, B, P, ctx = 64, 128, 32, 1024
    pool, o = _small_pool(K, B, P, ctx, resident={31: 0, 30: 0})
    rng = np.random.default_rng(5)
    sels = []
    for t in range(12):
        s = rng.choice(ctx, K, replace=False).astype(np.int32)
        if t % 3 == 0:
            s[rng.integers(0, K, 5)] = -1            # padding
        if t % 4 == 1:
            s[7] = ctx + 5                            # out of range
            s[9] = -3                                 # invalid negative
        if t % 5 == 2:
            s[11] = s[10]                             # repeat
        sels.append(s)
    _run_steps(pool, o, sels, expect_err=oracle.ERR_RANGE | oracle.ERR_DUPLICATE)
    pool.close()


def test_capacity_error_when_b_below_k():
    K, B, P, ctx = 96, 64, 32, 4096
    pool, o = _small_pool(K, B, P, ctx)
    rng = np.random.default_rng(6)
    sels = [rng.choice(ctx, K, replace=False) for _ in range(4)]
    _run_steps(pool, o, sels, expect_err=oracle.ERR_CAPACITY)
    pool.close()


def test_ragged_sizes_and_several_requests():
    # K, B not multiples of the CTA width; several requests and layers share a launch
    K, B, P, ctx, R = 300, 448, 64, 3008, 3
    pool, o = _small_pool(K, B, P, ctx, R=R, resident={46: 0})
    rng = np.random.default_rng(7)
    sels = [np.stack([rng.choice(ctx, K, replace=False) for _ in range(R)]) for _ in range(10)]
    _run_steps(pool, o, sels, R=R)
    pool.close()


def test_top1_and_all_padding():
    pool, o = _small_pool(1, 64, 64, 512)
    _run_steps(pool, o, [[5], [5], [-1], [7], [5]])
    pool.close()


def test_largest_supported_shapes():
    """K = 4096 with B = 4096, and B = 8192 (the pages' doubled buffer) with K = 2048."""
    for K, B in ((4096, 4096), (2048, 8192)):
        ctx = 65536
        pool, o = _small_pool(K, B, 256, ctx, host_rows=False)
        rng = np.random.default_rng(K + B)
        prev = rng.choice(ctx, K, replace=False)
        sels = [prev]
        for _ in range(3):
            keep = rng.choice(prev, int(0.7 * K), replace=False)
            new = np.setdiff1d(rng.choice(ctx, 2 * K, replace=False), keep)[: K - keep.size]
            prev = rng.permutation(np.concatenate([keep, new]))
            sels.append(prev)
        _run_steps(pool, o, sels)
        pool.close()


def test_gather_padding_and_bad_row_ids():
    pool, o = _small_pool(8, 64, 64, 512)
    rows = pool.blocks_per_layer * 64
    ids = torch.tensor([0, -1, 5, rows, rows + 100, 63], dtype=torch.int32, device="cuda")
    out = torch.empty((6, W.ROW_ELEMS), dtype=torch.int16, device="cuda")
    hs.hs_gather(pool.handle, 0, ids, 6, out)
    got = out.cpu().numpy()
    kv = pool.kv_pool[0].cpu().numpy()
    assert np.array_equal(got[0], kv[0]) and np.array_equal(got[2], kv[5])
    assert np.array_equal(got[5], kv[63])
    assert np.all(got[1] == 0) and np.all(got[3] == 0) and np.all(got[4] == 0)
    assert hs.hs_check_errors(pool.handle) == hs.DEV_ERR_BLOCK
    pool.close()


def test_graph_capture_replays_with_device_step():
    """The resolve of a step is captured once in a CUDA graph and replayed:
    the step counter is read from device memory, so each replay is a new step
    and the results match the oracle step by step."""
    w = W.make("tiny", steps=16)
    scen = W.Scenario.build(w)
    pool = harness.make_pool(w, scen)
    o = harness.make_oracle(w, scen)
    tr = harness.traces(w)
    d_topk = torch.empty((w.R, w.K), dtype=torch.int32, device="cuda")
    d_out = torch.empty((w.R, w.K), dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        d_topk.copy_(torch.from_numpy(tr[0, 0]))
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            hs.hs_resolve(pool.handle, 0, 1, d_topk, pool.step, d_out, None, None, s)
            hs.hs_step_advance(pool.step, s)
    for t in range(w.steps):
        d_topk.copy_(torch.from_numpy(tr[t, 0]))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ref, _, err = o.resolve(0, 0, tr[t, 0, 0], t)
        np.testing.assert_array_equal(d_out.cpu().numpy()[0], ref)
    assert int(pool.step.item()) == w.steps
    pool.close()


def test_host_read_copies_mapped_host_memory():
    pool, o = _small_pool(8, 64, 64, 4096)
    n = 4096 * W.ROW_BYTES
    dst = torch.empty(n, dtype=torch.uint8, device="cuda")
    hs.hs_host_read(int(pool.raw.host_pool_device), n, dst)
    torch.cuda.synchronize()
    assert np.array_equal(dst.cpu().numpy(), pool.host_pool[0, :4096].view(np.uint8).reshape(-1))
    with pytest.raises(hs.HsError):
        hs.hs_host_read(int(pool.raw.host_pool_device) + 8, 64, dst)   # misaligned
    pool.close()
