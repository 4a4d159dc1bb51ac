"""Speculative decoding on the GPU against the CPU oracle: hs_resolve_tokens
(the T verify tokens of each request resolved as one list) bit-exact on every
row id, miss count, miss-log entry and slot position; hs_sparse_mla_decode_tokens
(one decode per (request, token)) within the fp64 tolerance."""
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
    max_abs = float(err.max())
    mean_rel = float(err.sum() / np.abs(ref).sum())
    assert max_abs <= MAX_ABS and mean_rel <= MEAN_REL, (what, max_abs, mean_rel)


def replay_tokens(w, attn_steps=(), attn_requests=None, kv_format=0, check_state=False):
    scen = W.Scenario.build(w)
    pool = harness.make_pool(w, scen, kv_format)
    o = harness.make_oracle(w, scen)
    R, L, K, T, H = w.R, w.L, w.K, w.tokens, w.heads
    tr = np.stack([w.trace_tokens(r) for r in range(R)], axis=2)  # [steps][L][R][T][K]
    d_topk = torch.empty((R, T, K), dtype=torch.int32, device="cuda")
    d_rows = torch.empty((R, T, K), dtype=torch.int32, device="cuda")
    d_cnt = torch.empty((R,), dtype=torch.int32, device="cuda")
    d_log = torch.empty((R, T * K, 3), dtype=torch.int32, device="cuda")
    d_q = torch.empty((R, T, H, W.ROW_ELEMS), dtype=torch.int16, device="cuda")
    d_o = torch.empty((R, T, H, W.V_DIM), dtype=torch.bfloat16, device="cuda")
    d_lse = torch.empty((R, T, H), dtype=torch.float32, device="cuda")
    reqs = list(range(R)) if attn_requests is None else attn_requests
    for t in range(w.steps):
        for l in range(L):
            d_topk.copy_(torch.from_numpy(tr[t, l]))
            hs.hs_resolve_tokens(pool.handle, l, 1, T, d_topk, pool.step, d_rows, d_cnt, d_log)
            rows = d_rows.cpu().numpy()
            cnt = d_cnt.cpu().numpy()
            log = d_log.cpu().numpy()
            for r in range(R):
                ref_rows, ref_log, err = o.resolve_tokens(l, r, tr[t, l, r], t)
                assert err == 0
                np.testing.assert_array_equal(rows[r], ref_rows, err_msg=f"t={t} l={l} r={r}")
                assert cnt[r] == len(ref_log), (t, l, r)
                np.testing.assert_array_equal(log[r, :cnt[r]], ref_log)
                if check_state:  # every slot's position and stamp
                    ref_pos, ref_stamp = o.unit_state(l, r)
                    np.testing.assert_array_equal(pool.slot_pos[l, r].cpu().numpy(), ref_pos)
                    np.testing.assert_array_equal(pool.slot_stamp[l, r].cpu().numpy(), ref_stamp)
            if t in attn_steps:
                q = np.stack([np.stack([synth.q(w.seed, r, l, t * T + k, H) for k in range(T)])
                              for r in range(R)])
                d_q.copy_(torch.from_numpy(q.view(np.int16)))
                hs.hs_sparse_mla_decode_tokens(pool.handle, l, T, d_q, d_rows, H, W.V_DIM,
                                               W.SCALE, d_o, d_lse)
                out = d_o.float().cpu().numpy()
                lse = d_lse.cpu().numpy()
                for r in reqs:
                    for k in range(T):
                        kv = harness.rows_for_oracle(w, r, l, tr[t, l, r, k], kv_format)
                        ref, ref_lse = oracle.sparse_mla_decode(q[r, k], kv, None, W.SCALE)
                        _check(out[r, k], ref, (t, l, r, k))
                        assert np.allclose(lse[r, k], ref_lse, rtol=0, atol=2e-3)
        sp = pool.slot_pos.cpu().numpy()
        for l in range(L):
            for r in range(R):
                np.testing.assert_array_equal(sp[l, r], o.unit_state(l, r)[0])
        hs.hs_step_advance(pool.step)
    torch.cuda.synchronize()
    assert hs.hs_check_errors(pool.handle) == 0
    pool.close()


def test_spec_workload_scaled_down():
    """4 requests x 2 layers, T = 2 verify tokens, K 2048, B 8192, 6 steps."""
    w = W.make("spec", R=4, steps=6)
    replay_tokens(w, attn_steps={0, 5})


def test_spec_workload_full_size():
    """32 requests x 2 layers, ctx 65536, T = 2, K 2048, B 8192, 12 steps;
    attention checked on the last step for 4 requests (both tokens)."""
    w = W.make("spec", steps=12)
    replay_tokens(w, attn_steps={11}, attn_requests=[0, 5, 13, 31])


def test_spec_workload_fp8_rows():
    """The scaled-down spec workload on a pool of 656-byte FP8 rows."""
    w = W.make("spec", R=4, steps=4)
    replay_tokens(w, attn_steps={0, 3}, kv_format=1)


def test_one_token_is_the_plain_resolve():
    """hs_resolve_tokens with T = 1 gives hs_resolve's row ids and slot state."""
    w = W.make("attention", R=3, L=1, steps=5)
    scen = W.Scenario.build(w)
    a, b = harness.make_pool(w, scen), harness.make_pool(w, scen)
    tr = harness.traces(w)
    ra = torch.empty((w.R, w.K), dtype=torch.int32, device="cuda")
    rb = torch.empty((w.R, 1, w.K), dtype=torch.int32, device="cuda")
    for t in range(w.steps):
        d = torch.from_numpy(tr[t, 0]).cuda()
        hs.hs_resolve(a.handle, 0, 1, d, a.step, ra)
        hs.hs_resolve_tokens(b.handle, 0, 1, 1, d.view(w.R, 1, w.K), b.step, rb)
        assert torch.equal(ra, rb[:, 0])
        assert torch.equal(a.slot_pos, b.slot_pos) and torch.equal(a.slot_stamp, b.slot_stamp)
        hs.hs_step_advance(a.step)
        hs.hs_step_advance(b.step)
    torch.cuda.synchronize()
    assert hs.hs_check_errors(a.handle) == 0 and hs.hs_check_errors(b.handle) == 0
    a.close()
    b.close()


def test_repeats_within_and_across_tokens():
    """Hand-made lists on a small pool (K 8, one hot block of 256 slots): a
    position an earlier token selected shares that entry's row; a repeat whose
    first entry is in the same token is flagged and gets -1."""
    w = W.make("attention", R=1, L=1, steps=1)
    w.K, w.B = 8, 256
    scen = W.Scenario.build(w)
    pool = harness.make_pool(w, scen)
    o = harness.make_oracle(w, scen)
    lists = [np.array([[3, 9, 27, 81, 5, 6, 7, 8], [9, 3, 100, 101, 5, 200, 201, 202]]),
             np.array([[1, 2, 3, 4, 5, 6, 7, 8], [8, 7, 10, 10, 11, 12, 13, 14]])]
    d_rows = torch.empty((1, 2, 8), dtype=torch.int32, device="cuda")
    for t, lst in enumerate(lists):
        d_list = torch.from_numpy(lst.astype(np.int32)).view(1, 2, 8).cuda()
        hs.hs_resolve_tokens(pool.handle, 0, 1, 2, d_list, pool.step, d_rows)
        ref, _, err = o.resolve_tokens(0, 0, lst, t)
        got = d_rows.cpu().numpy()[0]
        np.testing.assert_array_equal(got, ref)
        assert err == (2 if t == 1 else 0)
        assert hs.hs_check_errors(pool.handle) == err
        assert got[1, 0] == got[0, 1 if t == 0 else 7] and got[1, 1] == got[0, 0 if t == 0 else 6]
        hs.hs_step_advance(pool.step)
    pool.close()


def test_five_verify_tokens_in_token_groups():
    """T = 5 tokens of K 2048 (10,240 entries, more than one CTA's 8,192), B =
    7 K: resolved as token groups (the tables of 4 tokens with B = 14,336 do
    not fit one CTA) after the pass that pins the whole list's hits; rows,
    miss counts and logs bit-exact against the oracle every step."""
    w = W.make("spec", R=4, steps=5, tokens=5)
    replay_tokens(w, attn_steps={0, 4}, attn_requests={0, 3}, check_state=True)


def test_six_verify_tokens_in_token_groups_with_the_largest_hot_buffer():
    """T = 6 (12,288 entries), B = 8 K = 16,384 slots, the most a unit takes."""
    w = W.make("spec", R=2, steps=4, tokens=6)
    replay_tokens(w, check_state=True)


def test_five_verify_tokens_through_the_decode_step():
    """T = 5 through hs_decode_step_tokens (later layers' RESOLVE on the copy stream)."""
    w = W.make("spec", R=4, steps=3, tokens=5)
    replay_step_tokens(w, check_steps={2}, attn_requests={0, 3})


def test_hot_buffers_above_16384_slots_are_rejected():
    """T = 7 at K 2048 needs B = 9 K = 18,432 slots: more than a unit takes
    (the pool refuses it)."""
    with pytest.raises(hs.HsError):
        hs.Pool(1, 1, 2048, 9 * 2048, 256, W.ROW_ELEMS, 256, 65536, 1)


def test_four_verify_tokens_scaled_down():
    """T = 4 verify tokens of K 2048 (8,192 entries per unit), B = 6 K."""
    w = W.make("spec", R=4, steps=5, tokens=4)
    replay_tokens(w, attn_steps={0, 4})


def test_four_verify_tokens_full_size_decode_step():
    """32 requests x 2 layers, T = 4, K 2048, B 12288, through hs_decode_step_tokens."""
    w = W.make("spec", steps=4, tokens=4)
    replay_step_tokens(w, check_steps={3}, attn_requests={0, 17})


def replay_step_tokens(w, check_steps, attn_requests, same_stream=False, kv_format=0):
    """hs_decode_step_tokens over every layer of each step against the oracle."""
    scen = W.Scenario.build(w)
    pool = harness.make_pool(w, scen, kv_format)
    o = harness.make_oracle(w, scen)
    R, L, K, T, H = w.R, w.L, w.K, w.tokens, w.heads
    tr = np.stack([w.trace_tokens(r) for r in range(R)], axis=2)  # [steps][L][R][T][K]
    d_topk = torch.empty((L, R, T, K), dtype=torch.int32, device="cuda")
    d_rows = torch.empty((L, R, T, K), dtype=torch.int32, device="cuda")
    d_cnt = torch.empty((L, R), dtype=torch.int32, device="cuda")
    d_q = torch.empty((L, R, T, H, W.ROW_ELEMS), dtype=torch.int16, device="cuda")
    d_o = torch.empty((L, R, T, H, W.V_DIM), dtype=torch.bfloat16, device="cuda")
    d_lse = torch.empty((L, R, T, H), dtype=torch.float32, device="cuda")
    main = torch.cuda.Stream()
    copy = main if same_stream else torch.cuda.Stream()
    for t in range(w.steps):
        q = np.stack([np.stack([np.stack([synth.q(w.seed, r, l, t * T + k, H) for k in range(T)])
                                for r in range(R)]) for l in range(L)])
        d_topk.copy_(torch.from_numpy(tr[t]))
        d_q.copy_(torch.from_numpy(q.view(np.int16)))
        torch.cuda.synchronize()
        with torch.cuda.stream(main):
            hs.hs_decode_step_tokens(pool.handle, 0, L, T, d_topk, d_q, H, W.V_DIM, W.SCALE,
                                     pool.step, d_rows, d_o, d_lse, d_cnt, main, copy)
            hs.hs_step_advance(pool.step, main)
        torch.cuda.synchronize()
        rows, cnt = d_rows.cpu().numpy(), d_cnt.cpu().numpy()
        out, lse = d_o.float().cpu().numpy(), d_lse.cpu().numpy()
        for l in range(L):
            for r in range(R):
                ref_rows, ref_log, err = o.resolve_tokens(l, r, tr[t, l, r], t)
                assert err == 0
                np.testing.assert_array_equal(rows[l, r], ref_rows, err_msg=f"t={t} l={l} r={r}")
                assert cnt[l, r] == len(ref_log), (t, l, r)
                if t in check_steps and r in attn_requests:
                    for k in range(T):
                        kv = harness.rows_for_oracle(w, r, l, tr[t, l, r, k], kv_format)
                        ref, ref_lse = oracle.sparse_mla_decode(q[l, r, k], kv, None, W.SCALE)
                        _check(out[l, r, k], ref, (t, l, r, k))
                        assert np.allclose(lse[l, r, k], ref_lse, rtol=0, atol=2e-3)
    assert hs.hs_check_errors(pool.handle) == 0
    pool.close()


def test_decode_step_tokens_spec_workload_full_size():
    """32 requests x 2 layers, T = 2, K 2048, B 8192: the spec benchmark's step,
    layer 1's RESOLVE on the copy stream."""
    w = W.make("spec", steps=6)
    replay_step_tokens(w, check_steps={0, 5}, attn_requests={0, 9, 31})


def test_decode_step_tokens_on_one_stream_scaled_down():
    w = W.make("spec", R=4, steps=4)
    replay_step_tokens(w, check_steps={0, 3}, attn_requests=set(range(4)), same_stream=True)


def test_decode_step_tokens_fp8_rows():
    w = W.make("spec", R=4, steps=4)
    replay_step_tokens(w, check_steps={0, 3}, attn_requests=set(range(4)), kv_format=1)


def test_decode_step_tokens_graph_captured():
    """One speculative step (two streams, events, step counter) captured once
    and replayed: row ids and miss counts match the oracle every step."""
    w = W.make("spec", R=3, steps=4)
    scen = W.Scenario.build(w)
    pool = harness.make_pool(w, scen)
    o = harness.make_oracle(w, scen)
    R, L, K, T, H = w.R, w.L, w.K, w.tokens, w.heads
    tr = np.stack([w.trace_tokens(r) for r in range(R)], axis=2)  # [steps][L][R][T][K]
    d_topk = torch.empty((L, R, T, K), dtype=torch.int32, device="cuda")
    d_rows = torch.empty((L, R, T, K), dtype=torch.int32, device="cuda")
    d_cnt = torch.empty((L, R), dtype=torch.int32, device="cuda")
    d_q = torch.zeros((L, R, T, H, W.ROW_ELEMS), dtype=torch.int16, device="cuda")
    d_o = torch.empty((L, R, T, H, W.V_DIM), dtype=torch.bfloat16, device="cuda")
    main, copy = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(main):
        with torch.cuda.graph(g, stream=main):
            hs.hs_decode_step_tokens(pool.handle, 0, L, T, d_topk, d_q, H, W.V_DIM, W.SCALE,
                                     pool.step, d_rows, d_o, None, d_cnt, main, copy)
            hs.hs_step_advance(pool.step, main)
    for t in range(w.steps):
        d_topk.copy_(torch.from_numpy(tr[t]))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        rows, cnt = d_rows.cpu().numpy(), d_cnt.cpu().numpy()
        for l in range(L):
            for r in range(R):
                ref_rows, ref_log, err = o.resolve_tokens(l, r, tr[t, l, r], t)
                assert err == 0
                np.testing.assert_array_equal(rows[l, r], ref_rows, err_msg=f"t={t} l={l} r={r}")
                assert cnt[l, r] == len(ref_log)
    assert hs.hs_check_errors(pool.handle) == 0
    pool.close()
