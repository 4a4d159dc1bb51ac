"""hs_decode_step (RESOLVE + attention for every layer of a step, with the
next layer's RESOLVE on a copy stream beside the current attention) against
the CPU oracle: row ids bit-exact every step, attention within the fp64
tolerance on sampled steps, for both stream arrangements and under graph
capture."""
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


def _queries(w, t):
    return np.stack([np.stack([synth.q(w.seed, r, l, t, w.heads) for r in range(w.R)])
                     for l in range(w.L)])  # [L][R][H][576] bf16 bits


def replay_steps(w, check_steps, same_stream=False, graph=False, kv_format=0):
    scen = W.Scenario.build(w)
    pool = harness.make_pool(w, scen, kv_format)
    o = harness.make_oracle(w, scen)
    tr = harness.traces(w)  # [steps][L][R][K]
    R, K, L, H = w.R, w.K, w.L, w.heads
    d_topk = torch.empty((L, R, K), dtype=torch.int32, device="cuda")
    d_q = torch.empty((L, R, H, W.ROW_ELEMS), dtype=torch.int16, device="cuda")
    d_rows = torch.empty((L, R, K), dtype=torch.int32, device="cuda")
    d_out = torch.empty((L, R, H, W.V_DIM), dtype=torch.bfloat16, device="cuda")
    d_lse = torch.empty((L, R, H), dtype=torch.float32, device="cuda")
    d_cnt = torch.empty((L, R), dtype=torch.int32, device="cuda")
    main = torch.cuda.Stream()
    copy = main if same_stream else torch.cuda.Stream()

    def step():
        hs.hs_decode_step(pool.handle, 0, L, d_topk, d_q, H, W.V_DIM, W.SCALE, pool.step, d_rows,
                          d_out, d_lse, d_cnt, main, copy)
        hs.hs_step_advance(pool.step, main)

    g = None
    if graph:
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(main):
            with torch.cuda.graph(g, stream=main):
                step()
    for t in range(w.steps):
        q = _queries(w, t)
        d_topk.copy_(torch.from_numpy(tr[t]))
        d_q.copy_(torch.from_numpy(q.view(np.int16)))
        torch.cuda.synchronize()
        if g is not None:
            g.replay()
        else:
            with torch.cuda.stream(main):
                step()
        torch.cuda.synchronize()
        rows = d_rows.cpu().numpy()
        cnt = d_cnt.cpu().numpy()
        out = d_out.float().cpu().numpy()
        lse = d_lse.cpu().numpy()
        for l in range(L):
            for r in range(R):
                ref_rows, ref_log, err = o.resolve(l, r, tr[t, l, r], t)
                assert err == 0
                np.testing.assert_array_equal(rows[l, r], ref_rows, err_msg=f"t={t} l={l} r={r}")
                assert cnt[l, r] == len(ref_log), (t, l, r)
                if t in check_steps:
                    kv = harness.rows_for_oracle(w, r, l, tr[t, l, r], kv_format)
                    ref, ref_lse = oracle.sparse_mla_decode(q[l, r], kv, None, W.SCALE)
                    _check(out[l, r], ref, (t, l, r))
                    assert np.allclose(lse[l, r], ref_lse, rtol=0, atol=2e-3)
    assert hs.hs_check_errors(pool.handle) == 0
    pool.close()


def test_decode_step_attention_workload_full_size():
    """32 requests x 2 layers, ctx 65536, K 2048, B 4096, 128 heads: the
    benchmark's step, with layer 1's RESOLVE beside layer 0's attention."""
    w = W.make("attention", steps=8)
    replay_steps(w, check_steps={0, 1, 7})


def test_decode_step_three_layers_scaled_down():
    """Two RESOLVE launches queued on the copy stream."""
    w = W.make("attention", R=4, L=3, steps=5)
    replay_steps(w, check_steps={0, 4})


def test_decode_step_on_one_stream():
    w = W.make("attention", R=3, L=2, steps=4)
    replay_steps(w, check_steps={0, 3}, same_stream=True)


def test_decode_step_graph_captured():
    """One step (both streams, events, step counter) captured once, replayed."""
    w = W.make("attention", R=2, L=2, steps=5)
    replay_steps(w, check_steps={0, 2, 4}, graph=True)


def test_decode_step_fp8_rows():
    """The full-size step on a pool of 656-byte FP8 rows."""
    w = W.make("attention", steps=4)
    replay_steps(w, check_steps={0, 3}, kv_format=1)


def test_decode_step_rejects_bad_arguments():
    w = W.make("attention", R=1, L=2, steps=1)
    scen = W.Scenario.build(w)
    pool = harness.make_pool(w, scen)
    t = torch.zeros((2, 1, w.K), dtype=torch.int32, device="cuda")
    q = torch.zeros((2, 1, w.heads, W.ROW_ELEMS), dtype=torch.int16, device="cuda")
    o = torch.empty((2, 1, w.heads, W.V_DIM), dtype=torch.bfloat16, device="cuda")
    rows = torch.empty((2, 1, w.K), dtype=torch.int32, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    bad = [
        dict(layer_begin=1, num_layers=2),       # past the last layer
        dict(layer_begin=0, num_layers=0),
        dict(layer_begin=0, num_layers=2, num_heads=129),
        dict(layer_begin=0, num_layers=2, v_dim=576),
        dict(layer_begin=0, num_layers=2, scale=0.0),
    ]
    for b in bad:
        args = dict(layer_begin=0, num_layers=2, num_heads=w.heads, v_dim=W.V_DIM, scale=W.SCALE)
        args.update(b)
        with pytest.raises(hs.HsError):
            hs.hs_decode_step(pool.handle, args["layer_begin"], args["num_layers"], t, q,
                              args["num_heads"], args["v_dim"], args["scale"], pool.step, rows, o,
                              None, None, s1, s2)
    torch.cuda.synchronize()
    assert hs.hs_check_errors(pool.handle) == 0
    pool.close()
