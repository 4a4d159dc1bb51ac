"""FP8 KV rows (656 bytes, HS_KV_FP8) on the GPU against the CPU oracle.

RESOLVE, the row gather, page loads and prefix offload move rows as opaque
bytes, so with an FP8 pool the row ids are still bit-exact against the oracle
and every gathered or offloaded row is byte-identical to the generator's FP8
row at that position."""
import numpy as np
import pytest

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


def _fp8_page(w, r, l, page):
    return torch.from_numpy(synth.rows_fp8(w.seed, r, l, page * w.P, w.P).view(np.int16))


def replay_fp8(w, gather_every=1):
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
    replay_fp8(W.make("attention", R=4, steps=6))


def test_fp8_resolve_workload_with_resident_tail():
    replay_fp8(W.make("resolve", R=4, steps=8), gather_every=2)


def test_fp8_mixed_residency_with_offload():
    replay_fp8(W.make("mixed", R=16, steps=12, ctx_hi=131072), gather_every=3)


def test_fp8_pool_needs_576_wide_rows():
    with pytest.raises(hs.HsError):
        hs.Pool(1, 1, 64, 256, 256, 512, 4, 1024, 1, FP8)
