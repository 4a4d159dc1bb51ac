"""The in-kernel bounded waits give up, report it, and leave the context
usable.  Two one-thread kernels wait on mbarriers that nothing arrives on,
with the wait helpers of the attention kernel and of RESOLVE limited to
20 ms; afterwards an attention call runs and is checked against the oracle.
Nothing here faults or hangs the GPU: the waits end by their time limit."""
import time

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


def test_waits_give_up_and_the_context_stays_usable():
    res = torch.full((2,), -7, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    hs.hs_selftest_bounded_waits(20_000_000, res)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert res.cpu().tolist() == [hs.DEV_ERR_WAIT, 1]
    assert elapsed < 5.0, elapsed

    # the context still serves work: attention over 64 rows of a small pool
    P = 256
    pool = hs.Pool(1, 1, 64, P, P, W.ROW_ELEMS, 1, P, 1)
    rows = synth.rows(77, 0, 0, 0, pool.blocks_per_layer * P)
    pool.kv_pool[0].copy_(torch.from_numpy(rows.view(np.int16)).cuda())
    ids = np.arange(3, 3 + 64, dtype=np.int32)[None]
    q = synth.q(77, 0, 0, 0, 128)[None]
    out = torch.empty((1, 128, W.V_DIM), dtype=torch.bfloat16, device="cuda")
    hs.hs_sparse_mla_decode(pool.handle, 0, torch.from_numpy(q.view(np.int16)).cuda(),
                            torch.from_numpy(ids).cuda(), 128, W.V_DIM, W.SCALE, out)
    torch.cuda.synchronize()
    ref, _ = oracle.sparse_mla_decode(q[0], rows[ids[0]], None, W.SCALE)
    err = np.abs(out[0].float().cpu().numpy() - ref)
    assert err.max() <= 1e-2 and err.sum() / np.abs(ref).sum() <= 2e-3
    assert hs.hs_check_errors(pool.handle) == 0
    pool.close()


def test_selftest_rejects_bad_arguments():
    res = torch.zeros((2,), dtype=torch.int32, device="cuda")
    for bad in (0, -1, 10 ** 9):
        with pytest.raises(hs.HsError):
            hs.hs_selftest_bounded_waits(bad, res)
