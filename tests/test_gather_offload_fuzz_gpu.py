"""Randomised row gathers and batched page offloads on the GPU.

Gather: random row ids (with -1 and ids past the layer) over a pool of seeded
rows, bf16 or FP8; every output row must be byte-identical to the pool row
(zero for -1 and for a bad id, which also sets error bit BLOCK).  Offload:
random sets of mapped pages copied by one hs_offload_pages call; the host
rows must then hold exactly those pages' device rows, and no other host row
may change."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import sparse_attention_kv_hs_gb300 as hs  # noqa: E402

ROW_ELEMS, P = 576, 256


@pytest.mark.parametrize("seed", range(24))
def test_random_gathers(seed):
    rng = np.random.default_rng(11000 + seed)
    fp8 = bool(rng.random() < 0.5)
    L, blocks = int(rng.integers(1, 3)), int(rng.integers(1, 6))
    pool = hs.Pool(1, L, 64, P, P, ROW_ELEMS, 1, P, blocks, 1 if fp8 else 0)
    n = pool.blocks_per_layer * P
    raws = []
    for l in range(L):
        raw = (synth.rows_fp8(12000 + seed, 0, l, 0, n) if fp8
               else synth.rows(12000 + seed, 0, l, 0, n)).view(np.uint8).reshape(n, -1)
        pool.kv_pool[l].copy_(torch.from_numpy(raw.view(np.int16)).cuda())
        raws.append(raw)
    row_bytes = raws[0].shape[1]
    m = int(rng.integers(1, 5000))
    ids = rng.integers(0, n, size=m).astype(np.int32)
    ids[rng.random(m) < 0.1] = -1
    bad = rng.random() < 0.3
    if bad:
        ids[rng.integers(m)] = n + int(rng.integers(0, 100))
    l = int(rng.integers(L))
    out = torch.full((m, row_bytes // 2), 0x5555, dtype=torch.int16, device="cuda")
    hs.hs_gather(pool.handle, l, torch.from_numpy(ids).cuda(), m, out)
    got = out.cpu().numpy().view(np.uint8).reshape(m, row_bytes)
    ok = (ids >= 0) & (ids < n)
    np.testing.assert_array_equal(got[ok], raws[l][ids[ok]])
    assert not got[~ok].any()
    assert hs.hs_check_errors(pool.handle) == (hs.DEV_ERR_BLOCK if bad else 0)
    pool.close()


@pytest.mark.parametrize("seed", range(16))
def test_random_batched_offloads(seed):
    rng = np.random.default_rng(13000 + seed)
    fp8 = bool(rng.random() < 0.5)
    R, L = int(rng.integers(1, 5)), int(rng.integers(1, 3))
    pages = int(rng.integers(2, 9))                              # pages per request
    resident = R * pages
    pool = hs.Pool(R, L, 64, P, P, ROW_ELEMS, pages, R * pages * P, resident,
                   1 if fp8 else 0)
    s, side = torch.cuda.current_stream(), torch.cuda.Stream()
    units = pool.row_units
    for r in range(R):
        hs.hs_set_request(pool.handle, r, pages * P, r * pages * P, s)
    # device rows: seeded bytes for every resident block
    first = R                                                     # hot blocks come first
    dev = torch.from_numpy(rng.integers(-2 ** 15, 2 ** 15, size=(L, resident * P, units),
                                        dtype=np.int16)).cuda()
    pool.kv_pool[:, first * P:(first + resident) * P].copy_(dev)
    # a random subset of (request, page) pairs mapped to distinct blocks and offloaded
    pairs = [(r, g) for r in range(R) for g in range(pages) if rng.random() < 0.6] or [(0, 0)]
    blocks = rng.permutation(resident)[:len(pairs)]
    for (r, g), b in zip(pairs, blocks):
        hs.hs_map_page(pool.handle, r, g, first + int(b), s)
    pool.host_pool[...] = 0
    before = pool.host_pool.copy()
    ev = torch.cuda.Event()
    hs.hs_offload_pages(pool.handle, [p[0] for p in pairs], [p[1] for p in pairs], s, side, ev)
    ev.synchronize()
    torch.cuda.synchronize()
    want = before
    host_dev = dev.cpu().numpy()
    for (r, g), b in zip(pairs, blocks):
        base = r * pages * P + g * P
        want[:, base:base + P] = host_dev[:, int(b) * P:(int(b) + 1) * P]
    np.testing.assert_array_equal(pool.host_pool, want)
    assert hs.hs_check_errors(pool.handle) == 0
    pool.close()
