"""Sparse MLA decode where the running score maximum moves: the softmax's lazy
rescale path against the fp64 oracle.

The kernel keeps a reference maximum per head and moves it only when a tile's
maximum exceeds it by more than 2^8 (8 in log2 units); then the already
accumulated output is multiplied by 2^(m_old - m_new).  Seeded N(0,1) queries
and rows never move the maximum that far, so these cases are built to: scores
that rise along the selection list (every tile, or now and then), a query
scaled up, one dominant row in the last tile of a K split, and a first tile
that is all padding; with bf16 and FP8 rows and one, two and many K splits.

Each case also counts, from the inputs alone, how many heads take the rescale
under the kernel's work split (``rescale_events``), and asserts that the case
does reach the path.  Outputs must be within max-abs 1e-2 and mean-rel 2e-3 of
the fp64 oracle; lse within 2e-3 plus a small part relative to its size
(the scores here are far larger than the seeded ones).  Exactness of the method (page
"59188saintaubert.com ... HiSparse", section 02: only placement changes, the
attention output does not) is what the oracle states.
"""
import math
import zlib

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import sparse_attention_kv_hs_gb300 as hs  # noqa: E402

D, V_DIM, P = 576, 512, 256
SCALE = 192 ** -0.5
LOG2E = 1.4426950408889634
MAX_ABS, MEAN_REL = 1e-2, 2e-3
# lse: 2e-3 plus a part relative to its size.  The scores here reach ~200
# (natural log units) and carry rounding relative to their size: fp32
# accumulation for bf16 rows; for FP8 rows also the group scale rounded to
# fp16 (2^-12 relative) in the latent columns.
LSE_RTOL = {False: 1e-5, True: 2.5e-4}


def _bf16(x):
    """float -> bf16 bits, round to nearest even."""
    f = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((f + 0x7FFF + ((f >> 16) & 1)) >> 16).astype(np.uint16)


def _fp8_rows(vals):
    """float rows [n, 576] -> 656-byte FP8 rows: E4M3 codes of the 512 latent
    values with one fp32 scale per group of 128 (the group's largest magnitude
    / 448), then the 64 rope values in bf16.  Encoding by torch's float8_e4m3fn
    (round to nearest even); the oracle decodes the bytes themselves."""
    n = vals.shape[0]
    lat = vals[:, :512].astype(np.float32).reshape(n, 4, 128)
    scale = (np.abs(lat).max(axis=2) / np.float32(448.0)).astype(np.float32)  # [n, 4]
    safe = np.where(scale > 0, scale, np.float32(1.0))
    codes = torch.from_numpy(np.ascontiguousarray(lat / safe[:, :, None])).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy().reshape(n, 512)
    out = np.empty((n, 656), dtype=np.uint8)
    out[:, :512] = codes
    out[:, 512:528] = scale.view(np.uint8).reshape(n, 16)
    out[:, 528:656] = _bf16(vals[:, 512:]).view(np.uint8).reshape(n, 128)
    return out


def kernel_segments(R, K, num_sms):
    """The kernel's work split of one request's list: K splits of whole 64-row
    tiles (enough CTA pairs to cover the SMs once, at most 2048 rows each)."""
    tiles = -(-K // 64)
    s = max(1, num_sms // (2 * R))
    s = min(s, tiles)
    s = max(s, -(-tiles * 64 // 2048))
    rows = -(-tiles // s) * 64
    return [(b, min(b + rows, K)) for b in range(0, K, rows)], 64


def rescale_events(s_log2, valid, segments, tile):
    """Heads whose accumulated output the kernel rescales: within each segment
    the reference maximum starts at -inf and moves to a tile's maximum (over
    valid rows) when that exceeds it by more than 8; a move after the
    segment's first tile that changes the reference from a finite value is a
    rescale of the output.  s_log2: [H, K] scores times log2(e)."""
    H = s_log2.shape[0]
    hit = np.zeros(H, dtype=bool)
    for b, e in segments:
        m = np.full(H, -np.inf)
        for t0 in range(b, e, tile):
            v = valid[t0:min(t0 + tile, e)]
            if not v.any():
                continue
            tmax = s_log2[:, t0:min(t0 + tile, e)][:, v].max(axis=1)
            move = tmax > m + 8.0
            hit |= move & np.isfinite(m) & (t0 > b)
            m = np.where(move, tmax, m)
    return int(hit.sum())


def make_case(kind, R, K, H, fp8, seed):
    """Rows in list order for each request, a query per request, and the row ids.
    The value columns (the first 512) are 0.5 x N(0,1), so every output stays
    below 2.5 in magnitude, where bf16 output rounding (half an ulp <= 2^-7)
    leaves room in the 1e-2 bound; the scores move through the 64 rope
    columns, which enter only the scores.  kinds:
      steep     - scores rise by ~9 (log2) every 64 rows along the list
      gentle    - scores rise by ~9 (log2) every 256 rows
      qscale    - rows 0.5 x N(0,1), seeded queries times 16 (scores ~20 log2
                  wide; times 8 for FP8 rows)
      dominant  - flat scores, plus one row 40 (log2) above the rest at the end
                  of every 1024-row stretch
      padfirst  - steep, with the first 64 rows of every 1024-row stretch padding
      falling   - steep reversed (the maximum comes first: no rescale needed)
    """
    rng = np.random.default_rng(seed)
    w = rng.choice([-1.0, 1.0], size=D - 512)  # rope direction shared by every head
    n_rows = R * K
    vals = np.empty((n_rows, D))
    q = np.empty((R, H, D), dtype=np.uint16)
    valid = np.ones((R, K), dtype=bool)
    per_raw = 1.0 / (SCALE * LOG2E)  # raw score per log2 unit
    for r in range(R):
        k = 0.5 * rng.standard_normal((K, D))
        if kind == "qscale":
            # FP8 rows reach the score product as fp16 operands (11 significant
            # bits), whose rounding moves a score by ~2^-12 |q| |k| sqrt(576):
            # their queries are scaled less (scores ~10 log2 units wide)
            base = synth.bf16_to_f32(synth.q(70 + seed, r, 0, 0, H)).astype(np.float64)
            q[r] = _bf16(base * (8.0 if fp8 else 16.0))
        else:
            qf = np.empty((H, D))
            qf[:, :512] = 0.5 * rng.standard_normal((H, 512))
            qf[:, 512:] = w
            q[r] = _bf16(qf)
            if kind == "dominant":
                for j in list(range(1023, K, 1024)) + [K - 1]:
                    k[j, 512:] = 40.0 * per_raw / (D - 512) * w
            else:
                j = np.arange(K, dtype=np.float64)
                rate = 9.0 / 256.0 if kind == "gentle" else 9.0 / 64.0  # log2 units per row
                a = rate * j * per_raw / (D - 512)  # q.k gains a * 64 from the rope columns
                if kind == "falling":
                    a = a[::-1]
                k[:, 512:] += a[:, None] * w[None, :]
                if kind == "padfirst":
                    for b in range(0, K, 1024):
                        valid[r, b:b + 64] = False
        vals[r * K:(r + 1) * K] = k
    ids = np.arange(n_rows, dtype=np.int32).reshape(R, K)
    ids[~valid] = -1
    if fp8:
        raw = _fp8_rows(vals)
        rows_f64 = oracle.fp8_rows_to_f64(raw)
    else:
        raw = _bf16(vals)
        rows_f64 = oracle.bf16_bits_to_f64(raw)
    return q, raw, rows_f64, ids, valid


CASES = [
    # kind, R, K, H, fp8
    ("steep", 32, 2048, 128, False),
    ("steep", 8, 2048, 128, False),
    ("steep", 8, 2048, 64, True),
    ("gentle", 32, 2048, 128, False),
    ("gentle", 16, 2048, 128, True),
    ("qscale", 32, 2048, 128, False),
    ("qscale", 6, 1500, 100, True),
    ("dominant", 32, 2048, 128, False),
    ("dominant", 32, 2048, 128, True),
    ("padfirst", 32, 2048, 128, False),
    ("padfirst", 3, 2048, 16, True),
    ("falling", 16, 2048, 128, False),
]


@pytest.mark.parametrize("kind,R,K,H,fp8", CASES)
def test_attention_with_moving_maximum(kind, R, K, H, fp8):
    seed = zlib.crc32(f"{kind}/{R}/{K}/{H}/{fp8}".encode()) & 0xFFFF
    q, raw, rows_f64, ids, valid = make_case(kind, R, K, H, fp8, seed)
    n_rows = R * K
    blocks = -(-n_rows // P) + 1
    pool = hs.Pool(R, 1, K, P, P, D, 1, P * R, blocks, 1 if fp8 else 0)
    dev = torch.from_numpy(raw.view(np.int16).reshape(n_rows, -1)).cuda()
    pool.kv_pool[0][:n_rows].copy_(dev)
    d_q = torch.from_numpy(q.view(np.int16)).cuda()
    d_ids = torch.from_numpy(ids).cuda()
    out = torch.empty((R, H, V_DIM), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((R, H), dtype=torch.float32, device="cuda")
    hs.hs_sparse_mla_decode(pool.handle, 0, d_q, d_ids, H, V_DIM, SCALE, out, lse)
    torch.cuda.synchronize()
    got, got_lse = out.float().cpu().numpy(), lse.cpu().numpy()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    segments, tile = kernel_segments(R, K, sms)
    qf = oracle.bf16_bits_to_f64(q)
    events = 0
    for r in range(R):
        rows = rows_f64[ids[r].clip(0)]
        ref, ref_lse = oracle.sparse_mla_decode(q[r], rows, valid[r], SCALE)
        err = np.abs(got[r].astype(np.float64) - ref)
        mean_rel = err.sum() / np.abs(ref).sum()
        assert err.max() <= MAX_ABS and mean_rel <= MEAN_REL, (kind, r, err.max(), mean_rel)
        assert np.allclose(got_lse[r], ref_lse, rtol=LSE_RTOL[fp8], atol=2e-3), (kind, r)
        s_log2 = SCALE * LOG2E * (qf[r] @ rows.T)
        events += rescale_events(s_log2, valid[r], segments, tile)
    assert hs.hs_check_errors(pool.handle) == 0
    pool.close()
    if kind == "falling":
        assert events == 0
    else:
        # the case reaches the rescale path: some heads' output is rescaled
        assert events > 0, (kind, events)
    print(f"{kind} R={R} K={K} H={H} fp8={fp8}: {events} (request, head) rescales")
