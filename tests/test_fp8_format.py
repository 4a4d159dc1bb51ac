"""Pins of the FP8 KV row format (656 bytes: 512 OCP E4M3 latent codes, 4 fp32
per-128 scales, 64 bf16 rope values), CPU only.

* the oracle's E4M3 decoding equals torch's float8_e4m3fn conversion on every
  code (a library routine);
* the generator's rounding equals torch's float -> float8_e4m3fn rounding on
  in-range values, including ties and subnormals;
* a generated FP8 row stands for its bf16 row within E4M3's half-ulp bound, with
  the rope values kept exactly and each group's largest value kept at 448 x
  scale;
* positions listed one by one give the same bytes as a contiguous fill.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")


def test_oracle_e4m3_table_matches_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.E4M3_TABLE
    assert np.all((ref == got) | (np.isnan(ref) & np.isnan(got)))
    assert np.nanmax(got) == 448.0 and np.nanmin(got[got > 0]) == 2.0 ** -9


def test_generator_rounding_matches_torch():
    rng = np.random.default_rng(3)
    vals = np.concatenate([
        rng.uniform(-448, 448, 3000),
        rng.uniform(-2.0 ** -6, 2.0 ** -6, 1000),           # subnormal range
        np.array([e4m3 for e4m3 in oracle.E4M3_TABLE if np.isfinite(e4m3)]),
        (oracle.E4M3_TABLE[1:0x7E] + oracle.E4M3_TABLE[2:0x7F]) / 2,   # ties
        -(oracle.E4M3_TABLE[1:0x7E] + oracle.E4M3_TABLE[2:0x7F]) / 2,
    ]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([synth.e4m3_encode(v) for v in vals], dtype=np.uint8)
    np.testing.assert_array_equal(got, ref)
    assert synth.e4m3_encode(1000.0) == 0x7E and synth.e4m3_encode(-1000.0) == 0xFE


def test_fp8_rows_stand_for_their_bf16_rows():
    raw = synth.rows_fp8(1004, 3, 1, 100, 64)
    bf = oracle.bf16_bits_to_f64(synth.rows(1004, 3, 1, 100, 64))
    deq = oracle.fp8_rows_to_f64(raw)
    np.testing.assert_array_equal(deq[:, 512:], bf[:, 512:])            # rope exact
    scales = raw[:, 512:528].copy().view(np.float32).astype(np.float64)
    for g in range(4):
        x, y, s = bf[:, 128 * g:128 * g + 128], deq[:, 128 * g:128 * g + 128], scales[:, g:g + 1]
        mx = np.abs(x).max(axis=1, keepdims=True)
        assert np.allclose(s, mx / 448.0, rtol=2 ** -23)
        bound = np.maximum(np.abs(x) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 2 ** -20)
        assert np.all(np.abs(y - x) <= bound)
        top = np.abs(x).argmax(axis=1)
        codes = raw[np.arange(64), 128 * g + top]
        assert np.all((codes & 0x7F) == 0x7E)                         # 448 x scale


def test_rows_at_matches_contiguous_fill():
    pos = np.array([5, 17, -1, 300, 5])
    got = synth.rows_fp8_at(1006, 2, 0, pos)
    for i, p in enumerate(pos):
        want = np.zeros(656, np.uint8) if p < 0 else synth.rows_fp8(1006, 2, 0, int(p), 1)[0]
        np.testing.assert_array_equal(got[i], want)
    big = synth.rows_fp8(1006, 2, 0, 0, 5000, threads=4)
    np.testing.assert_array_equal(big[300], got[3])


def test_e4m3_codes_worked_by_hand():
    """Codes decoded from E4M3's definition (sign, 4 exponent bits with bias 7,
    3 mantissa bits; exponent 0 is subnormal, 0x7F/0xFF are NaN), by hand."""
    cases = {
        0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
        0x30: 0.5, 0x38: 1.0, 0x3C: 1.5, 0x40: 2.0, 0x77: 240.0, 0x7E: 448.0,
        0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0,
    }
    for code, value in cases.items():
        assert oracle.E4M3_TABLE[code] == value, hex(code)
    assert np.isnan(oracle.E4M3_TABLE[0x7F]) and np.isnan(oracle.E4M3_TABLE[0xFF])
    assert np.signbit(oracle.E4M3_TABLE[0x80])
    # one row by hand: codes 0x38 (1.0) and 0x3C (1.5), group scales 0.5 .. 2
    raw = np.zeros((1, 656), dtype=np.uint8)
    raw[0, :512] = np.where(np.arange(512) % 2 == 0, 0x38, 0x3C)
    raw[0, 512:528] = np.array([0.5, 1.0, 1.5, 2.0], dtype=np.float32).view(np.uint8)
    raw[0, 528:656] = np.full(64, 0x3F80, dtype=np.uint16).view(np.uint8)    # bf16 1.0
    row = oracle.fp8_rows_to_f64(raw)[0]
    for g, sc in enumerate((0.5, 1.0, 1.5, 2.0)):
        np.testing.assert_array_equal(row[128 * g:128 * g + 128:2], sc * 1.0)
        np.testing.assert_array_equal(row[128 * g + 1:128 * g + 128:2], sc * 1.5)
    np.testing.assert_array_equal(row[512:], 1.0)


def test_e4m3_encoding_worked_by_hand():
    """The generator's encoder on values worked by hand: exact codes, a tie
    rounded to the even mantissa, saturation, and the subnormal range."""
    cases = [(1.0, 0x38), (-0.75, 0xB4), (448.0, 0x7E), (1000.0, 0x7E), (-1000.0, 0xFE),
             (1.0625, 0x38),          # halfway between 1.0 (mantissa 000) and 1.125: even
             (1.1875, 0x3A),          # halfway between 1.125 and 1.25 (mantissa 010): even
             (2.0 ** -9, 0x01), (3 * 2.0 ** -10, 0x02),   # 1.5 x 2^-9: tie to even (2 x 2^-9)
             (0.0, 0x00)]
    for value, code in cases:
        assert synth.e4m3_encode(value) == code, (value, hex(synth.e4m3_encode(value)))
