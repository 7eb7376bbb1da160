"""Pins of the oracle's MXFP8 encoding (oracle/mx.py) against the format's definition: the E4M3
bit fields, brute-force nearest rounding, a library conversion, closed forms of the E8M0 scale
and blocks worked by hand."""
import numpy as np
import pytest
import torch

from oracle import mx


def _finite_codes():
    c = np.arange(256, dtype=np.uint8)
    v = mx.e4m3_decode(c)
    keep = np.isfinite(v)
    return c[keep], v[keep]


def test_e4m3_code_table():
    """Facts of the E4M3 layout: 254 finite codes, largest 448 (0x7E), smallest normal 2^-6
    (0x08), smallest subnormal 2^-9 (0x01), NaN at S.1111.111, magnitudes increasing with the
    code."""
    v = mx.e4m3_decode(np.arange(256))
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert np.isfinite(v).sum() == 254
    assert v[0x7E] == 448.0 and v[0x08] == 2.0 ** -6 and v[0x01] == 2.0 ** -9
    assert v[0x38] == 1.0 and v[0xB8] == -1.0 and v[0x3C] == 1.5
    assert np.all(np.diff(v[:0x7F]) > 0)
    assert np.array_equal(v[0x80:0xFF], -v[:0x7F])


def test_e4m3_round_matches_brute_force():
    """Nearest finite E4M3 value by exhaustive search, ties to the even code, saturation past
    448: on every midpoint between neighbours, points beside them, and random values."""
    codes, vals = _finite_codes()
    pos = vals[(codes < 0x80)]
    pcodes = codes[(codes < 0x80)]
    mids = (pos[:-1] + pos[1:]) / 2
    rng = np.random.default_rng(7)
    xs = np.concatenate([pos, mids, np.nextafter(mids, 0), np.nextafter(mids, np.inf),
                         rng.uniform(0, 500, 4000), np.exp2(rng.uniform(-12, 9, 4000)),
                         [448.0, 463.9, 464.0, 470.0, 511.9, 1e6]])
    xs = np.concatenate([xs, -xs])

    def brute(x):
        a = min(abs(x), 448.0)
        dist = np.abs(pos - a)
        best = np.flatnonzero(dist == dist.min())
        pick = best[0] if len(best) == 1 else [b for b in best if pcodes[b] % 2 == 0][0]
        return np.copysign(pos[pick], x)
    want = np.array([brute(x) for x in xs])
    got = mx.e4m3_round(xs)
    assert np.array_equal(got, want)


def test_e4m3_round_matches_library_cast():
    """Within range, rounding equals torch's float8_e4m3fn cast (round to nearest even)."""
    rng = np.random.default_rng(8)
    xs = np.concatenate([rng.uniform(-448, 448, 20000), np.exp2(rng.uniform(-11, 8.8, 20000))])
    lib = torch.from_numpy(xs).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(mx.e4m3_round(xs), lib)


def test_e4m3_encode_round_trip():
    codes, vals = _finite_codes()
    back = mx.e4m3_encode(vals)
    assert np.array_equal(back, codes)


def test_mx_scale_code_closed_form():
    """floor(log2(amax)) - 8 + 127, clamped to [0, 254]; an all-zero block takes 0."""
    for k in range(-119, 136):
        for f in (1.0, 1.5, 2.0 - 2.0 ** -40):
            assert int(mx.mx_scale_code(np.float64(f * 2.0 ** k))) == k + 119
    assert int(mx.mx_scale_code(0.0)) == 0
    assert int(mx.mx_scale_code(2.0 ** -130)) == 0
    assert int(mx.mx_scale_code(2.0 ** 200)) == 254


def test_mxfp8_blocks_by_hand():
    """Two 32-feature blocks worked by hand from the definition.

    Block 0: amax 3 -> floor(log2 3) = 1 -> scale 2^-7, code 1 - 8 + 127 = 120. y / X:
    1 -> 128 = 2^7 (field 14, code 0x70); -0.5 -> -64 (field 13, sign: 0xE8); 3 -> 384 =
    1.5 * 2^8 (field 15, mantissa 4: 0x7C); 0.3 -> 38.4, spacing 4 in [32, 64), nearest 40 =
    1.25 * 2^5 (field 12, mantissa 2: 0x62).
    Block 1: amax 1.9 -> scale 2^-8, code 119. 1.9 -> 486.4 saturates to 448 (0x7E); 1.8 ->
    460.8, nearest 448 (0x7E); 0.001 -> 0.256 in [2^-2, 2^-1), spacing 2^-5: 8.19 steps -> 8,
    i.e. 0.25 (field 5, mantissa 0: 0x28)."""
    y = np.zeros((1, 64))
    y[0, :5] = [1.0, -0.5, 3.0, 0.0, 0.3]
    y[0, 32:35] = [1.9, 1.8, 0.001]
    codes, scale = mx.mxfp8_quantize(y)
    assert list(scale[0]) == [120, 119]
    assert list(codes[0, :5]) == [0x70, 0xE8, 0x7C, 0x00, 0x62]
    assert list(codes[0, 32:35]) == [0x7E, 0x7E, 0x28]
    assert np.all(codes[0, 5:32] == 0) and np.all(codes[0, 35:] == 0)
    deq = mx.mxfp8_dequantize(codes, scale)
    assert list(deq[0, :5]) == [1.0, -0.5, 3.0, 0.0, 40.0 / 128]
    assert list(deq[0, 32:35]) == [448.0 / 256, 448.0 / 256, 0.25 / 256]


def test_mxfp8_error_bound():
    """Every element is within half an E4M3 spacing (relative 2^-4) of y, or saturated, or
    below the block's subnormal step; the largest element lies in [256, 512) after scaling."""
    rng = np.random.default_rng(9)
    y = rng.standard_normal((64, 256)) * np.exp2(rng.integers(-20, 20, (64, 1)))
    codes, scale = mx.mxfp8_quantize(y)
    deq = mx.mxfp8_dequantize(codes, scale)
    X = np.repeat(np.exp2(scale.astype(np.float64) - 127.0), 32, axis=1)
    a = np.abs(y) / X
    err = np.abs(deq - y) / X
    ok = (err <= np.maximum(a, 2.0 ** -6) * 2.0 ** -4) | (a >= 448.0)
    assert ok.all()
    top = np.max(a.reshape(64, 8, 32), axis=2)
    assert np.all((top >= 256.0) & (top < 512.0))
