"""MXFP8 encoding of the sublayer input y (oracle; test infrastructure only).

The pages name the consumer of y -- the flow diagram of "2A · Single-Pass mHC", section 2
("Luồng"), lists an FP4 MoE among the blocks that follow the mHC step -- but define no format for
a quantised y. The format taken is the published OCP Microscaling (MX) Formats Specification
v1.0, concrete format MXFP8 with E4M3 elements:

  * a block is 32 consecutive features of one token (block b of token t covers y[t, 32b:32b+32]);
  * the block's shared scale is X = 2^(floor(log2(amax)) - 8), amax the largest |y| of the block
    and 8 the exponent of E4M3's largest power of two; X is stored as an E8M0 code
    (floor(log2(amax)) - 8 + 127), clamped to the code range [0, 254]; an all-zero block takes
    code 0;
  * each element is y / X rounded to the nearest E4M3 value (ties to even) with saturation to
    +-448, the largest finite E4M3 magnitude (the specification leaves overflow handling to the
    implementation; values y / X in [448, 512) occur by construction and clamp to 448).

E4M3 (the "fn" variant of the OCP FP8 formats): 1 sign bit, 4 exponent bits with bias 7,
3 mantissa bits; exponent field 0 holds subnormals m/8 * 2^-6; there are no infinities and the
codes S.1111.111 are NaN.

The values encoded are the bf16 y of the step (the sublayer input as the bf16 path delivers it),
so the encoding equals a separate MXFP8 pass over that y. The oracle's bf16 y and the kernel's
may differ by up to two bf16 ulps (the RMS statistic is summed in another order); the parity
tests compare the codes where that cannot change a decision and bound the rest.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
MX_BLOCK = 32
E4M3_EMAX = 8             # exponent of the largest power of two E4M3 represents (2^8 = 256)


def e4m3_decode(codes) -> np.ndarray:
    """Values of E4M3 codes (uint8) from their bit fields; NaN for the NaN codes."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_round(v) -> np.ndarray:
    """Round float64 values to the nearest E4M3 value, ties to even, saturating at +-448."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    out = np.zeros_like(a)
    nz = a > 0
    # spacing of E4M3 numbers around a: 2^(e-3) for a in [2^e, 2^(e+1)), e >= -6; 2^-9 below
    _, ex = np.frexp(a[nz])                       # a in [2^(ex-1), 2^ex)
    q = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)
    out[nz] = np.rint(a[nz] / q) * q              # np.rint: halves to even (even mantissa)
    out = np.minimum(out, E4M3_MAX)
    return np.copysign(out, v)


def e4m3_encode(v) -> np.ndarray:
    """E4M3 codes of values that are exactly representable (as e4m3_round returns them)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    code = np.zeros(a.shape, dtype=np.int64)
    sub = a < 2.0 ** -6
    code[sub] = np.rint(a[sub] / 2.0 ** -9).astype(np.int64)
    _, ex = np.frexp(a[~sub])
    e = ex - 1                                     # a in [2^e, 2^(e+1))
    m = np.rint((a[~sub] / np.ldexp(1.0, e) - 1.0) * 8.0).astype(np.int64)
    code[~sub] = ((e + 7) << 3) | m
    code = code | np.where(np.signbit(v), 0x80, 0)
    return code.astype(np.uint8)


def mx_scale_code(amax) -> np.ndarray:
    """E8M0 code of the shared scale of blocks with largest magnitude amax (float64 >= 0)."""
    amax = np.asarray(amax, dtype=np.float64)
    code = np.zeros(amax.shape, dtype=np.int64)
    pos = amax > 0
    _, ex = np.frexp(amax[pos])                    # floor(log2(amax)) = ex - 1
    code[pos] = np.clip(ex - 1 - E4M3_EMAX + 127, 0, 254)
    return code.astype(np.uint8)


def mxfp8_quantize(y):
    """y [N, d] (float64, d a multiple of 32) -> (codes uint8 [N, d], scale codes uint8 [N, d/32])."""
    y = np.asarray(y, dtype=np.float64)
    N, d = y.shape
    blocks = y.reshape(N, d // MX_BLOCK, MX_BLOCK)
    scale = mx_scale_code(np.max(np.abs(blocks), axis=2))
    X = np.exp2(scale.astype(np.float64) - 127.0)[:, :, None]
    codes = e4m3_encode(e4m3_round(blocks / X))
    return codes.reshape(N, d), scale


def mxfp8_dequantize(codes, scale) -> np.ndarray:
    """codes uint8 [N, d], scale codes uint8 [N, d/32] -> float64 values code * 2^(scale - 127)."""
    codes = np.asarray(codes)
    N, d = codes.shape
    X = np.exp2(np.asarray(scale, dtype=np.float64) - 127.0)
    return (e4m3_decode(codes).reshape(N, d // MX_BLOCK, MX_BLOCK) * X[:, :, None]).reshape(N, d)
