"""MXFP8 (e4m3 elements, E8M0 shared scale per 32-element block) codec in fp64.

TEST INFRASTRUCTURE (same rule as ``moe_oracle``: only tests, the smoke check
and the bench's CPU baseline leg may use it).

The pages say only that routed weights may be MXFP8: an FP8 payload plus E8M0
scales, compact per-32 blocks along the GEMM's K, with a columnwise copy whose
scale shape is (rows // 32, columns) ("Add Mixture-of-Kittens MoE backend on
main", PR #8210, review threads on _swizzle_mxfp8_scale and
quantized_routed_weights; "feat(moe): add a megakernel backend with MOK
integration", Design > MCore-owned parameters). They give no quantisation rule,
so this follows the OCP Microscaling (MX) v1.0 definition:

* element format OCP FP8 E4M3 ("FN": no infinities, S.1111.111 is NaN,
  largest finite 448, subnormals 2^-6 * m/8);
* block of 32 along K; shared exponent = floor(log2(amax)) - 8 (8 = the
  largest E4M3 exponent); E8M0 code = shared exponent + 127 clamped to [0, 254];
* elements = round-to-nearest-even of x / 2^shared_exp, saturating at +-448;
  an all-zero block gets scale code 0 and zero payload.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
BLOCK = 32


def e4m3_decode(codes):
    """uint8 E4M3 codes -> fp64 values (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes, np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    sub = man / 8.0 * 2.0 ** -6
    nrm = (1.0 + man / 8.0) * np.exp2(exp - 7.0)
    val = np.where(exp == 0, sub, nrm)
    val = np.where((exp == 15) & (man == 7), np.nan, val)
    return sign * val


# the 127 non-negative finite E4M3 values, in code order (codes 0x00..0x7E);
# the value grows with the code, so the nearest code is found by bisection
_POS_VALUES = e4m3_decode(np.arange(0x7F, dtype=np.uint8))


def e4m3_encode(x):
    """fp64 values -> uint8 E4M3 codes: round to nearest, ties to the even code
    (the even mantissa), saturate to +-448; NaN -> 0x7F."""
    x = np.asarray(x, np.float64)
    mag = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(_POS_VALUES, mag, side="left"), 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    d_hi = _POS_VALUES[hi] - mag
    d_lo = mag - _POS_VALUES[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(pick_lo, lo, hi).astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x80, code)   # the sign is kept, zero included
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def e8m0_value(codes):
    c = np.asarray(codes, np.uint8).astype(np.float64)
    return np.where(c == 255, np.nan, np.exp2(c - 127.0))


def e8m0_scale_code(amax):
    """Shared-exponent code for a block with largest magnitude ``amax``."""
    amax = np.asarray(amax, np.float64)
    _, ex = np.frexp(amax)                 # amax = m * 2^ex, m in [0.5, 1)
    shared_exp = (ex - 1) - 8              # floor(log2(amax)) - emax(E4M3)
    code = np.clip(shared_exp + 127, 0, 254)
    return np.where(amax > 0, code, 0).astype(np.uint8)


def quantize(x, axis):
    """Quantise ``x`` in blocks of 32 along ``axis`` (a multiple of 32 long).

    Returns (payload uint8 with x's shape, scale codes uint8 with that axis
    divided by 32)."""
    x = np.asarray(x, np.float64)
    xm = np.moveaxis(x, axis, -1)
    shp = xm.shape
    if shp[-1] % BLOCK:
        raise ValueError("quantised axis must be a multiple of 32")
    blocks = xm.reshape(shp[:-1] + (shp[-1] // BLOCK, BLOCK))
    amax = np.max(np.abs(blocks), axis=-1)
    sc = e8m0_scale_code(amax)
    scaled = blocks / e8m0_value(sc)[..., None]
    payload = e4m3_encode(scaled).reshape(shp)
    return np.moveaxis(payload, -1, axis), np.moveaxis(sc, -1, axis)


_DECODE_TABLE = e4m3_decode(np.arange(256, dtype=np.uint8))
_E8M0_TABLE = e8m0_value(np.arange(256, dtype=np.uint8))


def dequantize(payload, scale, axis):
    """Exact fp64 value of an MXFP8 tensor: decode(payload) * 2^(scale - 127),
    one scale per 32 elements along ``axis`` (decoding through 256-entry tables
    of e4m3_decode and e8m0_value)."""
    v = _DECODE_TABLE[np.asarray(payload, np.uint8)]
    s = np.repeat(_E8M0_TABLE[np.asarray(scale, np.uint8)], BLOCK, axis=axis)
    return v * s
