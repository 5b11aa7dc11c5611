"""FP8 E4M3 codec and the block-128 dynamic quantizer of the lightning indexer.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

[P3] section "Indexer 的结构与计算流程": the indexer query and key are
quantized dynamically to FP8 with block size 128; section "双 KV 缓存" stores
the key in float8_e4m3fn with a float32 scale per token.

The 8-bit format is the OCP 8-bit floating point E4M3 encoding: 1 sign bit,
4 exponent bits with bias 7, 3 mantissa bits, subnormals at exponent field 0,
no infinities, and S.1111.111 (0x7F / 0xFF) the only NaN codes; the largest
finite magnitude is 448.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
BLOCK = 128


def _decode_one(code: int) -> float:
    sign = -1.0 if (code >> 7) & 1 else 1.0
    exp_field = (code >> 3) & 0xF
    man = code & 0x7
    if exp_field == 0xF and man == 0x7:
        return float("nan")
    if exp_field == 0:
        # subnormal: 0.mmm * 2^(1 - bias)
        return sign * (man / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp_field - 7)


_TABLE = np.array([_decode_one(c) for c in range(256)], dtype=np.float64)


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """Decode uint8 E4M3 codes to float64 (exact)."""
    codes = np.asarray(codes, dtype=np.uint8)
    return _TABLE[codes]


# Non-negative finite values in code order (codes 0x00..0x7E are monotonic).
_POS_VALUES = _TABLE[:0x7F].copy()


def encode_e4m3_rne_satfinite(y: np.ndarray) -> np.ndarray:
    """Round float values to the nearest E4M3 code, ties to the even code,
    saturating magnitudes above 448 to +-448 (no NaN produced for finite input);
    the sign bit always follows the input's sign.

    Done by search over the 127 non-negative representable values: the two
    neighbours of |y| are found, the nearer one taken, and on an exact tie the
    one whose code is even (mantissa LSB 0) is taken.
    """
    y = np.asarray(y, dtype=np.float64)
    a = np.minimum(np.abs(y), E4M3_MAX)
    hi = np.searchsorted(_POS_VALUES, a, side="left")  # first value >= a
    hi = np.clip(hi, 0, len(_POS_VALUES) - 1)
    lo = np.clip(hi - 1, 0, len(_POS_VALUES) - 1)
    v_hi = _POS_VALUES[hi]
    v_lo = _POS_VALUES[lo]
    d_hi = v_hi - a
    d_lo = a - v_lo
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo).astype(np.uint8)
    # exact hits (including a == 0)
    code = np.where(v_hi == a, hi.astype(np.uint8), code)
    # the sign bit is kept for every result, zero included (a negative value
    # that rounds to zero gives the negative-zero code 0x80)
    neg = np.signbit(y)
    return (code | (neg.astype(np.uint8) << 7)).astype(np.uint8)


def quantize_block128(x: np.ndarray):
    """Dynamic block-128 FP8 quantization of the last axis.

    For every block of 128 contiguous elements: amax = max |x|;
    scale = amax / 448 (scale = 1 when amax == 0); code = RNE-satfinite(x / scale).
    The scale and the division are float32 operations (the scale is stored as
    float32 per [P3] "双 KV 缓存"), so the result is defined bit for bit.

    Returns (codes uint8 with x's shape, scales float32 with the last axis
    divided by 128).
    """
    x = np.asarray(x, dtype=np.float32)
    n = x.shape[-1]
    if n % BLOCK != 0:
        raise ValueError("last axis must be a multiple of 128")
    xb = x.reshape(x.shape[:-1] + (n // BLOCK, BLOCK))
    amax = np.max(np.abs(xb), axis=-1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    y = (xb / scale[..., None]).astype(np.float32)
    codes = encode_e4m3_rne_satfinite(y.astype(np.float64))
    return codes.reshape(x.shape), scale
