"""Element and scale codecs of the NVFP4 / MXFP4 / MXFP8 block formats (oracle).

Test infrastructure: see the package docstring for who may import this.

Formats named by the pages: NVFP4 and MXFP4 weights, NVFP4 / MXFP8 activations
(b12x project page, "What's in here": moe.fused_moe and quantization.{nvfp4,mxfp8};
vLLM docs "b12x Linear and MoE Backends", "Supported Configurations"), with
E8M0 scales one per 32 values for MXFP8 (b12x project page, "PCIe DMA wire
modes").  The bit layouts below are the OCP microscaling ones:

* E2M1  : s.ee.m, exponent bias 1, no inf/NaN.  Magnitudes of codes 0..7 are
          {0, 0.5, 1, 1.5, 2, 3, 4, 6}; bit 3 is the sign (code 8 is -0).
* E4M3FN: s.eeee.mmm, bias 7, max 448, no inf; 0x7F / 0xFF are NaN.
* E8M0  : unsigned exponent, value 2^(b-127); 0xFF is NaN.

Encoders round to nearest with ties to the even code (the code whose last
mantissa bit is 0) and saturate to the largest finite magnitude.  The sign bit
of the code is the sign bit of the input, so a negative input that rounds to
zero encodes as -0.

Everything here is written as table look-ups over the decoded value of every
code, which is slow but can be checked by eye.
"""

from __future__ import annotations

import numpy as np

# --------------------------------------------------------------------- decode

E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def e2m1_value(code: int) -> float:
    """Value of one 4-bit E2M1 code (bit 3 = sign, bits 2..0 index the magnitude)."""
    mag = E2M1_MAGNITUDES[code & 7]
    return -mag if code & 8 else mag


def e4m3_value(byte: int) -> float:
    """Value of one E4M3FN byte: sign, 4-bit exponent (bias 7), 3-bit mantissa."""
    sign = -1.0 if byte & 0x80 else 1.0
    exp = (byte >> 3) & 0xF
    man = byte & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:  # subnormal: 0.mmm * 2^(1-7)
        return sign * (man / 8.0) * 2.0 ** -6
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


def e8m0_value(byte: int) -> float:
    """Value of one E8M0 byte: 2^(byte-127); 0xFF is NaN."""
    if byte == 0xFF:
        return float("nan")
    return 2.0 ** (byte - 127)


# Lookup tables (float32, indexed by code) built from the scalar definitions.
E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float32)
E4M3_TABLE = np.array([e4m3_value(b) for b in range(256)], dtype=np.float32)
E8M0_TABLE = np.array([e8m0_value(b) for b in range(256)], dtype=np.float32)


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    """Decode an array of 4-bit codes (one code per uint8) to float32."""
    return E2M1_TABLE[np.asarray(codes, dtype=np.uint8) & 0xF]


def e4m3_decode(b: np.ndarray) -> np.ndarray:
    return E4M3_TABLE[np.asarray(b, dtype=np.uint8)]


def e8m0_decode(b: np.ndarray) -> np.ndarray:
    return E8M0_TABLE[np.asarray(b, dtype=np.uint8)]


# --------------------------------------------------------------------- encode


def _nearest_even(mag: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the nearest entry of the increasing ``grid`` for each ``mag``.

    ``mag`` must lie in [grid[0], grid[-1]].  An exact tie between two
    neighbours picks the even index; grid indices are magnitude codes, so this
    is "ties to the even code".  All arithmetic is float64 on values that are
    exactly float32, so the distance comparison is exact.
    """
    mag = np.asarray(mag, dtype=np.float64)
    hi = np.minimum(np.searchsorted(grid, mag, side="left"), len(grid) - 1)  # in [0, n-1]
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - grid[lo]
    d_hi = grid[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    return np.where(pick_hi, hi, lo)


_E2M1_GRID = np.array(E2M1_MAGNITUDES, dtype=np.float64)
# Non-negative finite E4M3 magnitudes, codes 0x00..0x7E, strictly increasing.
_E4M3_GRID = np.array([e4m3_value(b) for b in range(0x7F)], dtype=np.float64)


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """float32 -> 4-bit E2M1 code (uint8), RNE, saturating at 6, sign kept."""
    v = np.asarray(v, dtype=np.float32)
    assert np.all(np.isfinite(v)), "e2m1_encode: non-finite input"
    mag = np.minimum(np.abs(v).astype(np.float64), 6.0)
    idx = _nearest_even(mag, _E2M1_GRID).astype(np.uint8)
    return idx | (np.signbit(v).astype(np.uint8) << 3)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """float32 -> E4M3FN byte, RNE, saturating at 448 (never NaN), sign kept."""
    v = np.asarray(v, dtype=np.float32)
    assert np.all(np.isfinite(v)), "e4m3_encode: non-finite input"
    mag = np.minimum(np.abs(v).astype(np.float64), 448.0)
    idx = _nearest_even(mag, _E4M3_GRID).astype(np.uint8)
    return idx | (np.signbit(v).astype(np.uint8) << 7)


def floor_log2(a: np.ndarray) -> np.ndarray:
    """Exact floor(log2(a)) for finite a > 0 (float32), via the binary exponent.

    frexp writes a = m * 2^e with m in [0.5, 1), so floor(log2 a) = e - 1.
    """
    a = np.asarray(a, dtype=np.float32)
    assert np.all(a > 0) and np.all(np.isfinite(a))
    _, e = np.frexp(a.astype(np.float64))
    return (e - 1).astype(np.int32)


# ----------------------------------------------------------------- nibbles


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """[..., 2n] 4-bit codes -> [..., n] bytes; element 2j in the low nibble.

    Reading of "source_format=modelopt_nvfp4" (b12x project page, "Using it"):
    row-major codes, K contiguous, two codes per byte, even element low.
    """
    c = np.asarray(codes, dtype=np.uint8)
    assert c.shape[-1] % 2 == 0
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    """Inverse of :func:`pack_nibbles`."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out
