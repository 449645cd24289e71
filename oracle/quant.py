"""NVFP4 and MX block quantisers / dequantisers (oracle).

Test infrastructure: see the package docstring for who may import this.

NVFP4 (b12x project page, "What's in here": quantization.nvfp4 row quantizer;
vLLM docs "b12x Linear and MoE Backends", "Supported Configurations": NVFP4
weights with BF16 or NVFP4 activations):

    g      = amax / (6 * 448)                  FP32 global scale
    s_b    = E4M3_RNE_sat( (amax_b / 6) / g )  one E4M3 scale per 16 elements
    d_b    = float(s_b) * g                    FP32
    q_i    = E2M1_RNE_sat( x_i / d_b )         0 when d_b == 0
    x^_i   = E2M1(q_i) * E4M3(s_b) * g

``amax`` is taken over the whole matrix for weights (one global per expert and
per matrix: gate, up, down) and over one row for activations (one global per
token row).  With amax = 0 the global, the scales and the codes are all zero.

MXFP4 / MXFP8 (b12x project page, "PCIe DMA wire modes": E8M0 scales, one per
32 values; vLLM docs "b12x Linear and MoE Backends": MXFP8 activations for
MXFP4 MoE) use the OCP microscaling rule for the shared exponent:

    X      = floor(log2(amax_b)) - emax_elem   (emax 2 for E2M1, 8 for E4M3),
             clamped to [-127, 127]; X = -127 when amax_b = 0
    s_b    = X + 127                           E8M0 byte
    q_i    = ELEM_RNE_sat( x_i / 2^X )
    x^_i   = ELEM(q_i) * 2^X

Every step is an FP32 operation in the order written (numpy float32 division is
IEEE round-to-nearest), so a GPU quantiser that performs the same FP32
operations produces the same bytes.
"""

from __future__ import annotations

import numpy as np

from . import codecs

NVFP4_BLOCK = 16
MX_BLOCK = 32
E2M1_MAX = np.float32(6.0)
E4M3_MAX = np.float32(448.0)
NVFP4_GLOBAL_DIV = np.float32(6.0 * 448.0)  # 2688, exact in FP32
MX_EMAX = {"e2m1": 2, "e4m3": 8}


def _f32(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float32)


# ------------------------------------------------------------------- NVFP4


def nvfp4_global(amax) -> np.ndarray:
    """FP32 global scale g = amax / (6*448)."""
    return _f32(amax) / NVFP4_GLOBAL_DIV


def nvfp4_quantize_with_global(x: np.ndarray, g: np.ndarray):
    """Quantise rows of ``x`` [R, C] with per-row FP32 globals ``g`` [R].

    Returns (codes [R, C/2] packed nibbles, scales [R, C/16] E4M3 bytes).
    """
    x = _f32(x)
    R, C = x.shape
    assert C % NVFP4_BLOCK == 0
    g = _f32(g).reshape(R, 1, 1)
    blk = x.reshape(R, C // NVFP4_BLOCK, NVFP4_BLOCK)
    amax_b = np.max(np.abs(blk), axis=2, keepdims=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        s_val = (amax_b / E2M1_MAX) / g
    s_val = np.where(g > 0, s_val, np.float32(0.0)).astype(np.float32)
    s = codecs.e4m3_encode(s_val)
    d = codecs.e4m3_decode(s) * g  # FP32 multiply
    with np.errstate(divide="ignore", invalid="ignore"):
        v = blk / d
    v = np.where(d > 0, v, np.float32(0.0)).astype(np.float32)
    q = codecs.e2m1_encode(v)
    q = np.where(d > 0, q, np.uint8(0)).astype(np.uint8)
    return codecs.pack_nibbles(q.reshape(R, C)), s.reshape(R, C // NVFP4_BLOCK)


def nvfp4_quantize_rows(x: np.ndarray):
    """Activation quantiser: one FP32 global per row.  Returns (codes, scales, g[R])."""
    x = _f32(x)
    g = nvfp4_global(np.max(np.abs(x), axis=1))
    codes, scales = nvfp4_quantize_with_global(x, g)
    return codes, scales, g


def nvfp4_quantize_tensor(w: np.ndarray):
    """Weight quantiser: one FP32 global for the whole matrix.  Returns (codes, scales, g)."""
    w = _f32(w)
    g = nvfp4_global(np.max(np.abs(w)))
    codes, scales = nvfp4_quantize_with_global(w, np.full(w.shape[0], g, dtype=np.float32))
    return codes, scales, np.float32(g)


def nvfp4_dequant(codes: np.ndarray, scales: np.ndarray, g) -> np.ndarray:
    """x^ = E2M1(q) * E4M3(s) * g; ``g`` is a scalar or one value per row."""
    codes = np.asarray(codes, dtype=np.uint8)
    R = codes.shape[0]
    vals = codecs.e2m1_decode(codecs.unpack_nibbles(codes))  # [R, C]
    C = vals.shape[1]
    sc = np.repeat(codecs.e4m3_decode(scales), NVFP4_BLOCK, axis=1)
    gg = _f32(g).reshape(-1, 1) if np.ndim(g) else _f32(g)
    return ((vals * sc) * gg).astype(np.float32).reshape(R, C)


# ---------------------------------------------------------------------- MX


def mx_quantize(x: np.ndarray, elem: str):
    """OCP MX quantiser over 32-element blocks along rows.

    ``elem`` is "e2m1" (MXFP4; codes packed two per byte) or "e4m3" (MXFP8;
    one byte per code).  Returns (codes, scales [R, C/32] E8M0 bytes).
    """
    x = _f32(x)
    R, C = x.shape
    assert C % MX_BLOCK == 0
    blk = x.reshape(R, C // MX_BLOCK, MX_BLOCK)
    amax_b = np.max(np.abs(blk), axis=2)
    X = np.full(amax_b.shape, -127, dtype=np.int32)
    nz = amax_b > 0
    if np.any(nz):
        X[nz] = codecs.floor_log2(amax_b[nz]) - MX_EMAX[elem]
    X = np.clip(X, -127, 127)
    scale_bytes = (X + 127).astype(np.uint8)
    pow2 = np.ldexp(np.float32(1.0), X).astype(np.float32)[..., None]
    v = (blk / pow2).astype(np.float32)
    if elem == "e2m1":
        q = codecs.e2m1_encode(v).reshape(R, C)
        return codecs.pack_nibbles(q), scale_bytes
    if elem == "e4m3":
        return codecs.e4m3_encode(v).reshape(R, C), scale_bytes
    raise ValueError(elem)


def mx_dequant(codes: np.ndarray, scales: np.ndarray, elem: str) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    if elem == "e2m1":
        vals = codecs.e2m1_decode(codecs.unpack_nibbles(codes))
    elif elem == "e4m3":
        vals = codecs.e4m3_decode(codes)
    else:
        raise ValueError(elem)
    sc = np.repeat(codecs.e8m0_decode(scales), MX_BLOCK, axis=1)
    return (vals * sc).astype(np.float32)


# ------------------------------------------------ quantise-dequantise helpers


def qdq_rows(x: np.ndarray, afmt: str) -> np.ndarray:
    """Activation path: x -> dequant(quant(x)) per row, or x itself for bf16."""
    x = _f32(x)
    if afmt == "bf16":
        return x
    if afmt == "nvfp4":
        c, s, g = nvfp4_quantize_rows(x)
        return nvfp4_dequant(c, s, g)
    if afmt == "mxfp8":
        c, s = mx_quantize(x, "e4m3")
        return mx_dequant(c, s, "e4m3")
    raise ValueError(afmt)


def quantize_weight_matrix(w: np.ndarray, wfmt: str):
    """Checkpoint-style weight quantiser for one [N, K] matrix.

    NVFP4: (codes, scales, g) with a per-matrix global.  MXFP4: (codes, scales, None).
    """
    if wfmt == "nvfp4":
        return nvfp4_quantize_tensor(w)
    if wfmt == "mxfp4":
        c, s = mx_quantize(w, "e2m1")
        return c, s, None
    raise ValueError(wfmt)


def dequant_weight_matrix(codes, scales, g, wfmt: str) -> np.ndarray:
    if wfmt == "nvfp4":
        return nvfp4_dequant(codes, scales, np.float32(g))
    if wfmt == "mxfp4":
        return mx_dequant(codes, scales, "e2m1")
    raise ValueError(wfmt)
