"""Pins of the oracle's NVFP4 / MX quantisers: exact on-grid round trips,
nearest-code brute force, zero blocks, and the MXFP8 block size printed on the
b12x project page ("PCIe DMA wire modes")."""

import os

import numpy as np
import pytest

from oracle import codecs, quant

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
E4M3_POS = codecs.E4M3_TABLE[1:0x7F]  # positive finite E4M3 values


def _on_grid_nvfp4(rng, R, C, k_global, min_scale=2.0 ** -6):
    """Rows x = E2M1(q) * s_b * 2^k with one +-6 per block and one 6*448*2^k per row,
    so that amax = 2688 * 2^k, g = 2^k and every block scale is recovered exactly."""
    q = rng.integers(0, 16, (R, C)).astype(np.uint8)
    nb = C // 16
    s = rng.choice(E4M3_POS[E4M3_POS >= min_scale], size=(R, nb)).astype(np.float32)
    s[:, 0] = 448.0
    for r in range(R):
        for b in range(nb):
            q[r, b * 16 + rng.integers(0, 16)] = 7 | (8 * rng.integers(0, 2))
    g = np.float32(2.0 ** k_global)
    x = codecs.E2M1_TABLE[q] * np.repeat(s, 16, axis=1) * g
    return x.astype(np.float32), q, codecs.e4m3_encode(s), g


@pytest.mark.parametrize("k_global", [-10, 0, 3])
def test_nvfp4_rows_round_trip_exact(k_global):
    rng = np.random.default_rng(10 + k_global)
    x, q, s_bytes, g = _on_grid_nvfp4(rng, 6, 128, k_global)
    codes, scales, gg = quant.nvfp4_quantize_rows(x)
    assert np.all(gg == g)
    assert np.array_equal(scales, s_bytes)
    # -0 and +0 codes decode alike; compare decoded values and the packed magnitude bits
    assert np.array_equal(codecs.unpack_nibbles(codes) & 7, q & 7)
    assert np.array_equal(quant.nvfp4_dequant(codes, scales, gg), x)


def test_nvfp4_tensor_global_is_matrix_amax():
    rng = np.random.default_rng(3)
    # halving keeps every scale a normal E4M3 value, so the grid is preserved
    x, q, s_bytes, g = _on_grid_nvfp4(rng, 8, 64, 0, min_scale=2.0 ** -5)
    x[1:] *= np.float32(0.5)  # only row 0 keeps the 2688 element
    codes, scales, gg = quant.nvfp4_quantize_tensor(x)
    assert gg == np.float32(1.0)
    assert np.array_equal(quant.nvfp4_dequant(codes, scales, gg), x)


def test_nvfp4_codes_are_nearest_for_their_scale():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((16, 256)) * np.exp2(rng.integers(-6, 6, (16, 1)))).astype(np.float32)
    codes, scales, g = quant.nvfp4_quantize_rows(x)
    # scale: E4M3 nearest to (amax_b/6)/g
    blk = x.reshape(16, 16, 16)
    amax_b = np.abs(blk).max(axis=2)
    want_s = (amax_b.astype(np.float32) / np.float32(6)) / g[:, None].astype(np.float32)
    got_s = codecs.e4m3_decode(scales).astype(np.float64)
    err = np.abs(got_s - want_s)
    alt = np.abs(codecs.E4M3_TABLE[:0x7F].astype(np.float64)[None, None, :] - want_s[..., None]).min(axis=2)
    assert np.all(err <= alt)
    # codes: nearest grid value of x/d in the E2M1 grid (brute force over all 8 magnitudes)
    d = (codecs.e4m3_decode(scales) * g[:, None]).astype(np.float32)
    v = (blk / d[..., None]).astype(np.float64)
    vals = codecs.unpack_nibbles(codes).reshape(16, 16, 16)
    got = codecs.E2M1_TABLE[vals].astype(np.float64)
    clipped = np.clip(v, -6, 6)
    best = np.abs(np.abs(clipped)[..., None] - np.array(codecs.E2M1_MAGNITUDES)).min(axis=-1)
    assert np.all(np.abs(got - clipped) == best)


def test_nvfp4_zero_row_and_zero_block():
    x = np.zeros((2, 64), dtype=np.float32)
    x[1, 16:32] = 3.0
    codes, scales, g = quant.nvfp4_quantize_rows(x)
    assert g[0] == 0 and np.all(codes[0] == 0) and np.all(scales[0] == 0)
    assert np.all(scales[1, [0, 2, 3]] == 0) and np.all(codecs.unpack_nibbles(codes)[1, :16] == 0)
    deq = quant.nvfp4_dequant(codes, scales, g)
    assert np.all(deq[0] == 0) and np.all(deq[1, :16] == 0) and np.all(deq[1, 32:] == 0)
    # g = 3/2688 is not exact in FP32, so the non-zero block comes back to within rounding
    assert np.allclose(deq[1, 16:32], 3.0, rtol=1e-6, atol=0)


def test_nvfp4_rounding_ties_inside_a_block():
    # Row with amax 2688 -> g = 1; block 1 holds 6*s with s = 1, so d = 1 and the
    # elements 0.25, 0.75, 2.5, 5 sit exactly on E2M1 ties.
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 0] = 2688.0
    x[0, 16:22] = [6.0, 0.25, 0.75, 2.5, 5.0, -1.25]
    codes, scales, g = quant.nvfp4_quantize_rows(x)
    assert g[0] == 1.0 and codecs.e4m3_decode(scales)[0, 1] == 1.0
    deq = quant.nvfp4_dequant(codes, scales, g)[0, 16:22]
    assert deq.tolist() == [6.0, 0.0, 1.0, 2.0, 4.0, -1.0]


@pytest.mark.parametrize("elem,emax,grid", [
    ("e2m1", 2, codecs.E2M1_TABLE[:8]),
    ("e4m3", 8, codecs.E4M3_TABLE[:0x7F]),
])
def test_mx_round_trip_exact(elem, emax, grid):
    rng = np.random.default_rng(5)
    R, C = 4, 256
    top = grid[grid >= 2.0 ** emax]  # magnitudes whose floor(log2) is emax
    X = rng.integers(-20, 20, (R, C // 32))
    vals = rng.choice(grid, size=(R, C)).astype(np.float32) * rng.choice([-1, 1], size=(R, C))
    for r in range(R):
        for b in range(C // 32):
            vals[r, b * 32 + rng.integers(0, 32)] = rng.choice(top)
    x = (vals * np.exp2(np.repeat(X, 32, axis=1))).astype(np.float32)
    codes, scales = quant.mx_quantize(x, elem)
    assert np.array_equal(scales.astype(np.int64) - 127, X)
    assert np.array_equal(quant.mx_dequant(codes, scales, elem), x)


def test_mx_zero_block_and_clamp():
    x = np.zeros((1, 64), dtype=np.float32)
    x[0, 32] = 2.0 ** -140  # subnormal: X clamps at -127
    codes, scales = quant.mx_quantize(x, "e4m3")
    assert scales.tolist() == [[0, 0]]
    assert np.all(codes[0, :32] == 0)


def test_mxfp8_block_bytes_match_page_golden():
    facts = {}
    for line in open(os.path.join(GOLDEN, "mxfp8_wire_block.txt")):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            facts[k] = int(v)
    x = np.random.default_rng(6).standard_normal((1, facts["values"])).astype(np.float32)
    codes, scales = quant.mx_quantize(x, "e4m3")
    assert scales.size == facts["scale_bytes"]
    assert codes.nbytes + scales.nbytes == facts["total_bytes"]
    assert x.size * 2 == facts["bf16_bytes"]
