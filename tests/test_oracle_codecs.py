"""Pins of the oracle's element / scale codecs against library casts and the bit layouts."""

import math

import numpy as np
import pytest
import torch

from oracle import codecs


def test_e2m1_table_matches_bit_layout():
    # OCP E2M1: s.ee.m, bias 1; exponent 0 is subnormal (m/2).  Written from the
    # bit layout, independently of the magnitude table in the oracle.
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        mag = (m / 2.0) if e == 0 else 2.0 ** (e - 1) * (1 + m / 2.0)
        want = -mag if s else mag
        got = float(codecs.E2M1_TABLE[code])
        assert got == want and math.copysign(1, got) == math.copysign(1, want), code
    assert sorted(set(abs(float(v)) for v in codecs.E2M1_TABLE)) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_e4m3_table_matches_torch_all_codes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    got = codecs.E4M3_TABLE
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))
    assert got[0x7E] == 448.0


def test_e8m0_table_matches_torch_all_codes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).float().numpy()
    got = codecs.E8M0_TABLE
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(ref[:255], got[:255])
    for b in range(255):  # exact powers of two
        assert got[b] == np.float32(2.0 ** (b - 127))


def test_e4m3_encode_matches_torch_rne_in_range():
    rng = np.random.default_rng(1)
    # random magnitudes across the whole range, plus every midpoint (tie) between codes
    v = (rng.standard_normal(200000) * np.exp2(rng.integers(-12, 9, 200000))).astype(np.float32)
    grid = codecs.E4M3_TABLE[:0x7F].astype(np.float64)
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (grid[:-1] + grid[1:]) / 2)  # exact in FP32
    v = np.concatenate([v, mids, -mids, grid.astype(np.float32)])
    v = v[np.abs(v) <= 448.0]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = codecs.e4m3_encode(v)
    assert np.array_equal(ref, got)


def test_e4m3_encode_saturates():
    v = np.array([448.0, 449.0, 463.9, 464.0, 500.0, 1e30, -1e30, -460.0], dtype=np.float32)
    got = codecs.e4m3_encode(v)
    assert list(got) == [0x7E] * 6 + [0xFE, 0xFE]


def test_e2m1_encode_ties_saturation_sign():
    # Round-to-nearest-even ties on the value grid {0,.5,1,1.5,2,3,4,6}.
    cases = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0,
             0.2: 0.0, 0.26: 0.5, 2.6: 3.0, 4.9: 4.0, 5.1: 6.0, 6.0: 6.0, 7.0: 6.0, 1e9: 6.0}
    for x, want in cases.items():
        for sgn in (1.0, -1.0):
            c = int(codecs.e2m1_encode(np.array([sgn * x], dtype=np.float32))[0])
            assert codecs.E2M1_TABLE[c] == sgn * want, (x, sgn, c)
            assert (c >> 3) == (1 if sgn < 0 else 0)  # sign kept, even for -0
    assert int(codecs.e2m1_encode(np.array([-0.0], dtype=np.float32))[0]) == 8
    assert int(codecs.e2m1_encode(np.array([0.0], dtype=np.float32))[0]) == 0


def test_e2m1_encode_is_nearest_brute_force():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(20000) * 3).astype(np.float32)
    got = codecs.e2m1_encode(v)
    vals = codecs.E2M1_TABLE.astype(np.float64)
    for x, c in zip(v.astype(np.float64), got):
        xs = min(abs(x), 6.0) * (1 if x >= 0 else -1)
        best = np.min(np.abs(vals - xs))
        assert abs(vals[c] - xs) == best


def test_floor_log2_exact_over_float32_range():
    for k in range(-149, 128):
        p = np.float32(2.0 ** k)
        assert codecs.floor_log2(np.array([p]))[0] == k
        if k < 127:
            nxt = np.nextafter(np.float32(2.0 ** (k + 1)), np.float32(0))
            assert codecs.floor_log2(np.array([nxt]))[0] == k


def test_nibble_order_low_nibble_first():
    # Reading of the modelopt_nvfp4 source format: element 2j low nibble, 2j+1 high.
    codes = np.array([[1, 2, 0xF, 0x8]], dtype=np.uint8)
    packed = codecs.pack_nibbles(codes)
    assert packed.tolist() == [[0x21, 0x8F]]
    assert np.array_equal(codecs.unpack_nibbles(packed), codes)


@pytest.mark.parametrize("n", [2, 32, 4096])
def test_nibble_round_trip(n):
    rng = np.random.default_rng(n)
    codes = rng.integers(0, 16, (3, n)).astype(np.uint8)
    assert np.array_equal(codecs.unpack_nibbles(codecs.pack_nibbles(codes)), codes)
