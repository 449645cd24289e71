"""GPU packer (moe_prepare_weights) against an unpacking of its documented layout.

The packed buffer holds, per stage (W13, then W2), every 128-row block of an
expert as 64-K steps of mma.m16n8k16 A-fragment code bytes (slot-order K,
gate / up rows interleaved 8 + 8 per 16-row tile) followed by the step's block
scales, then an [E][4] FP32 table of global scales, then (optionally) the
block-scaled FP4 MMA's 128 x 256 code tiles (128-byte swizzle) with their scales
in tensor-memory order.  This test undoes that layout on the CPU and must
recover the checkpoint codes, scales and globals bit-exactly, each checkpoint
nibble and scale byte from exactly one packed position.
"""

import numpy as np
import pytest
import torch

from block_quantised_moe_gb300 import synth

pytestmark = pytest.mark.gpu


def align(v, a=256):
    return (v + a - 1) // a * a


def src_row(tile, rr, gated, I):
    """Checkpoint row of row rr (0..15) of 16-row tile `tile` (8 gate + 8 up rows when gated)."""
    if gated:
        return np.where(rr < 8, tile * 8 + rr, I + tile * 8 + rr - 8)
    return tile * 16 + rr


def unpack_fragments(seg, E, R, K, gated, I, bs):
    per = 64 // bs
    nsteps, nblk, step = K // 64, R // 128, 4096 + 128 * per
    v = seg.reshape(E, nblk, nsteps, step)
    # codes: [blk, step q, tile in block, lane t, register i, byte j]
    cb = v[..., :4096].reshape(E, nblk, nsteps, 8, 32, 4, 4)
    blk, q, tl, t, i, j = np.indices((nblk, nsteps, 8, 32, 4, 4))
    row = src_row(blk * 8 + tl, (t >> 2) + 8 * (j & 1), gated, I)
    k = 64 * q + 32 * (i >> 1) + 8 * (i & 1) + (t & 3) + 4 * (j >> 1)  # low nibble; high nibble is k + 16
    nib = np.zeros((E, R, K), np.uint8)
    nib[:, row, k] = cb & 0xF
    nib[:, row, k + 16] = cb >> 4
    cnt = np.zeros((R, K), np.int64)
    np.add.at(cnt, (row, k), 1)
    np.add.at(cnt, (row, k + 16), 1)
    assert (cnt == 1).all(), "code positions"
    codes = nib[:, :, 0::2] | (nib[:, :, 1::2] << 4)
    # scales: [blk, q, tile in block, lane group g, byte b]; b = (block, row lo/hi) pairs
    sb = v[..., 4096:].reshape(E, nblk, nsteps, 8, 8, 2 * per)
    blk, q, tl, g, b = np.indices((nblk, nsteps, 8, 8, 2 * per))
    row = src_row(blk * 8 + tl, g + 8 * ((b >> 1) & 1), gated, I)
    col = per * q + (b & 1) + 2 * (b >> 2)
    sc = np.zeros((E, R, K // bs), np.uint8)
    sc[:, row, col] = sb
    cnt = np.zeros((R, K // bs), np.int64)
    np.add.at(cnt, (row, col), 1)
    assert (cnt == 1).all(), "scale positions"
    return codes, sc


def unpack_fp4_tiles(seg, E, R, K, gated, I):
    nblk, nkb = R // 128, K // 256
    tb = seg.reshape(E, nblk, nkb, 16384 + 2048)
    r, c, b = np.indices((128, 8, 16))
    pos = (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ r) & 7) * 16 + b
    blk, kb = np.indices((nblk, nkb))
    codes = np.zeros((E, R, K // 2), np.uint8)
    row = src_row(blk[..., None, None, None] * 8 + r // 16, r % 16, gated, I)
    col = kb[..., None, None, None] * 128 + c * 16 + b
    codes[:, row, col] = tb[:, :, :, pos]
    words = tb[..., 16384:].reshape(E, nblk, nkb, 512, 4)
    w, byte = np.indices((512, 4))
    st, lane, cc = w >> 7, (w >> 2) & 31, w & 3
    rr = lane + 32 * cc
    row = src_row(blk[..., None, None] * 8 + rr // 16, rr % 16, gated, I)
    col = kb[..., None, None] * 16 + st * 4 + byte
    sc = np.zeros((E, R, K // 16), np.uint8)
    sc[:, row, col] = words
    cnt = np.zeros((R, K // 16), np.int64)
    np.add.at(cnt, (row, col), 1)
    assert (cnt == 1).all(), "FP4 tile scale positions"
    return codes, sc


@pytest.mark.parametrize("wfmt,act,fp4_tiles", [("nvfp4", "silu", True), ("nvfp4", "relu2", True),
                                                ("nvfp4", "silu", False), ("mxfp4", "relu2", False),
                                                ("mxfp4", "silu", False)])
def test_packer_layout_round_trips(wfmt, act, fp4_tiles):
    from block_quantised_moe_gb300 import build
    build.build()
    from block_quantised_moe_gb300 import layer
    E, H, I = 3, 512, 256
    gated = act == "silu"
    n13, bs = (2 if gated else 1) * I, 16 if wfmt == "nvfp4" else 32
    ref = synth.make_random_codes(E, H, I, wfmt, gated, seed=11)
    dev = {k: (v.cuda() if v is not None else None) for k, v in ref.items()}
    ck = layer.CheckpointExperts(wfmt, act, dev["w13_codes"], dev["w13_scales"], dev["w13_global"],
                                 dev["w2_codes"], dev["w2_scales"], dev["w2_global"])
    packed = layer.PackedLayer(ck, H, I, fp4_tiles=fp4_tiles)
    buf = packed.packed.cpu().numpy()
    blk13 = n13 * H // 2 + n13 * H // bs
    blk2 = H * I // 2 + H * I // bs
    off_c2 = align(E * blk13)
    off_g = align(off_c2 + E * blk2)
    off_t13 = align(off_g + E * 16)
    t13 = (n13 // 128) * (H // 256) * (16384 + 2048)
    t2 = (H // 128) * (I // 256) * (16384 + 2048)
    off_t2 = align(off_t13 + E * t13)
    assert buf.size == (align(off_t2 + E * t2) if fp4_tiles else off_t13)

    for seg, rows, K, g, ck_codes, ck_scales in (
            (buf[:E * blk13], n13, H, gated, ref["w13_codes"], ref["w13_scales"]),
            (buf[off_c2:off_c2 + E * blk2], H, I, False, ref["w2_codes"], ref["w2_scales"])):
        codes, scales = unpack_fragments(seg, E, rows, K, g, I, bs)
        assert np.array_equal(codes, ck_codes.numpy())
        assert np.array_equal(scales, ck_scales.numpy())

    glob = buf[off_g:off_g + E * 16].view(np.float32).reshape(E, 4)
    if wfmt == "nvfp4":
        g13 = ref["w13_global"].numpy()
        want = np.stack([g13[:, 0], g13[:, 1] if gated else np.ones(E, np.float32),
                         ref["w2_global"].numpy(), np.ones(E, np.float32)], axis=1)
    else:
        want = np.ones((E, 4), np.float32)
    assert np.array_equal(glob, want)

    if fp4_tiles:
        for seg, rows, K, g, ck_codes, ck_scales in (
                (buf[off_t13:off_t13 + E * t13], n13, H, gated, ref["w13_codes"], ref["w13_scales"]),
                (buf[off_t2:off_t2 + E * t2], H, I, False, ref["w2_codes"], ref["w2_scales"])):
            codes, scales = unpack_fp4_tiles(seg, E, rows, K, g, I)
            assert np.array_equal(codes, ck_codes.numpy())
            assert np.array_equal(scales, ck_scales.numpy())
