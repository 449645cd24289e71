"""Guard bands around every device buffer the library writes.

A memory sanitizer is not available for these runs, so out-of-bounds writes
are caught the old way: the packed experts, the scratch and the output are
carved out of one device allocation with 4 KB of sentinel bytes before and
after each of them (the scratch ends exactly at the size moe_plan reported).
Every weight format, activation format and kernel path runs once; afterwards
every sentinel byte must be intact, the inputs unchanged and the output must
still match the oracle.  The same forward also runs in a zero-filled
allocation and must give the same output bytes: nothing may depend on what the
scratch held before the call.
"""

import numpy as np
import pytest
import torch

import moe_testlib as tl

pytestmark = pytest.mark.gpu

GUARD = 4096
SENTINEL = 0xA5


@pytest.fixture(scope="module")
def lib():
    from block_quantised_moe_gb300 import build
    build.build()
    from block_quantised_moe_gb300 import abi, layer
    return abi, layer


def _round(n, a=256):
    return (n + a - 1) // a * a


CASES = (
    # register-dequant kernels (16 tokens), every format pair
    [(w, a, f, 16, False) for (w, a, f) in [
        ("nvfp4", "silu", "bf16"), ("nvfp4", "silu", "nvfp4"), ("nvfp4", "silu", "mxfp8"),
        ("nvfp4", "relu2", "bf16"), ("nvfp4", "relu2", "nvfp4"), ("mxfp4", "relu2", "mxfp8"),
        ("mxfp4", "relu2", "bf16"), ("mxfp4", "silu", "mxfp8")]]
    # tcgen05 kernels (700 tokens x top-2 on 8 experts: ragged 128-token tiles)
    + [(w, a, f, 700, False) for (w, a, f) in [
        ("nvfp4", "silu", "bf16"), ("nvfp4", "silu", "nvfp4"), ("nvfp4", "silu", "mxfp8"),
        ("nvfp4", "relu2", "bf16"), ("mxfp4", "relu2", "mxfp8"), ("mxfp4", "relu2", "bf16")]]
    # block-scaled FP4 kernels (W4A4 with the weights' FP4 tiles)
    + [("nvfp4", "silu", "nvfp4", 700, True), ("nvfp4", "relu2", "nvfp4", 700, True)]
)


def _run_guarded(abi, ck, wplan, packed_bytes, plan, scratch_bytes, x, ids, w, T, H, fill):
    """One forward in a single allocation [guard | packed | guard | scratch | guard | out | guard]
    pre-filled with `fill`; returns (host copy of the allocation, offsets, sizes, ends)."""
    out_bytes = T * H * 2
    sizes = [_round(packed_bytes), _round(scratch_bytes), _round(out_bytes)]
    offs, o = [], GUARD
    for sz in sizes:
        offs.append(o)
        o += sz + GUARD
    buf = torch.full((o,), fill, dtype=torch.uint8, device="cuda")
    base = buf.data_ptr()
    assert base % 256 == 0
    p_packed, p_scratch, p_out = (base + off for off in offs)
    abi.moe_prepare_weights(wplan, ck.w13_codes, ck.w13_scales, ck.w13_global, ck.w2_codes, ck.w2_scales,
                            ck.w2_global, p_packed)
    b = abi.moe_bind(plan, p_scratch, scratch_bytes, p_packed, x, ids, w, T, p_out)
    abi.moe_run(b)
    rc, st = abi.moe_device_status(b)
    torch.cuda.synchronize()
    abi.moe_destroy_binding(b)
    assert rc == abi.MOE_OK and st[0] == 0
    return buf.cpu().numpy(), offs, sizes, [packed_bytes, scratch_bytes, out_bytes]


@pytest.mark.parametrize("wfmt,act,afmt,T,fp4_tiles", CASES)
def test_no_write_outside_the_buffers(lib, wfmt, act, afmt, T, fp4_tiles):
    abi, layer = lib
    E, H, I, K = 8, 256, 512, 2
    ck = layer.make_experts_gpu(E, H, I, wfmt, act)
    flags = abi.MOE_WFLAG_FP4_TILES if fp4_tiles else 0
    wplan, packed_bytes = abi.moe_plan_weights(E, H, I, wfmt, act, flags)
    plan, scratch_bytes, _ = abi.moe_plan(wplan, K, T, afmt)
    cfg = dict(E=E, H=H, I=I, K=K, zipf=None)
    x, ids, w = tl.make_inputs(cfg, T, seed=T + 1)
    x0, ids0, w0 = x.clone(), ids.clone(), w.clone()
    runs = {}
    for fill in (SENTINEL, 0):
        runs[fill] = _run_guarded(abi, ck, wplan, packed_bytes, plan, scratch_bytes, x, ids, w, T, H, fill)
    host, offs, sizes, ends = runs[SENTINEL]
    for name, off, end, sz in zip(("packed", "scratch", "out"), offs, ends, sizes):
        before = host[off - GUARD:off]
        after = host[off + end:off + sz + GUARD]
        assert (before == SENTINEL).all(), f"{name}: a write landed in the guard band before it"
        bad = np.nonzero(after != SENTINEL)[0]
        assert bad.size == 0, f"{name}: {bad.size} bytes written past its end (first at +{bad[0]})"
    assert torch.equal(x, x0) and torch.equal(ids, ids0) and torch.equal(w, w0), "an input was modified"
    out_bytes = ends[2]
    out_raw = host[offs[2]:offs[2] + out_bytes].reshape(T, H * 2)
    assert not (out_raw == SENTINEL).all(axis=1).any(), "an output row was left unwritten"
    # nothing may depend on the initial contents of scratch: a zero-filled run
    # gives the same bytes as the sentinel-filled one
    host0 = runs[0][0]
    assert np.array_equal(host0[offs[2]:offs[2] + out_bytes], host[offs[2]:offs[2] + out_bytes]), \
        "the output depends on the initial contents of scratch"
    out = torch.from_numpy(out_raw.copy()).view(torch.bfloat16).view(T, H)
    tl.check_close(out.float().numpy(), tl.oracle_forward(ck, H, I, x, ids, w, afmt),
                   f"guarded {wfmt}/{act}/{afmt} T={T}")
    abi.moe_destroy_plan(plan)
    abi.moe_destroy_weight_plan(wplan)
