"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/moe.h declares, and rejects bad arguments with status
codes before touching the device."""

import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def abi():
    from block_quantised_moe_gb300 import build
    build.build()
    from block_quantised_moe_gb300 import abi as a
    return a


def declared_entry_points():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"^MOE_API\s+[\w\s\*]*?\b(moe_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_plan_bind_run_contract():
    names = declared_entry_points()
    for n in ("moe_plan_weights", "moe_prepare_weights", "moe_plan", "moe_bind", "moe_run"):
        assert n in names


def test_library_exports_every_declared_symbol(abi):
    out = subprocess.run(["nm", "-D", "--defined-only", abi.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (moe_\w+)$", out, flags=re.M))
    declared = set(declared_entry_points())
    assert declared <= exported, declared - exported
    assert set(abi.EXPORTS) == declared
    for n in declared:
        assert hasattr(abi._lib, n)


def test_status_strings(abi):
    assert abi.moe_status_str(0) == "MOE_OK"
    assert abi.moe_status_str(4) == "MOE_ERR_SCRATCH_TOO_SMALL"
    assert abi.moe_status_str(99) == "MOE_ERR_UNKNOWN"


@pytest.mark.parametrize("args,code", [
    ((0, 256, 512, "nvfp4", "silu"), 1),
    ((8, 200, 512, "nvfp4", "silu"), 2),    # hidden not a multiple of 128
    ((8, 256, 96, "nvfp4", "silu"), 2),     # intermediate not a multiple of 64
    ((8, 256, 512, 7, "silu"), 1),
    ((8, 256, 512, "nvfp4", 9), 1),
    ((4096, 256, 512, "nvfp4", "silu"), 2),
])
def test_plan_weights_rejects(abi, args, code):
    with pytest.raises(abi.MoeError) as ei:
        abi.moe_plan_weights(*args)
    assert ei.value.status == code


def test_plan_weights_sizes(abi):
    E, H, I = 8, 256, 512
    h, n = abi.moe_plan_weights(E, H, I, "nvfp4", "silu")
    codes = E * (2 * I * H + H * I) // 2
    scales = E * (2 * I * H + H * I) // 16
    assert codes + scales <= n <= codes + scales + 16 * E + 5 * 256
    abi.moe_destroy_weight_plan(h)


def test_is_supported_and_plan_errors(abi):
    w, _ = abi.moe_plan_weights(8, 256, 512, "nvfp4", "silu")
    wm, _ = abi.moe_plan_weights(8, 256, 512, "mxfp4", "relu2")
    assert abi.moe_is_supported(w, 2, 16, "bf16") == 0
    assert abi.moe_is_supported(w, 2, 16, "nvfp4") == 0
    assert abi.moe_is_supported(w, 2, 16, "mxfp8") == 0
    assert abi.moe_is_supported(wm, 4, 16, "mxfp8") == 0
    assert abi.moe_is_supported(wm, 4, 16, "nvfp4") == abi.MOE_ERR_UNSUPPORTED
    assert abi.moe_is_supported(w, 0, 16, "bf16") == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_is_supported(w, 17, 16, "bf16") == abi.MOE_ERR_UNSUPPORTED
    assert abi.moe_is_supported(w, 2, 0, "bf16") == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_is_supported(w, 2, 16, 9) == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_is_supported(None, 2, 16, "bf16") == abi.MOE_ERR_INVALID_ARG
    with pytest.raises(abi.MoeError):
        abi.moe_plan(wm, 4, 16, "nvfp4")
    p, nbytes, m_tile = abi.moe_plan(w, 2, 16, "bf16")
    assert m_tile == 16 and nbytes > 0
    p2, nbytes2, _ = abi.moe_plan(w, 2, 1024, "bf16")
    assert nbytes2 > nbytes  # scratch grows with capacity, not with live counts
    abi.moe_destroy_plan(p), abi.moe_destroy_plan(p2)
    abi.moe_destroy_weight_plan(w), abi.moe_destroy_weight_plan(wm)


def test_bind_rejects_without_touching_the_device(abi):
    w, _ = abi.moe_plan_weights(8, 256, 512, "nvfp4", "silu")
    p, nbytes, _ = abi.moe_plan(w, 2, 16, "bf16")
    fake = 1 << 40  # an aligned address that is never dereferenced on the host
    ok = dict(scratch=fake, scratch_bytes=nbytes, packed=fake, x=fake, topk_ids=fake,
              topk_weights=fake, num_tokens=16, out=fake)

    def bind(**kw):
        a = dict(ok)
        a.update(kw)
        return abi.moe_bind(p, a["scratch"], a["scratch_bytes"], a["packed"], a["x"], a["topk_ids"],
                            a["topk_weights"], a["num_tokens"], a["out"])

    b = bind()
    abi.moe_destroy_binding(b)
    for kw, code in [
        (dict(scratch_bytes=nbytes - 1), abi.MOE_ERR_SCRATCH_TOO_SMALL),
        (dict(num_tokens=17), abi.MOE_ERR_CAPACITY),
        (dict(num_tokens=-1), abi.MOE_ERR_INVALID_ARG),
        (dict(scratch=None), abi.MOE_ERR_INVALID_ARG),
        (dict(scratch=fake + 16), abi.MOE_ERR_INVALID_ARG),   # scratch must be 256-byte aligned
        (dict(x=fake + 2), abi.MOE_ERR_INVALID_ARG),
        (dict(out=None), abi.MOE_ERR_INVALID_ARG),
        (dict(topk_ids=None), abi.MOE_ERR_INVALID_ARG),
    ]:
        with pytest.raises(abi.MoeError) as ei:
            bind(**kw)
        assert ei.value.status == code, kw
    # zero tokens binds without activation pointers and runs as a no-op
    b0 = bind(num_tokens=0, x=None, topk_ids=None, topk_weights=None, out=None, packed=None)
    abi.moe_run(b0, 0)
    abi.moe_destroy_binding(b0)
    abi.moe_destroy_plan(p)
    abi.moe_destroy_weight_plan(w)


def test_quantize_argument_checks(abi):
    import ctypes
    call = abi._lib.moe_quantize
    fake = 1 << 40
    assert call(9, 0, 0, fake, 1, 1, 32, fake, fake, None, None) == abi.MOE_ERR_INVALID_ARG
    assert call(abi.MOE_Q_NVFP4, abi.MOE_G_PER_ROW, 0, fake, 1, 1, 24, fake, fake, fake, None) == 1
    assert call(abi.MOE_Q_NVFP4, abi.MOE_G_NONE, 0, fake, 1, 1, 32, fake, fake, fake, None) == 1
    assert call(abi.MOE_Q_NVFP4, abi.MOE_G_PER_ROW, 0, fake, 1, 1, 32, fake, fake, None, None) == 1
    assert call(abi.MOE_Q_MXFP8, abi.MOE_G_NONE, 0, fake, 1, 1, 48, fake, fake, None, None) == 1
    assert call(abi.MOE_Q_MXFP8, abi.MOE_G_PER_ROW, 0, fake, 1, 1, 64, fake, fake, fake, None) == 1
    assert call(abi.MOE_Q_MXFP8, abi.MOE_G_NONE, 0, fake, 0, 1, 64, fake, fake, None, None) == 0  # empty
    assert call(abi.MOE_Q_MXFP8, abi.MOE_G_NONE, 0, fake + 8, 1, 1, 64, fake, fake, None, None) == 1
    del ctypes


def test_prepare_weights_argument_checks(abi):
    w, _ = abi.moe_plan_weights(8, 256, 512, "nvfp4", "silu")
    fake = 1 << 40
    call = abi._lib.moe_prepare_weights
    assert call(w, fake, fake, None, fake, fake, fake, fake, None) == 1   # NVFP4 needs globals
    assert call(w, fake, fake, fake, fake, fake, fake, fake + 8, None) == 1  # misaligned packed
    assert call(None, fake, fake, fake, fake, fake, fake, fake, None) == 1
    wm, _ = abi.moe_plan_weights(8, 256, 512, "mxfp4", "relu2")
    assert call(wm, fake, fake, fake, fake, fake, None, fake, None) == 1  # MXFP4 takes no globals
    abi.moe_destroy_weight_plan(w), abi.moe_destroy_weight_plan(wm)


def test_single_launch_option_follows_the_plan(abi):
    # decode plans (at most 1024 pairs) of the supported formats may run as one
    # launch; a plan with tensor-core experts (1024+ pairs) may not
    wp, _ = abi.moe_plan_weights(128, 2048, 768, "nvfp4", "silu")
    small, _, _ = abi.moe_plan(wp, 8, 64, "bf16")
    big, _, _ = abi.moe_plan(wp, 8, 4096, "bf16")
    abi.moe_plan_set_option(small, abi.MOE_OPT_SINGLE_LAUNCH, 0)
    abi.moe_plan_set_option(small, abi.MOE_OPT_SINGLE_LAUNCH, 1)
    with pytest.raises(abi.MoeError) as ei:
        abi.moe_plan_set_option(big, abi.MOE_OPT_SINGLE_LAUNCH, 1)
    assert ei.value.status == abi.MOE_ERR_UNSUPPORTED
    abi.moe_plan_set_option(big, abi.MOE_OPT_SINGLE_LAUNCH, 0)
    for bad in ((99, 1), (abi.MOE_OPT_SINGLE_LAUNCH, 2)):
        with pytest.raises(abi.MoeError) as ei:
            abi.moe_plan_set_option(small, *bad)
        assert ei.value.status == abi.MOE_ERR_INVALID_ARG
    # MXFP4 weights with NVFP4 activations are not a supported pair at all
    wmx, _ = abi.moe_plan_weights(128, 4096, 1024, "mxfp4", "relu2")
    mx, _, _ = abi.moe_plan(wmx, 4, 64, "mxfp8")
    abi.moe_plan_set_option(mx, abi.MOE_OPT_SINGLE_LAUNCH, 1)
    # FP32 output (a tensor-parallel rank's partial) excludes the single launch, both ways round
    with pytest.raises(abi.MoeError) as ei:
        abi.moe_plan_set_option(mx, abi.MOE_OPT_OUT_F32, 1)
    assert ei.value.status == abi.MOE_ERR_UNSUPPORTED
    abi.moe_plan_set_option(mx, abi.MOE_OPT_SINGLE_LAUNCH, 0)
    abi.moe_plan_set_option(mx, abi.MOE_OPT_OUT_F32, 1)
    with pytest.raises(abi.MoeError) as ei:
        abi.moe_plan_set_option(mx, abi.MOE_OPT_SINGLE_LAUNCH, 1)
    assert ei.value.status == abi.MOE_ERR_UNSUPPORTED
    with pytest.raises(abi.MoeError) as ei:
        abi.moe_plan_set_option(mx, abi.MOE_OPT_OUT_F32, 3)
    assert ei.value.status == abi.MOE_ERR_INVALID_ARG
    abi.moe_plan_set_option(mx, abi.MOE_OPT_OUT_F32, 0)
    for p in (small, big, mx):
        abi.moe_destroy_plan(p)
    abi.moe_destroy_weight_plan(wp)
    abi.moe_destroy_weight_plan(wmx)
