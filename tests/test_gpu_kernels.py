"""GPU checks of the individual stages through the C ABI: quantisers and routing
bit-exact against the oracle, determinism and slot-permutation invariance of the
output (bit-exact), dropped ids, the host-buffer entry point and graph capture."""

import numpy as np
import pytest
import torch

from block_quantised_moe_gb300 import synth
import moe_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from block_quantised_moe_gb300 import build
    build.build()
    from block_quantised_moe_gb300 import abi, layer
    return abi, layer


# -------------------------------------------------------------- quantisers

def _special_rows(R, C, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(R, C, generator=g) * torch.exp2(torch.randint(-20, 20, (R, 1), generator=g).float())
    x[0] = 0.0                                   # all-zero row
    x[1, :C // 2] = 0.0                          # zero blocks in a live row
    x[2] = torch.randn(C, generator=g) * 1e-40   # subnormal FP32 values
    x[3, ::7] = -0.0
    x[4] = torch.tensor([0.25, 0.75, 1.25, 2.5, 5.0, 6.0, 448.0, 2688.0] * (C // 8))  # ties on the grids
    x[5] = torch.randn(C, generator=g) * 1e30
    return x


@pytest.mark.parametrize("C", [512, 4096])  # per-row NVFP4: a warp per row up to 2048 columns, a CTA above
@pytest.mark.parametrize("src_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("mode", ["nvfp4_row", "nvfp4_tensor", "mxfp4", "mxfp8"])
def test_quantiser_bit_exact(lib, mode, src_dtype, C):
    from oracle import quant
    abi, _ = lib
    B, R = 3, 24
    x = torch.stack([_special_rows(R, C, s) for s in range(B)]).to(src_dtype)
    xd = x.cuda()
    xf = x.float().numpy()
    if mode.startswith("nvfp4"):
        codes = torch.empty(B, R, C // 2, dtype=torch.uint8, device="cuda")
        scales = torch.empty(B, R, C // 16, dtype=torch.uint8, device="cuda")
        per_row = mode == "nvfp4_row"
        g = torch.empty(B * R if per_row else B, dtype=torch.float32, device="cuda")
        abi.moe_quantize(abi.MOE_Q_NVFP4, abi.MOE_G_PER_ROW if per_row else abi.MOE_G_PER_TENSOR,
                         xd, B, R, C, codes, scales, g)
        torch.cuda.synchronize()
        for b in range(B):
            if per_row:
                c, s, gg = quant.nvfp4_quantize_rows(xf[b])
                assert np.array_equal(g.view(B, R)[b].cpu().numpy(), gg)
            else:
                c, s, gg = quant.nvfp4_quantize_tensor(xf[b])
                assert g[b].item() == gg
            assert np.array_equal(scales[b].cpu().numpy(), s), f"scales batch {b}"
            assert np.array_equal(codes[b].cpu().numpy(), c), f"codes batch {b}"
    else:
        elem = "e2m1" if mode == "mxfp4" else "e4m3"
        cb = C // 2 if mode == "mxfp4" else C
        codes = torch.empty(B, R, cb, dtype=torch.uint8, device="cuda")
        scales = torch.empty(B, R, C // 32, dtype=torch.uint8, device="cuda")
        abi.moe_quantize(abi.MOE_Q_MXFP4 if mode == "mxfp4" else abi.MOE_Q_MXFP8, abi.MOE_G_NONE,
                         xd, B, R, C, codes, scales, None)
        torch.cuda.synchronize()
        for b in range(B):
            c, s = quant.mx_quantize(xf[b], elem)
            assert np.array_equal(scales[b].cpu().numpy(), s), f"scales batch {b}"
            assert np.array_equal(codes[b].cpu().numpy(), c), f"codes batch {b}"


# ------------------------------------------------------------------ routing

@pytest.mark.parametrize("T,K,E", [(1, 8, 128), (16, 2, 8), (64, 8, 128), (128, 8, 256), (341, 3, 512),
                                   (129, 8, 64), (8192, 8, 256), (3000, 4, 512), (1, 1, 1), (1025, 1, 1),
                                   (600, 4, 3)])
def test_routing_bit_exact(lib, T, K, E):
    from oracle import routing
    abi, layer = lib
    ck = layer.CheckpointExperts(
        "nvfp4", "silu", torch.zeros(E, 128, 64, dtype=torch.uint8, device="cuda"),
        torch.zeros(E, 128, 8, dtype=torch.uint8, device="cuda"), torch.zeros(E, 2, device="cuda"),
        torch.zeros(E, 128, 32, dtype=torch.uint8, device="cuda"),
        torch.zeros(E, 128, 4, dtype=torch.uint8, device="cuda"), torch.zeros(E, device="cuda"))
    packed = layer.PackedLayer(ck, 128, 64)
    rng = np.random.default_rng(T + K + E)
    ids = rng.integers(0, E, (T, K)).astype(np.int32)
    if T > 4:
        ids[1, 0], ids[3, K - 1] = -5, E  # dropped
    x = torch.zeros(T, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(T, K, device="cuda")
    plan = layer.Plan(packed, K, T, "bf16")
    out = torch.empty(T, 128, dtype=torch.bfloat16, device="cuda")
    b = plan.bind(x, torch.from_numpy(ids).cuda(), w, out)
    b.run()
    got = b.routing()
    want = routing.route(ids, E, plan.m_tile)
    for key in ("counts", "offsets", "sorted_pair", "pair_pos"):
        assert np.array_equal(got[key], want[key]), key
    rc, st = b.device_status()
    assert rc == abi.MOE_OK
    assert st[1] == want["dropped"] and bool(st[0] & 1) == (want["dropped"] > 0)


# ------------------------------------------------- determinism and invariance

@pytest.fixture(scope="module")
def decode_layer(lib):
    _, layer = lib
    cfg = synth.CONFIGS["decode_e128_h2048_i768_k8"]
    ck = layer.make_experts_gpu(cfg["E"], cfg["H"], cfg["I"], cfg["wfmt"], cfg["act"])
    return cfg, ck, layer.PackedLayer(ck, cfg["H"], cfg["I"])


def _forward(lib, packed, x, ids, w, K, afmt="bf16"):
    _, layer = lib
    plan = layer.Plan(packed, K, x.shape[0], afmt)
    out = torch.empty(x.shape[0], packed.H, dtype=torch.bfloat16, device="cuda")
    b = plan.bind(x, ids, w, out)
    b.run()
    torch.cuda.synchronize()
    return out, b, plan


def test_repeat_runs_bit_identical(lib, decode_layer):
    cfg, ck, packed = decode_layer
    x, ids, w = tl.make_inputs(cfg, 64)
    _, layer = lib
    plan = layer.Plan(packed, cfg["K"], 64, "bf16")
    out = torch.empty(64, cfg["H"], dtype=torch.bfloat16, device="cuda")
    b = plan.bind(x, ids, w, out)
    b.run()
    first = out.clone()
    for _ in range(3):
        out.zero_()
        b.run()
        torch.cuda.synchronize()
        assert torch.equal(out, first)


def test_permuting_topk_slots_is_bit_identical(lib, decode_layer):
    cfg, ck, packed = decode_layer
    x, ids, w = tl.make_inputs(cfg, 16)
    perm = torch.tensor([3, 7, 0, 5, 1, 6, 2, 4], device="cuda")
    a, _, _ = _forward(lib, packed, x, ids, w, cfg["K"])
    b, _, _ = _forward(lib, packed, x, ids[:, perm].contiguous(), w[:, perm].contiguous(), cfg["K"])
    assert torch.equal(a, b)


def test_dropped_ids_are_reported_and_skipped(lib, decode_layer):
    abi, _ = lib
    cfg, ck, packed = decode_layer
    x, ids, w = tl.make_inputs(cfg, 8)
    ids2 = ids.clone()
    ids2[0, 3], ids2[5, 0], ids2[7, 7] = -1, cfg["E"], 100000
    out, b, _ = _forward(lib, packed, x, ids2, w, cfg["K"])
    rc, st = b.device_status()
    assert rc == abi.MOE_OK and st[0] & 1 and st[1] == 3
    y_ref = tl.oracle_forward(ck, cfg["H"], cfg["I"], x, ids2, w, "bf16")
    tl.check_close(out.float().cpu().numpy(), y_ref, "dropped ids")


def test_fully_dropped_token_and_duplicate_ids(lib, decode_layer):
    # A token whose every id is out of range gets an exact zero row (the output
    # starts as NaN), and a token routed twice to one expert counts both pairs.
    abi, layer = lib
    cfg, ck, packed = decode_layer
    K = cfg["K"]
    x, ids, w = tl.make_inputs(cfg, 16)
    ids2 = ids.clone()
    ids2[2, :] = -1
    ids2[9, 1] = ids2[9, 0]
    plan = layer.Plan(packed, K, 16, "bf16")
    out = torch.full((16, cfg["H"]), float("nan"), dtype=torch.bfloat16, device="cuda")
    b = plan.bind(x, ids2, w, out)
    b.run()
    torch.cuda.synchronize()
    rc, st = b.device_status()
    assert rc == abi.MOE_OK and st[1] == K
    assert torch.equal(out[2], torch.zeros_like(out[2]))
    y_ref = tl.oracle_forward(ck, cfg["H"], cfg["I"], x, ids2, w, "bf16")
    tl.check_close(out.float().cpu().numpy(), y_ref, "dropped token, duplicate ids")


def test_zero_weights_and_zero_tokens(lib, decode_layer):
    _, layer = lib
    cfg, ck, packed = decode_layer
    x, ids, w = tl.make_inputs(cfg, 4)
    out, _, _ = _forward(lib, packed, x, ids, torch.zeros_like(w), cfg["K"])
    assert torch.count_nonzero(out) == 0
    plan = layer.Plan(packed, cfg["K"], 4, "bf16")
    empty = torch.empty(0, cfg["H"], dtype=torch.bfloat16, device="cuda")
    b = plan.bind(empty, ids[:0], w[:0], empty)
    b.run()
    torch.cuda.synchronize()


def test_host_buffer_entry_point_matches_device_run(lib, decode_layer):
    abi, layer = lib
    cfg, ck, packed = decode_layer
    x, ids, w = tl.make_inputs(cfg, 16)
    ref, _, _ = _forward(lib, packed, x, ids, w, cfg["K"])
    plan = layer.Plan(packed, cfg["K"], 16, "bf16")
    xd, idd, wd = torch.empty_like(x), torch.empty_like(ids), torch.empty_like(w)
    od = torch.empty(16, cfg["H"], dtype=torch.bfloat16, device="cuda")
    b = plan.bind(xd, idd, wd, od)
    xh, ih, wh = x.cpu().pin_memory(), ids.cpu().pin_memory(), w.cpu().pin_memory()
    oh = torch.empty(16, cfg["H"], dtype=torch.bfloat16).pin_memory()
    abi.moe_run_host(b.handle, xh, ih, wh, oh)
    assert torch.equal(oh, ref.cpu())


def test_cuda_graph_capture_and_replay(lib, decode_layer):
    _, layer = lib
    cfg, ck, packed = decode_layer
    x, ids, w = tl.make_inputs(cfg, 4)
    ref, _, _ = _forward(lib, packed, x, ids, w, cfg["K"])
    plan = layer.Plan(packed, cfg["K"], 4, "bf16")
    out = torch.empty(4, cfg["H"], dtype=torch.bfloat16, device="cuda")
    b = plan.bind(x, ids, w, out)
    b.run()  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.capture_begin()
        b.run(s)
        g.capture_end()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
