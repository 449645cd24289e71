"""GPU parity of the fused MoE through the C ABI against the CPU oracle.

Every workload is run on the GPU; outputs are compared with the oracle element
by element (all tokens where the oracle finishes in seconds, sampled tokens of
the full-size prefill / large-layer workloads).  Routing is compared bit-exactly,
and so are the quantised experts both sides start from.
"""

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


_LAYERS = {}


def gpu_layer(lib, E, H, I, wfmt, act, seed=0, fp4_tiles=False):
    abi, layer = lib
    key = (E, H, I, wfmt, act, seed, fp4_tiles)
    if key not in _LAYERS:
        ck = layer.make_experts_gpu(E, H, I, wfmt, act, seed=seed)
        _LAYERS.clear()  # keep at most one large layer resident
        _LAYERS[key] = (ck, layer.PackedLayer(ck, H, I, fp4_tiles=fp4_tiles))
    return _LAYERS[key]


def run(lib, packed, x, ids, w, top_k, afmt, max_tokens=None):
    abi, layer = lib
    T = x.shape[0]
    plan = layer.Plan(packed, top_k, max_tokens or max(T, 1), afmt)
    out = torch.empty(T, packed.H, dtype=torch.bfloat16, device="cuda")
    b = plan.bind(x, ids, w, out)
    b.run()
    torch.cuda.synchronize()
    return out, b, plan


def cfg_of(name):
    return synth.CONFIGS[name]


# ----------------------------------------------------------- small, all modes

TINY_MODES = [("nvfp4", "silu", "bf16"), ("nvfp4", "silu", "nvfp4"), ("nvfp4", "silu", "mxfp8"),
              ("mxfp4", "relu2", "mxfp8"), ("mxfp4", "relu2", "bf16"), ("nvfp4", "relu2", "bf16"),
              ("mxfp4", "silu", "mxfp8"), ("nvfp4", "relu2", "nvfp4")]


@pytest.mark.parametrize("wfmt,act,afmt", TINY_MODES)
def test_tiny_layer_every_mode(lib, wfmt, act, afmt):
    cfg = cfg_of("tiny_e8_h256_i512_k2")
    E, H, I, K = cfg["E"], cfg["H"], cfg["I"], cfg["K"]
    ck, packed = gpu_layer(lib, E, H, I, wfmt, act)
    x, ids, w = tl.make_inputs(cfg, 16)
    out, _, _ = run(lib, packed, x, ids, w, K, afmt)
    y_ref = tl.oracle_forward(ck, H, I, x, ids, w, afmt)
    tl.check_close(out.float().cpu().numpy(), y_ref, f"tiny {wfmt}/{act}/{afmt}")


@pytest.mark.parametrize("T", [1, 3, 16, 40])
def test_tiny_ragged_token_counts(lib, T):
    cfg = cfg_of("tiny_e8_h256_i512_k2")
    ck, packed = gpu_layer(lib, cfg["E"], cfg["H"], cfg["I"], "nvfp4", "silu")
    x, ids, w = tl.make_inputs(cfg, T, seed=T)
    out, _, _ = run(lib, packed, x, ids, w, cfg["K"], "bf16", max_tokens=64)
    tl.check_close(out.float().cpu().numpy(), tl.oracle_forward(ck, cfg["H"], cfg["I"], x, ids, w, "bf16"))


# ----------------------------------------------------- decode, full layers

@pytest.mark.parametrize("T", [1, 4, 16, 64])
def test_decode_e128_h2048(lib, T):
    cfg = cfg_of("decode_e128_h2048_i768_k8")
    ck, packed = gpu_layer(lib, cfg["E"], cfg["H"], cfg["I"], cfg["wfmt"], cfg["act"])
    x, ids, w = tl.make_inputs(cfg, T)
    out, b, _ = run(lib, packed, x, ids, w, cfg["K"], cfg["afmt"])
    tl.check_close(out.float().cpu().numpy(), tl.oracle_forward(ck, cfg["H"], cfg["I"], x, ids, w, "bf16"),
                   f"decode T={T}")


@pytest.mark.parametrize("T", [1, 64, 4096])
def test_mxfp4_mxfp8_relu2(lib, T):
    cfg = cfg_of("mxfp4_mxfp8_relu2_e128_h4096_i1024_k4")
    ck, packed = gpu_layer(lib, cfg["E"], cfg["H"], cfg["I"], cfg["wfmt"], cfg["act"])
    x, ids, w = tl.make_inputs(cfg, T)
    out, _, _ = run(lib, packed, x, ids, w, cfg["K"], cfg["afmt"])
    toks = tl.sample_tokens(T, 64)
    y_ref = tl.oracle_forward(ck, cfg["H"], cfg["I"], x, ids, w, cfg["afmt"], tokens=toks)
    tl.check_close(out.float().cpu().numpy()[toks], y_ref, f"mxfp4 T={T}")


@pytest.mark.parametrize("T", [1, 8, 32, 128])
def test_decode_zipf_e256_h7168(lib, T):
    cfg = cfg_of("decode_zipf_e256_h7168_i2048_k8")
    ck, packed = gpu_layer(lib, cfg["E"], cfg["H"], cfg["I"], cfg["wfmt"], cfg["act"])
    x, ids, w = tl.make_inputs(cfg, T)
    out, _, _ = run(lib, packed, x, ids, w, cfg["K"], cfg["afmt"])
    toks = tl.sample_tokens(T, 16)
    y_ref = tl.oracle_forward(ck, cfg["H"], cfg["I"], x, ids, w, cfg["afmt"], tokens=toks)
    tl.check_close(out.float().cpu().numpy()[toks], y_ref, f"zipf T={T}")


@pytest.mark.parametrize("name,fp4_tiles", [("prefill_w4a16_e256_h7168_i2048_k8", False),
                                            ("prefill_w4a4_e256_h7168_i2048_k8", False),
                                            ("prefill_w4a4_e256_h7168_i2048_k8", True)])
def test_prefill_e256_h7168(lib, name, fp4_tiles):
    cfg = cfg_of(name)
    ck, packed = gpu_layer(lib, cfg["E"], cfg["H"], cfg["I"], cfg["wfmt"], cfg["act"], fp4_tiles=fp4_tiles)
    T = cfg["tokens"][0]
    x, ids, w = tl.make_inputs(cfg, T)
    out, _, _ = run(lib, packed, x, ids, w, cfg["K"], cfg["afmt"])
    toks = tl.sample_tokens(T, 8, seed=1)
    y_ref = tl.oracle_forward(ck, cfg["H"], cfg["I"], x, ids, w, cfg["afmt"], tokens=toks)
    tl.check_close(out.float().cpu().numpy()[toks], y_ref, name)
    # every output row is finite and no row was left unwritten
    assert torch.isfinite(out.float()).all()


# --------------------------------------- full-length K, every token compared

FULL_K_MODES = [  # E, H, I, K, weights, activation, activations, FP4 tiles
    (8, 7168, 2048, 4, "nvfp4", "silu", "bf16", False),
    (8, 7168, 2048, 4, "nvfp4", "silu", "nvfp4", False),
    (8, 7168, 2048, 4, "nvfp4", "silu", "mxfp8", False),
    (8, 7168, 2048, 4, "nvfp4", "silu", "nvfp4", True),
    (8, 4096, 1024, 4, "mxfp4", "relu2", "mxfp8", False),
]


@pytest.mark.parametrize("E,H,I,K,wfmt,act,afmt,fp4_tiles", FULL_K_MODES)
def test_full_length_k_every_token(lib, E, H, I, K, wfmt, act, afmt, fp4_tiles):
    # The large-layer shapes (112 or 64 k-blocks of 64 per GEMM1 tile, 32 or 16
    # per GEMM2 tile) on 8 experts: 256 tokens x top-4 = 1024 pairs, about 128
    # per expert, so every expert runs on the tcgen05 kernels and ragged
    # 128-token tiles occur; every output element is compared with the oracle.
    T = 256
    ck, packed = gpu_layer(lib, E, H, I, wfmt, act, fp4_tiles=fp4_tiles)
    cfg = dict(E=E, H=H, I=I, K=K, zipf=None)
    x, ids, w = tl.make_inputs(cfg, T, seed=7)
    counts = np.bincount(ids.cpu().numpy().reshape(-1), minlength=E)
    assert counts.min() >= 32 and (counts % 128 != 0).any()
    out, b, _ = run(lib, packed, x, ids, w, K, afmt)
    assert b.device_status()[0] == 0
    y_ref = tl.oracle_forward(ck, H, I, x, ids, w, afmt)
    tl.check_close(out.float().cpu().numpy(), y_ref, f"full K {wfmt}/{act}/{afmt} tiles={fp4_tiles}")


# ------------------------------------------- tcgen05 path (experts with many pairs)

TC_MODES = [("nvfp4", "silu", "bf16"), ("nvfp4", "silu", "nvfp4"), ("nvfp4", "silu", "mxfp8"),
            ("nvfp4", "relu2", "bf16"), ("mxfp4", "relu2", "mxfp8"), ("mxfp4", "relu2", "bf16"),
            ("mxfp4", "silu", "mxfp8")]


@pytest.mark.parametrize("wfmt,act,afmt", TC_MODES)
@pytest.mark.parametrize("T", [512, 700])
def test_tcgen05_path_small_layer(lib, wfmt, act, afmt, T):
    # 8 experts x top-2: ~128-175 pairs per expert -> ragged 128-token tiles on the tcgen05 kernel
    cfg = dict(cfg_of("tiny_e8_h256_i512_k2"))
    E, H, I, K = cfg["E"], cfg["H"], cfg["I"], cfg["K"]
    ck, packed = gpu_layer(lib, E, H, I, wfmt, act)
    x, ids, w = tl.make_inputs(cfg, T, seed=T)
    out, _, _ = run(lib, packed, x, ids, w, K, afmt)
    y_ref = tl.oracle_forward(ck, H, I, x, ids, w, afmt)
    tl.check_close(out.float().cpu().numpy(), y_ref, f"tcgen05 {wfmt}/{act}/{afmt} T={T}")


@pytest.mark.parametrize("act", ["silu", "relu2"])
@pytest.mark.parametrize("T", [512, 700])
def test_block_scaled_fp4_path_small_layer(lib, act, T):
    # W4A4 with the weights' FP4 tiles: experts with 32+ pairs run on the
    # kind::mxf4nvf4 kernel, both operands as E2M1 codes with E4M3 block scales
    cfg = dict(cfg_of("tiny_e8_h256_i512_k2"))
    E, H, I, K = cfg["E"], cfg["H"], cfg["I"], cfg["K"]
    ck, packed = gpu_layer(lib, E, H, I, "nvfp4", act, fp4_tiles=True)
    x, ids, w = tl.make_inputs(cfg, T, seed=T)
    out, _, _ = run(lib, packed, x, ids, w, K, "nvfp4")
    tl.check_close(out.float().cpu().numpy(), tl.oracle_forward(ck, H, I, x, ids, w, "nvfp4"), f"fp4 {act} T={T}")


@pytest.mark.parametrize("wfmt,act,afmt", [("nvfp4", "silu", "bf16"), ("mxfp4", "relu2", "mxfp8")])
def test_tcgen05_and_decode_kernels_share_a_forward(lib, wfmt, act, afmt):
    # skewed routing: hot experts (>= 32 pairs) on tcgen05, the rest on the
    # register-dequant (NVFP4) or CUDA-core (MXFP4) kernel
    cfg = dict(E=64, H=256, I=512, K=4, zipf=1.5)
    ck, packed = gpu_layer(lib, cfg["E"], cfg["H"], cfg["I"], wfmt, act)
    x, ids, w = tl.make_inputs(cfg, 256, seed=5)
    counts = np.bincount(ids.cpu().numpy().reshape(-1), minlength=cfg["E"])
    assert counts.max() >= 32 and (counts[counts > 0] < 32).any()
    out, _, _ = run(lib, packed, x, ids, w, cfg["K"], afmt)
    tl.check_close(out.float().cpu().numpy(), tl.oracle_forward(ck, cfg["H"], cfg["I"], x, ids, w, afmt))
