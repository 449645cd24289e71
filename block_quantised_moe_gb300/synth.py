"""Seeded synthetic inputs for the fused MoE layer.

This module is the only code that both the CUDA path and the CPU oracle
consume.  It draws random numbers and nothing else of the method: no
quantisation, no expert arithmetic.  The router (softmax -> top-k ->
renormalise) lives here because the op takes ``topk_ids`` / ``topk_weights``
as inputs rather than computing them.

Recipe (base seed 0 unless a caller says otherwise):

* activations  x ~ N(0, 1) drawn in FP32 and rounded to BF16, stream seed*1000+1;
* router       logits ~ N(0, 1) [T, E], stream seed*1000+2; optional per-expert
               bias -s*ln(r_e) with r a random permutation of 1..E (stream
               seed*1000+3), a Zipf(s) prior that skews expert load; softmax in
               float64, top-K by descending probability (ties: lower expert id),
               weights renormalised over the K picks and stored as FP32;
* experts      FP32 weights ~ N(0, 0.02), expert e from stream seed*1000+100+e,
               drawn in the order gate [I,H], up [I,H], down [H,I] (gated) or
               w1 [I,H], down [H,I] (ReLU^2), so a layer does not depend on T;
* raw codes    uniform random checkpoint bytes (every E2M1 code, finite E4M3 or
               E8M0 scales) for edge-case tests of the byte paths.
"""

from __future__ import annotations

import numpy as np
import torch

WEIGHT_STD = 0.02

# Workloads, named by what they are.  ``tokens`` lists the batch sizes each one
# is run at; ``afmt`` is the activation format, ``wfmt`` the weight format.
CONFIGS = {
    "tiny_e8_h256_i512_k2": dict(
        E=8, H=256, I=512, K=2, tokens=(16,), wfmt="nvfp4", afmt="bf16", act="silu", zipf=None),
    "decode_e128_h2048_i768_k8": dict(
        E=128, H=2048, I=768, K=8, tokens=(1, 4, 16, 64), wfmt="nvfp4", afmt="bf16", act="silu", zipf=None),
    "decode_zipf_e256_h7168_i2048_k8": dict(
        E=256, H=7168, I=2048, K=8, tokens=(1, 8, 32, 128), wfmt="nvfp4", afmt="bf16", act="silu", zipf=1.1),
    "prefill_w4a16_e256_h7168_i2048_k8": dict(
        E=256, H=7168, I=2048, K=8, tokens=(8192,), wfmt="nvfp4", afmt="bf16", act="silu", zipf=None),
    "prefill_w4a4_e256_h7168_i2048_k8": dict(
        E=256, H=7168, I=2048, K=8, tokens=(8192,), wfmt="nvfp4", afmt="nvfp4", act="silu", zipf=None),
    "mxfp4_mxfp8_relu2_e128_h4096_i1024_k4": dict(
        E=128, H=4096, I=1024, K=4, tokens=(1, 64, 4096), wfmt="mxfp4", afmt="mxfp8", act="relu2", zipf=None),
}


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_x(T: int, H: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Activations [T, H] BF16."""
    g = _gen(seed * 1000 + 1, device)
    return torch.randn(T, H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_routing(T: int, E: int, K: int, seed: int = 0, zipf: float | None = None):
    """Router outputs (topk_ids int32 [T, K], topk_weights float32 [T, K]) on the CPU."""
    logits = torch.randn(T, E, generator=_gen(seed * 1000 + 2), dtype=torch.float32).double().numpy()
    if zipf is not None:
        ranks = torch.randperm(E, generator=_gen(seed * 1000 + 3)).numpy().astype(np.float64) + 1.0
        logits = logits - zipf * np.log(ranks)[None, :]
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    p = p / p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")[:, :K]
    pk = np.take_along_axis(p, order, axis=1)
    w = pk / pk.sum(axis=1, keepdims=True)
    return (torch.from_numpy(order.astype(np.int32)),
            torch.from_numpy(w.astype(np.float32)))


def make_expert_weights(e: int, H: int, I: int, gated: bool, seed: int = 0, device="cpu"):
    """FP32 weights of expert ``e``: ([gate, up] or [w1], down)."""
    g = _gen(seed * 1000 + 100 + e, device)
    n13 = 2 if gated else 1
    w13 = [torch.randn(I, H, generator=g, device=device) * WEIGHT_STD for _ in range(n13)]
    w2 = torch.randn(H, I, generator=g, device=device) * WEIGHT_STD
    return w13, w2


def make_random_codes(E: int, H: int, I: int, wfmt: str, gated: bool, seed: int = 0):
    """Uniform random checkpoint bytes (CPU tensors) covering every E2M1 code.

    Scales are finite, non-negative E4M3 bytes 0x00..0x7E (NVFP4) or E8M0 bytes
    in [117, 137] (MXFP4); NVFP4 globals are drawn in [1e-4, 1e-2).
    """
    g = _gen(seed * 1000 + 7)
    bs = 16 if wfmt == "nvfp4" else 32
    n13 = (2 if gated else 1) * I

    def codes(*shape):
        return torch.randint(0, 256, shape, generator=g, dtype=torch.int32).to(torch.uint8)

    def scales(*shape):
        if wfmt == "nvfp4":
            return torch.randint(0, 0x7F, shape, generator=g, dtype=torch.int32).to(torch.uint8)
        return torch.randint(117, 138, shape, generator=g, dtype=torch.int32).to(torch.uint8)

    out = dict(
        w13_codes=codes(E, n13, H // 2), w13_scales=scales(E, n13, H // bs),
        w2_codes=codes(E, H, I // 2), w2_scales=scales(E, H, I // bs),
        w13_global=None, w2_global=None)
    if wfmt == "nvfp4":
        out["w13_global"] = (torch.rand(E, n13 // I, generator=g) * 0.0099 + 1e-4).float()
        out["w2_global"] = (torch.rand(E, generator=g) * 0.0099 + 1e-4).float()
    return out
