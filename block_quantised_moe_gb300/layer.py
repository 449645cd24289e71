"""Device-memory plumbing around the C ABI: allocate with torch, call ``abi``.

Nothing here computes any part of the layer: quantisation, packing, routing,
the expert contractions and the combine all run in libmoe's kernels.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

from . import abi, synth


@dataclass
class CheckpointExperts:
    """Quantised experts on the device, in the checkpoint layout of moe_prepare_weights."""

    wfmt: str
    act: str
    w13_codes: torch.Tensor
    w13_scales: torch.Tensor
    w13_global: torch.Tensor | None
    w2_codes: torch.Tensor
    w2_scales: torch.Tensor
    w2_global: torch.Tensor | None

    @property
    def num_experts(self):
        return self.w13_codes.shape[0]


def quantize_matrices(w: torch.Tensor, wfmt: str):
    """Quantise a batch of FP32 matrices [B, N, K] on the GPU with moe_quantize.

    NVFP4 uses one global per matrix.  Returns (codes [B,N,K/2], scales [B,N,K/bs], global [B] | None).
    """
    B, N, Kd = w.shape
    dev = w.device
    codes = torch.empty(B, N, Kd // 2, dtype=torch.uint8, device=dev)
    if wfmt == "nvfp4":
        scales = torch.empty(B, N, Kd // 16, dtype=torch.uint8, device=dev)
        g = torch.empty(B, dtype=torch.float32, device=dev)
        abi.moe_quantize(abi.MOE_Q_NVFP4, abi.MOE_G_PER_TENSOR, w, B, N, Kd, codes, scales, g)
        return codes, scales, g
    scales = torch.empty(B, N, Kd // 32, dtype=torch.uint8, device=dev)
    abi.moe_quantize(abi.MOE_Q_MXFP4, abi.MOE_G_NONE, w, B, N, Kd, codes, scales, None)
    return codes, scales, None


def make_experts_gpu(E, H, I, wfmt, act, seed=0, device="cuda", gen_device=None) -> CheckpointExperts:
    """Seeded N(0, 0.02) FP32 experts (synth), quantised expert by expert on the GPU."""
    gated = act == "silu"
    n13 = 2 * I if gated else I
    bs = 16 if wfmt == "nvfp4" else 32
    c13 = torch.empty(E, n13, H // 2, dtype=torch.uint8, device=device)
    s13 = torch.empty(E, n13, H // bs, dtype=torch.uint8, device=device)
    c2 = torch.empty(E, H, I // 2, dtype=torch.uint8, device=device)
    s2 = torch.empty(E, H, I // bs, dtype=torch.uint8, device=device)
    g13 = torch.empty(E, n13 // I, dtype=torch.float32, device=device) if wfmt == "nvfp4" else None
    g2 = torch.empty(E, dtype=torch.float32, device=device) if wfmt == "nvfp4" else None
    for e in range(E):
        w13, w2 = synth.make_expert_weights(e, H, I, gated, seed, device=gen_device or device)
        a = torch.stack(w13).to(device)
        c, s, g = quantize_matrices(a, wfmt)
        c13[e].copy_(c.reshape(n13, H // 2))
        s13[e].copy_(s.reshape(n13, H // bs))
        if g is not None:
            g13[e].copy_(g)
        c, s, g = quantize_matrices(w2.to(device)[None], wfmt)
        c2[e].copy_(c[0])
        s2[e].copy_(s[0])
        if g is not None:
            g2[e].copy_(g[0])
    return CheckpointExperts(wfmt, act, c13, s13, g13, c2, s2, g2)


class PackedLayer:
    """Packed experts of one layer (moe_plan_weights + moe_prepare_weights)."""

    def __init__(self, ck: CheckpointExperts, hidden: int, intermediate: int, fp4_tiles: bool = False):
        self.wfmt, self.act = ck.wfmt, ck.act
        self.E, self.H, self.I = ck.num_experts, hidden, intermediate
        flags = abi.MOE_WFLAG_FP4_TILES if fp4_tiles else 0
        self.wplan, nbytes = abi.moe_plan_weights(self.E, hidden, intermediate, ck.wfmt, ck.act, flags)
        dev = ck.w13_codes.device
        self.packed = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        abi.moe_prepare_weights(self.wplan, ck.w13_codes, ck.w13_scales, ck.w13_global, ck.w2_codes,
                                ck.w2_scales, ck.w2_global, self.packed)

    def __del__(self):
        if getattr(self, "wplan", None):
            abi.moe_destroy_weight_plan(self.wplan)
            self.wplan = None


class Plan:
    """moe_plan for a capacity, with its scratch allocated once."""

    def __init__(self, layer: PackedLayer, top_k: int, max_tokens: int, afmt: str):
        self.layer, self.top_k, self.max_tokens, self.afmt = layer, top_k, max_tokens, afmt
        self.handle, self.scratch_bytes, self.m_tile = abi.moe_plan(layer.wplan, top_k, max_tokens, afmt)
        self.scratch = torch.empty(self.scratch_bytes, dtype=torch.uint8, device=layer.packed.device)

    def bind(self, x, topk_ids, topk_weights, out, packed=None):
        return Binding(self, x, topk_ids, topk_weights, out, packed)

    def __del__(self):
        if getattr(self, "handle", None):
            abi.moe_destroy_plan(self.handle)
            self.handle = None


class Binding:
    def __init__(self, plan: Plan, x, topk_ids, topk_weights, out, packed=None):
        self.plan = plan
        self.T = x.shape[0]
        self.keep = (x, topk_ids, topk_weights, out, packed)
        pk = plan.layer.packed if packed is None else packed
        self.handle = abi.moe_bind(plan.handle, plan.scratch, plan.scratch_bytes, pk, x, topk_ids,
                                   topk_weights, self.T, out)

    def run(self, stream=None):
        abi.moe_run(self.handle, stream)

    def device_status(self, stream=None):
        return abi.moe_device_status(self.handle, stream)

    def hidden(self):
        L = self.plan.layer
        return abi.moe_debug_hidden(self.handle, L.I, self.T * self.plan.top_k + L.E * self.plan.m_tile)

    def routing(self):
        L = self.plan.layer
        return abi.moe_debug_routing(self.handle, L.E, self.T * self.plan.top_k,
                                     self.T * self.plan.top_k + L.E * self.plan.m_tile)

    def __del__(self):
        if getattr(self, "handle", None):
            abi.moe_destroy_binding(self.handle)
            self.handle = None
