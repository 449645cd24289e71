"""Tensor parallelism over the intermediate dimension.

Each of `world` ranks holds a contiguous slice of every expert's intermediate
features: the W13 rows of its slice of the gate and of the up projection (or of
the single W1 for ReLU^2) and the same slice of W2's columns.  A rank runs the
whole layer (routing, GEMM1, activation, GEMM2, combine) on its slice; its
output is a partial sum over the intermediate dimension, and the ranks add the
FP32 partials in rank order before rounding (the fused FP4 TP MoE of the b12x
project page, "What's in here").  The fixed order makes every rank's result the
same bytes, run after run.

What the slice boundary may not change: h is re-quantised between the
contractions per 32-element block for MXFP8 activations and not at all for
BF16 activations, so with slices on multiples of 64 every decision is the
unsharded layer's and the sum equals it up to the order of the FP32 additions.
NVFP4 activations quantise h with one global per token row over the whole
intermediate dimension, which one rank does not see; that would take a
cross-rank maximum per row first, and is not supported here.

The slicing and the reduction are host code on any torch.distributed backend;
the per-rank forward is the library's (moe_run with MOE_OPT_OUT_F32).
"""

from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist

from . import abi, layer


def shard_bounds(intermediate: int, rank: int, world: int) -> tuple[int, int]:
    """[lo, hi) of this rank's intermediate features (equal slices, multiples of 64)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of {world}")
    if intermediate % world != 0 or (intermediate // world) % 64 != 0:
        raise ValueError(f"intermediate {intermediate} does not split into {world} slices of a multiple of 64")
    n = intermediate // world
    return rank * n, (rank + 1) * n


def shard_arrays(w: dict, intermediate: int, gated: bool, rank: int, world: int) -> dict:
    """Slice checkpoint tensors (numpy or torch, the checkpoint layout) to a rank.

    w13_codes [E, N13, H/2] and w13_scales [E, N13, H/bs]: rows [lo, hi) of W1,
    or of the gate rows [0, I) and of the up rows [I, 2I) one after the other;
    w2_codes [E, H, I/2] and w2_scales [E, H, I/bs]: the columns of [lo, hi)
    (two E2M1 codes per byte, one scale per bs elements).  The global scales
    (NVFP4) belong to whole matrices and are kept."""
    lo, hi = shard_bounds(intermediate, rank, world)
    I = intermediate
    bs = I // w["w2_scales"].shape[2]
    if bs not in (16, 32):
        raise ValueError("scale block of W2 is neither 16 nor 32")
    is_torch = isinstance(w["w2_codes"], torch.Tensor)

    def rows(a):
        if not gated:
            return a[:, lo:hi]
        parts = (a[:, lo:hi], a[:, I + lo:I + hi])
        return torch.cat(parts, dim=1) if is_torch else np.concatenate(parts, axis=1)

    out = dict(w)
    out["w13_codes"] = rows(w["w13_codes"])
    out["w13_scales"] = rows(w["w13_scales"])
    out["w2_codes"] = w["w2_codes"][:, :, lo // 2:hi // 2]
    out["w2_scales"] = w["w2_scales"][:, :, lo // bs:hi // bs]
    for k in ("w13_codes", "w13_scales", "w2_codes", "w2_scales"):
        out[k] = out[k].contiguous() if is_torch else np.ascontiguousarray(out[k])
    return out


def shard_experts(ck: layer.CheckpointExperts, intermediate: int, rank: int, world: int) -> layer.CheckpointExperts:
    """A rank's slice of quantised experts on the device."""
    keys = ("w13_codes", "w13_scales", "w13_global", "w2_codes", "w2_scales", "w2_global")
    d = shard_arrays({k: getattr(ck, k) for k in keys}, intermediate, ck.act == "silu", rank, world)
    return layer.CheckpointExperts(wfmt=ck.wfmt, act=ck.act, **{k: d[k] for k in keys})


def ordered_all_reduce(t: torch.Tensor, group=None) -> torch.Tensor:
    """Sum of every rank's `t`, added in rank order (the same bytes on every rank)."""
    world = dist.get_world_size(group)
    parts = [torch.empty_like(t) for _ in range(world)]
    dist.all_gather(parts, t.contiguous(), group=group)
    acc = parts[0].clone()
    for p in parts[1:]:
        acc += p
    return acc


class TPLayer:
    """One rank's slice of a layer: its packed experts and a plan whose output is
    the FP32 partial sum."""

    def __init__(self, ck: layer.CheckpointExperts, hidden: int, intermediate: int, rank: int, world: int,
                 top_k: int, max_tokens: int, afmt: str):
        if afmt == "nvfp4":
            raise ValueError("NVFP4 activations re-quantise h with a per-row global over the whole "
                             "intermediate dimension; tensor parallelism supports BF16 and MXFP8 activations")
        self.rank, self.world = rank, world
        self.ck = shard_experts(ck, intermediate, rank, world)
        self.packed = layer.PackedLayer(self.ck, hidden, intermediate // world)
        self.plan = layer.Plan(self.packed, top_k, max_tokens, afmt)
        abi.moe_plan_set_option(self.plan.handle, abi.MOE_OPT_OUT_F32, 1)

    def partial(self, x, topk_ids, topk_weights) -> torch.Tensor:
        """This rank's FP32 partial output [T, H]."""
        out = torch.empty(x.shape[0], self.packed.H, dtype=torch.float32, device=x.device)
        b = self.plan.bind(x, topk_ids, topk_weights, out)
        b.run()
        return out

    def forward(self, x, topk_ids, topk_weights, group=None) -> torch.Tensor:
        """The layer's BF16 output: the ranks' partials added in rank order, then rounded."""
        return ordered_all_reduce(self.partial(x, topk_ids, topk_weights), group).to(torch.bfloat16)
