"""Expert parallelism: each rank holds a contiguous range of the experts.

`moe.ep_moe` of the b12x project page ("What's in here") shards the experts
across GPUs.  Here every rank sees every token (the activations and the
router's choices are replicated) and runs the whole layer on its own experts:
the (token, slot) pairs routed to another rank's experts get the id -1, which
the routing drops (recorded in the status word, not an error), so a rank's
GEMMs cover only its experts' pairs.  Its output, with an FP32 output
(MOE_OPT_OUT_F32), is the sum over those pairs; the ranks' partials are added
in rank order (tp.ordered_all_reduce), which gives every rank the same bytes.

Unlike the intermediate-dimension split, nothing a rank computes depends on
another rank: x is quantised per token row and h per (token, slot) row, and
each pair lives on one rank, so every activation format is supported.  Because
the ranges are contiguous and ascending, the rank-ordered sum adds the
experts' contributions in the unsharded layer's expert order, grouped by rank;
only the grouping of the FP32 additions differs.

This is the replicated-activation form of expert parallelism (no token
dispatch between ranks); the slicing and the reduction are host code on any
torch.distributed backend, the per-rank forward is the library's.
"""

from __future__ import annotations

import numpy as np
import torch

from . import abi, layer
from .tp import ordered_all_reduce

_EXPERT_KEYS = ("w13_codes", "w13_scales", "w13_global", "w2_codes", "w2_scales", "w2_global")


def expert_bounds(num_experts: int, rank: int, world: int) -> tuple[int, int]:
    """[e0, e1) of this rank's experts (equal contiguous ranges)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of {world}")
    if num_experts % world != 0:
        raise ValueError(f"{num_experts} experts do not split into {world} equal ranges")
    n = num_experts // world
    return rank * n, (rank + 1) * n


def shard_expert_arrays(w: dict, num_experts: int, rank: int, world: int) -> dict:
    """This rank's experts of checkpoint arrays (numpy or torch; every array's
    first axis is the expert; None entries, e.g. MXFP4's absent global scales,
    stay None)."""
    e0, e1 = expert_bounds(num_experts, rank, world)
    out = dict(w)
    for k in _EXPERT_KEYS:
        a = w.get(k)
        if a is None:
            continue
        if a.shape[0] != num_experts:
            raise ValueError(f"{k}: first axis {a.shape[0]} is not the {num_experts} experts")
        s = a[e0:e1]
        out[k] = s.contiguous() if isinstance(s, torch.Tensor) else np.ascontiguousarray(s)
    return out


def local_ids(topk_ids, e0: int, e1: int):
    """Router ids in this rank's numbering: id - e0 for its experts, -1 for the
    others (dropped by the routing).  numpy or torch, int32 out."""
    if isinstance(topk_ids, torch.Tensor):
        ids = topk_ids.to(torch.int32)
        mine = (ids >= e0) & (ids < e1)
        return torch.where(mine, ids - e0, torch.full_like(ids, -1)).contiguous()
    ids = np.asarray(topk_ids).astype(np.int32)
    return np.where((ids >= e0) & (ids < e1), ids - e0, -1).astype(np.int32)


def shard_experts(ck: layer.CheckpointExperts, rank: int, world: int) -> layer.CheckpointExperts:
    """A rank's experts on the device."""
    d = shard_expert_arrays({k: getattr(ck, k) for k in _EXPERT_KEYS}, ck.num_experts, rank, world)
    return layer.CheckpointExperts(wfmt=ck.wfmt, act=ck.act, **{k: d[k] for k in _EXPERT_KEYS})


class EPLayer:
    """One rank's experts of a layer: its packed experts and a plan whose output
    is the FP32 partial sum over the pairs routed to them."""

    def __init__(self, ck: layer.CheckpointExperts, hidden: int, intermediate: int, rank: int, world: int,
                 top_k: int, max_tokens: int, afmt: str):
        self.rank, self.world = rank, world
        self.e0, self.e1 = expert_bounds(ck.num_experts, rank, world)
        self.ck = shard_experts(ck, rank, world)
        self.packed = layer.PackedLayer(self.ck, hidden, intermediate)
        self.plan = layer.Plan(self.packed, top_k, max_tokens, afmt)
        abi.moe_plan_set_option(self.plan.handle, abi.MOE_OPT_OUT_F32, 1)

    def partial(self, x, topk_ids, topk_weights) -> torch.Tensor:
        """This rank's FP32 partial output [T, H] (zero rows for tokens with no
        pair on this rank)."""
        out = torch.empty(x.shape[0], self.packed.H, dtype=torch.float32, device=x.device)
        ids = local_ids(topk_ids, self.e0, self.e1)
        b = self.plan.bind(x, ids, topk_weights, out)
        b.run()
        return out

    def forward(self, x, topk_ids, topk_weights, group=None) -> torch.Tensor:
        """The layer's BF16 output: the ranks' partials added in rank order, then rounded."""
        return ordered_all_reduce(self.partial(x, topk_ids, topk_weights), group).to(torch.bfloat16)
