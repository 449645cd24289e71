"""Fused routed-expert MoE FFN forward in FP32 (oracle).

Test infrastructure: see the package docstring for who may import this.

The op is ``moe.fused_moe``: a routed-expert FFN over FP4 block-quantised
expert weights with gated SiLU or non-gated ReLU^2 (b12x project page, "What's
in here"; vLLM docs "b12x Linear and MoE Backends", "ModelOpt block codecs":
routed experts use bias-free SiLU or non-gated ReLU^2).  Its inputs are the
activations, the prepared experts and the router's ``topk_ids`` /
``topk_weights`` (b12x project page, "Using it").  Definition, in FP32:

1. Decode weights: W^ = E2M1(code) * E4M3(s_b) * g_m (NVFP4, one global per
   expert and matrix) or E2M1(code) * 2^(E8M0(s_b)-127) (MXFP4).
2. Activations: x^ = x (BF16 activations, "W4A16"), or dequant(quant_row(x))
   for NVFP4 (W4A4) / MXFP8 (W4A8) activations.
3. For each pair (t, k) with expert e = topk_ids[t, k]:
   gated:   h = SiLU(W^g_e x^_t) * (W^u_e x^_t),  SiLU(a) = a * 1/(1+exp(-a));
   ReLU^2:  h = max(W^1_e x^_t, 0)^2.
4. h^ = h (W4A16), or dequant(quant_row(h)) with the activation format.
5. y_t = sum_k w_tk * (W^2_e h^), summed in slot order k = 0..K-1.

W13 of a gated expert stacks the gate rows [0, I) above the up rows [I, 2I).
Pairs whose id lies outside [0, E) contribute nothing.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import quant


@dataclass
class QuantLayer:
    """Quantised expert weights in the checkpoint layout.

    wfmt: "nvfp4" | "mxfp4";  act: "silu" (gated) | "relu2".
    w13_codes  [E, N13, H/2]  uint8, two E2M1 codes per byte (N13 = 2I gated, I otherwise)
    w13_scales [E, N13, H/bs] uint8 (E4M3 for nvfp4, bs=16; E8M0 for mxfp4, bs=32)
    w13_global [E, 2] (gate, up) or [E, 1] float32 for nvfp4; None for mxfp4
    w2_codes   [E, H, I/2], w2_scales [E, H, I/bs], w2_global [E] or None
    """

    wfmt: str
    act: str
    w13_codes: np.ndarray
    w13_scales: np.ndarray
    w13_global: np.ndarray | None
    w2_codes: np.ndarray
    w2_scales: np.ndarray
    w2_global: np.ndarray | None

    @property
    def num_experts(self) -> int:
        return self.w13_codes.shape[0]

    @property
    def hidden(self) -> int:
        return self.w2_codes.shape[1]

    @property
    def intermediate(self) -> int:
        return self.w2_codes.shape[2] * 2

    @property
    def gated(self) -> bool:
        return self.act == "silu"

    def dequant_expert(self, e: int):
        """(list of W13 matrices [gate, up] or [w1], W2) as dense float32."""
        I = self.intermediate
        g13 = self.w13_global[e] if self.w13_global is not None else (None, None)
        if self.gated:
            mats = [
                quant.dequant_weight_matrix(self.w13_codes[e, :I], self.w13_scales[e, :I], g13[0], self.wfmt),
                quant.dequant_weight_matrix(self.w13_codes[e, I:], self.w13_scales[e, I:], g13[1], self.wfmt),
            ]
        else:
            mats = [quant.dequant_weight_matrix(self.w13_codes[e], self.w13_scales[e], g13[0], self.wfmt)]
        g2 = self.w2_global[e] if self.w2_global is not None else None
        w2 = quant.dequant_weight_matrix(self.w2_codes[e], self.w2_scales[e], g2, self.wfmt)
        return mats, w2


def quantize_layer(w13: list, w2: list, wfmt: str, act: str) -> QuantLayer:
    """Checkpoint-style quantisation of FP32 expert weights.

    ``w13[e]`` is (gate [I,H], up [I,H]) for gated SiLU or (w1 [I,H],) for ReLU^2;
    ``w2[e]`` is down [H, I].  Each matrix gets its own NVFP4 global scale.
    """
    c13, s13, g13, c2, s2, g2 = [], [], [], [], [], []
    for e in range(len(w13)):
        cs, ss, gs = [], [], []
        for m in w13[e]:
            c, s, g = quant.quantize_weight_matrix(m, wfmt)
            cs.append(c), ss.append(s), gs.append(g)
        c13.append(np.concatenate(cs, 0)), s13.append(np.concatenate(ss, 0)), g13.append(gs)
        c, s, g = quant.quantize_weight_matrix(w2[e], wfmt)
        c2.append(c), s2.append(s), g2.append(g)
    nv = wfmt == "nvfp4"
    return QuantLayer(
        wfmt=wfmt, act=act,
        w13_codes=np.stack(c13), w13_scales=np.stack(s13),
        w13_global=np.array(g13, dtype=np.float32) if nv else None,
        w2_codes=np.stack(c2), w2_scales=np.stack(s2),
        w2_global=np.array(g2, dtype=np.float32) if nv else None,
    )


def silu(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a, dtype=np.float32)
    with np.errstate(over="ignore"):
        return a * (np.float32(1.0) / (np.float32(1.0) + np.exp(-a)))


def expert_hidden(layer: QuantLayer, e: int, xh: np.ndarray, dequant=None) -> np.ndarray:
    """Step 3: h [n, I] float32 of expert ``e`` for activation rows ``xh`` [n, H]."""
    mats = (dequant if dequant is not None else layer.dequant_expert(e))[0]
    if layer.gated:
        a = xh @ mats[0].T
        b = xh @ mats[1].T
        return (silu(a) * b).astype(np.float32)
    r = np.maximum(xh @ mats[0].T, np.float32(0.0))
    return (r * r).astype(np.float32)


def expert_ffn(layer: QuantLayer, e: int, xh: np.ndarray, afmt: str, dequant=None) -> np.ndarray:
    """Steps 3-4 and W^2_e h^ for rows ``xh`` [n, H] routed to expert ``e``."""
    dq = dequant if dequant is not None else layer.dequant_expert(e)
    w2 = dq[1]
    h = expert_hidden(layer, e, xh, dq)
    hh = quant.qdq_rows(h, afmt)
    return (hh @ w2.T).astype(np.float32)


def moe_forward(x: np.ndarray, topk_ids: np.ndarray, topk_weights: np.ndarray,
                layer: QuantLayer, afmt: str) -> np.ndarray:
    """y [T, H] float32 for activations ``x`` [T, H] (BF16 values as float32)."""
    x = np.asarray(x, dtype=np.float32)
    ids = np.asarray(topk_ids, dtype=np.int64)
    w = np.asarray(topk_weights, dtype=np.float32)
    T, K = ids.shape
    H = x.shape[1]
    E = layer.num_experts
    xh = quant.qdq_rows(x, afmt)
    o = np.zeros((T, K, H), dtype=np.float32)
    for e in np.unique(ids[(ids >= 0) & (ids < E)]):
        t_idx, k_idx = np.nonzero(ids == e)
        o[t_idx, k_idx] = expert_ffn(layer, int(e), xh[t_idx], afmt)
    y = np.zeros((T, H), dtype=np.float32)
    for k in range(K):
        y = y + w[:, k:k + 1] * o[:, k]
    return y
