"""How far the layer output may legitimately move when h is re-quantised
(test infrastructure, built from the oracle's own quantiser pieces).

With NVFP4 or MXFP8 activations the hidden vector h of every (token, slot)
pair is re-quantised before the second contraction (the reading that both
operands of the block-scaled MMAs are block-quantised).  Each code and block
scale of that re-quantisation is a rounding decision on a value both sides
compute in FP32, but with different summation orders (the GPU's tensor-core
accumulation against numpy's).  Where h lies within a rounding error of a
decision boundary, either code is a correct result of the definition, and the
two choices differ by one code step times the block scale.  Such an element is
"fragile"; the envelope of an output element is the largest change that any
combination of fragile decisions can make to it:

    env[t, n] = sum_k |w_tk| * sum_i |W2_e[n, i]| * dh[t, k, i]

with dh the code step of every fragile element of h (0 elsewhere).  The layer
tests allow |y - y_ref| up to the per-element tolerance plus this envelope;
the normwise bound is unchanged.  Away from boundaries the envelope is zero.

A decision is counted as fragile when moving its input by EPS relative (plus
EPS times the row's rms for values near zero, where summation errors are
absolute) changes it.  Two FP32 summation orders leave a relative difference
of about 1e-7 to 1e-6 in h, so EPS = 1e-5 is a margin of ten or more.  A
fragile code contributes its exact code step; a fragile block scale (NVFP4
E4M3, or the MXFP8 shared exponent) contributes the exact change of every
element of its block when re-quantised with the neighbouring scale.
"""

from __future__ import annotations

import numpy as np

EPS = 1e-5


def flip_delta(h: np.ndarray, afmt: str, eps: float = EPS) -> np.ndarray:
    """|change of h^| per element of h [n, I] if its fragile decisions flip; 0 elsewhere."""
    from oracle import codecs, quant
    h = np.asarray(h, dtype=np.float32)
    n, I = h.shape
    if afmt == "bf16" or n == 0:
        return np.zeros_like(h)
    rms = np.sqrt(np.mean(h.astype(np.float64) ** 2, axis=1)).astype(np.float32).reshape(n, 1, 1)
    f32 = lambda a: np.asarray(a, dtype=np.float32)  # noqa: E731
    if afmt == "nvfp4":
        bs = quant.NVFP4_BLOCK
        amax = np.max(np.abs(h), axis=1)
        g = quant.nvfp4_global(amax).reshape(n, 1, 1)
        blk = h.reshape(n, I // bs, bs)
        amax_b = np.max(np.abs(blk), axis=2, keepdims=True)
        with np.errstate(divide="ignore", invalid="ignore"):
            sv = f32(np.where(g > 0, (amax_b / quant.E2M1_MAX) / g, 0))

        def qdq(scale_codes):
            d = f32(codecs.e4m3_decode(scale_codes) * g)
            with np.errstate(divide="ignore", invalid="ignore"):
                v = f32(np.where(d > 0, blk / d, 0))
            return d, v, f32(codecs.e2m1_decode(codecs.e2m1_encode(v)) * d)

        s0 = codecs.e4m3_encode(sv)
        d, v, hh = qdq(s0)
        # codes: the exact step between the two roundings of a fragile value
        with np.errstate(divide="ignore", invalid="ignore"):
            slack = f32(eps * (2 * np.abs(v) + np.where(d > 0, rms / d, 0)))
        lo = codecs.e2m1_decode(codecs.e2m1_encode(f32(v - slack)))
        hi = codecs.e2m1_decode(codecs.e2m1_encode(f32(v + slack)))
        dh = np.abs(hi - lo) * d
        # block scales: amax_b and the row global each move by eps
        s_lo = codecs.e4m3_encode(f32(sv * (1 - 2 * eps)))
        s_hi = codecs.e4m3_encode(f32(sv * (1 + 2 * eps)))
        for alt in (s_lo, s_hi):
            frag = alt != s0
            if frag.any():
                _, _, ha = qdq(alt)
                dh = np.where(frag, np.maximum(dh, np.abs(ha - hh)), dh)
        return np.where(d > 0, dh, 0).reshape(n, I).astype(np.float32)
    if afmt == "mxfp8":
        bs = quant.MX_BLOCK
        blk = h.reshape(n, I // bs, bs)
        amax_b = np.max(np.abs(blk), axis=2, keepdims=True)
        nz = amax_b > 0
        safe = f32(np.where(nz, amax_b, 1))
        X = np.clip(codecs.floor_log2(safe) - quant.MX_EMAX["e4m3"], -127, 127)

        def qdq(Xs):
            p2 = f32(np.ldexp(np.float32(1.0), Xs))
            v = f32(blk / p2)
            return p2, v, f32(codecs.e4m3_decode(codecs.e4m3_encode(v)) * p2)

        p2, v, hh = qdq(X)
        slack = f32(eps * (2 * np.abs(v) + rms / p2))
        lo = codecs.e4m3_decode(codecs.e4m3_encode(f32(np.clip(v - slack, -448, 448))))
        hi = codecs.e4m3_decode(codecs.e4m3_encode(f32(np.clip(v + slack, -448, 448))))
        dh = np.abs(hi - lo) * p2
        for direction in (-1, 1):
            Xa = np.clip(codecs.floor_log2(f32(safe * (1 + direction * eps))) - quant.MX_EMAX["e4m3"], -127, 127)
            frag = nz & (Xa != X)
            if frag.any():
                _, _, ha = qdq(Xa)
                dh = np.where(frag, np.maximum(dh, np.abs(ha - hh)), dh)
        return np.where(nz, dh, 0).reshape(n, I).astype(np.float32)
    raise ValueError(afmt)


def forward_with_envelope(x, ids_c, w, layer, afmt):
    """(oracle y [T, H], envelope [T, H]) for activations x [T, H]."""
    from oracle import moe, quant
    y = moe.moe_forward(x, ids_c, w, layer, afmt)
    T, K = ids_c.shape
    env = np.zeros_like(y, dtype=np.float64)
    if afmt == "bf16":
        return y, env
    xh = quant.qdq_rows(np.asarray(x, np.float32), afmt)
    E = layer.num_experts
    for e in np.unique(ids_c[(ids_c >= 0) & (ids_c < E)]):
        t_idx, k_idx = np.nonzero(ids_c == e)
        dq = layer.dequant_expert(int(e))
        h = moe.expert_hidden(layer, int(e), xh[t_idx], dq)
        dh = flip_delta(h, afmt)
        rows = np.nonzero(dh.any(axis=1))[0]
        if rows.size:
            wt = np.abs(w[t_idx[rows], k_idx[rows]]).astype(np.float64)[:, None]
            contrib = wt * (dh[rows].astype(np.float64) @ np.abs(dq[1]).T.astype(np.float64))
            np.add.at(env, t_idx[rows], contrib)
    return y, env
