"""Pins of the oracle's MoE forward and routing: float64 brute force on tiny layers,
the method's invariants, and a brute-force sort for the routing reference."""

import math

import numpy as np
import pytest
import torch

from oracle import moe, quant, routing
from block_quantised_moe_gb300 import synth

MAG = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
E4M3_VALS = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().tolist()
F = np.float32


# ------------------------------------------------------------ brute force

def bf_code(packed_row, k):
    byte = int(packed_row[k // 2])
    c = byte & 15 if k % 2 == 0 else byte >> 4
    return (-1.0 if c & 8 else 1.0) * MAG[c & 7]


def bf_weight(codes, scales, g, n, k, wfmt):
    if wfmt == "nvfp4":
        return bf_code(codes[n], k) * E4M3_VALS[int(scales[n][k // 16])] * float(g)
    return bf_code(codes[n], k) * 2.0 ** (int(scales[n][k // 32]) - 127)


def bf_nearest(v, grid):
    """Index of the nearest grid value; ties to the even index."""
    best, bi = None, None
    for i, gv in enumerate(grid):
        d = abs(v - gv)
        if best is None or d < best or (d == best and i % 2 == 0):
            best, bi = d, i
    return bi


POS_E4M3 = [E4M3_VALS[b] for b in range(0x7F)]


def bf_qdq(row, afmt):
    """Scalar-loop quantise-dequantise of one activation row, FP32 steps."""
    row = [float(F(v)) for v in row]
    if afmt == "bf16":
        return row
    out = []
    if afmt == "nvfp4":
        g = F(max(abs(v) for v in row)) / F(2688.0)
        for b in range(0, len(row), 16):
            blk = row[b:b + 16]
            if g == 0:
                out += [0.0] * 16
                continue
            sv = F(F(max(abs(v) for v in blk)) / F(6.0)) / g
            s = POS_E4M3[bf_nearest(min(float(sv), 448.0), POS_E4M3)]
            d = F(s) * g
            for v in blk:
                if d == 0:
                    out.append(0.0)
                    continue
                q = float(F(v) / d)
                m = MAG[bf_nearest(min(abs(q), 6.0), MAG)]
                out.append(math.copysign(m, q) * s * float(g))
        return [float(F(v)) for v in out]
    if afmt == "mxfp8":
        for b in range(0, len(row), 32):
            blk = row[b:b + 32]
            amax = max(abs(v) for v in blk)
            X = -127 if amax == 0 else max(-127, min(127, math.frexp(amax)[1] - 1 - 8))
            for v in blk:
                q = float(F(v) / F(2.0 ** X))
                m = POS_E4M3[bf_nearest(min(abs(q), 448.0), POS_E4M3)]
                out.append(math.copysign(m, q) * 2.0 ** X)
        return out
    raise ValueError(afmt)


def bf_forward(x, ids, w, L, afmt):
    T, K = ids.shape
    E, H, I = L.num_experts, L.hidden, L.intermediate
    y = np.zeros((T, H))
    for t in range(T):
        xh = bf_qdq(x[t], afmt)
        for k in range(K):
            e = int(ids[t, k])
            if not 0 <= e < E:
                continue
            c13, s13, c2, s2 = L.w13_codes[e], L.w13_scales[e], L.w2_codes[e], L.w2_scales[e]
            g13 = L.w13_global[e] if L.w13_global is not None else [None, None]
            g2 = L.w2_global[e] if L.w2_global is not None else None
            h = []
            for i in range(I):
                if L.gated:
                    a = sum(bf_weight(c13, s13, g13[0], i, j, L.wfmt) * xh[j] for j in range(H))
                    u = sum(bf_weight(c13, s13, g13[1], I + i, j, L.wfmt) * xh[j] for j in range(H))
                    h.append(a / (1.0 + math.exp(-a)) * u)
                else:
                    r = sum(bf_weight(c13, s13, g13[0], i, j, L.wfmt) * xh[j] for j in range(H))
                    h.append(max(r, 0.0) ** 2)
            hh = bf_qdq(h, afmt)
            for n in range(H):
                o = sum(bf_weight(c2, s2, g2, n, i, L.wfmt) * hh[i] for i in range(I))
                y[t, n] += float(w[t, k]) * o
    return y


def make_layer(E, H, I, wfmt, act, seed=0):
    gated = act == "silu"
    w13, w2 = [], []
    for e in range(E):
        a, b = synth.make_expert_weights(e, H, I, gated, seed)
        w13.append([m.numpy() for m in a]), w2.append(b.numpy())
    return moe.quantize_layer(w13, w2, wfmt, act)


def make_inputs(T, H, E, K, seed=0):
    x = synth.make_x(T, H, seed).float().numpy()
    ids, w = synth.make_routing(T, E, K, seed)
    return x, ids.numpy(), w.numpy()


MODES = [("nvfp4", "silu", "bf16"), ("nvfp4", "silu", "nvfp4"), ("mxfp4", "relu2", "mxfp8"),
         ("nvfp4", "relu2", "bf16"), ("mxfp4", "silu", "mxfp8"), ("mxfp4", "silu", "bf16")]


@pytest.mark.parametrize("wfmt,act,afmt", MODES)
def test_forward_matches_float64_brute_force(wfmt, act, afmt):
    E, H, I, T, K = 4, 64, 32, 3, 2
    L = make_layer(E, H, I, wfmt, act, seed=1)
    x, ids, w = make_inputs(T, H, E, K, seed=1)
    ids[2, 1] = E  # an out-of-range id is dropped
    y = moe.moe_forward(x, ids, w, L, afmt)
    yb = bf_forward(x, ids, w, L, afmt)
    err = np.linalg.norm(y - yb) / np.linalg.norm(yb)
    assert err < 2e-6, err
    assert np.max(np.abs(y - yb)) <= 1e-5 * (np.abs(yb) + np.sqrt(np.mean(yb ** 2))).max()


def bf_hidden(xh, L, e):
    """Step 3 for one activation row by scalar loops in float64: h [I]."""
    H, I = L.hidden, L.intermediate
    c13, s13 = L.w13_codes[e], L.w13_scales[e]
    g13 = L.w13_global[e] if L.w13_global is not None else [None, None]
    h = []
    for i in range(I):
        if L.gated:
            a = sum(bf_weight(c13, s13, g13[0], i, j, L.wfmt) * xh[j] for j in range(H))
            u = sum(bf_weight(c13, s13, g13[1], I + i, j, L.wfmt) * xh[j] for j in range(H))
            h.append(a / (1.0 + math.exp(-a)) * u)
        else:
            r = sum(bf_weight(c13, s13, g13[0], i, j, L.wfmt) * xh[j] for j in range(H))
            h.append(max(r, 0.0) ** 2)
    return np.array(h)


@pytest.mark.parametrize("wfmt,act,afmt", MODES)
def test_expert_hidden_matches_float64_brute_force(wfmt, act, afmt):
    # step 3 on its own (the GPU's GEMM1 output is compared with this function)
    E, H, I, T = 3, 64, 32, 3
    L = make_layer(E, H, I, wfmt, act, seed=4)
    x, _, _ = make_inputs(T, H, E, 1, seed=4)
    xh = quant.qdq_rows(x, afmt)
    for e in range(E):
        h = moe.expert_hidden(L, e, xh)
        hb = np.stack([bf_hidden(bf_qdq(x[t], afmt), L, e) for t in range(T)])
        assert h.shape == (T, I) and h.dtype == np.float32
        assert np.linalg.norm(h - hb) / np.linalg.norm(hb) < 2e-6
        assert np.max(np.abs(h - hb)) <= 1e-5 * (np.abs(hb) + np.sqrt(np.mean(hb ** 2))).max()


# ------------------------------------------------------------- invariants

@pytest.fixture(scope="module", params=MODES[:3], ids=lambda m: "-".join(m))
def case(request):
    wfmt, act, afmt = request.param
    E, H, I, T, K = 8, 128, 64, 16, 4
    L = make_layer(E, H, I, wfmt, act, seed=2)
    x, ids, w = make_inputs(T, H, E, K, seed=2)
    return L, x, ids, w, afmt


def test_top1_weight1_equals_single_expert_ffn(case):
    L, x, ids, w, afmt = case
    ids1 = ids[:, :1].copy()
    y = moe.moe_forward(x, ids1, np.ones_like(w[:, :1]), L, afmt)
    for t in range(x.shape[0]):
        e = int(ids1[t, 0])
        mats, w2 = L.dequant_expert(e)
        xh = quant.qdq_rows(x[t:t + 1], afmt).astype(np.float64)
        if L.gated:
            a, b = xh @ mats[0].T.astype(np.float64), xh @ mats[1].T.astype(np.float64)
            h = a / (1 + np.exp(-a)) * b
        else:
            h = np.maximum(xh @ mats[0].T.astype(np.float64), 0) ** 2
        hh = quant.qdq_rows(h.astype(np.float32), afmt).astype(np.float64)
        want = hh @ w2.T.astype(np.float64)
        assert np.linalg.norm(y[t] - want) <= 1e-5 * np.linalg.norm(want)


def test_zero_weights_give_zero(case):
    L, x, ids, w, afmt = case
    y = moe.moe_forward(x, ids, np.zeros_like(w), L, afmt)
    assert np.all(y == 0)


def test_linear_in_topk_weights(case):
    # Also pins where topk_weights act: on the expert output, after h is re-quantised.
    L, x, ids, w, afmt = case
    alpha = np.float32(0.37)
    y1 = moe.moe_forward(x, ids, w, L, afmt)
    y2 = moe.moe_forward(x, ids, w * alpha, L, afmt)
    assert np.linalg.norm(y2 - alpha * y1) <= 1e-6 * np.linalg.norm(y1)


def test_permuting_topk_slots(case):
    L, x, ids, w, afmt = case
    perm = np.array([2, 0, 3, 1])
    y1 = moe.moe_forward(x, ids, w, L, afmt)
    y2 = moe.moe_forward(x, ids[:, perm], w[:, perm], L, afmt)
    assert np.linalg.norm(y2 - y1) <= 1e-6 * np.linalg.norm(y1)


def test_tokens_are_independent(case):
    # Activation quantisation is per token row: other rows cannot change a token's output.
    L, x, ids, w, afmt = case
    y1 = moe.moe_forward(x, ids, w, L, afmt)
    x2 = x.copy()
    x2[1:] *= np.float32(1000.0)
    y2 = moe.moe_forward(x2, ids, w, L, afmt)
    assert np.array_equal(y1[0], y2[0])


def test_dropped_ids_contribute_nothing(case):
    L, x, ids, w, afmt = case
    E = L.num_experts
    ids2, w0 = ids.copy(), w.copy()
    ids2[0, 1], ids2[3, 0] = -1, E + 5
    w0[0, 1], w0[3, 0] = 0.0, 0.0
    assert np.array_equal(moe.moe_forward(x, ids2, w, L, afmt), moe.moe_forward(x, ids, w0, L, afmt))


# ---------------------------------------------------------------- routing

@pytest.mark.parametrize("T,K,E,pad", [(16, 2, 8, 16), (64, 8, 128, 16), (5, 3, 4, 1), (33, 4, 16, 128), (0, 4, 8, 16)])
def test_routing_matches_brute_force_sort(T, K, E, pad):
    rng = np.random.default_rng(T * 7 + E)
    ids = rng.integers(-1, E + 1, (T, K)).astype(np.int32)  # includes out-of-range ids
    r = routing.route(ids, E, pad)
    flat = ids.reshape(-1).tolist()
    pairs = sorted((e, p) for p, e in enumerate(flat) if 0 <= e < E)
    off, sorted_pair, pos = [0], [], {}
    for e in range(E):
        ps = [p for (ee, p) in pairs if ee == e]
        for p in ps:
            pos[p] = len(sorted_pair)
            sorted_pair.append(p)
        n = len(ps)
        sorted_pair += [-1] * ((-n) % pad)
        off.append(len(sorted_pair))
        assert r["counts"][e] == n
    assert r["offsets"].tolist() == off
    assert r["sorted_pair"].tolist() == sorted_pair
    assert r["pair_pos"].tolist() == [pos.get(p, -1) for p in range(len(flat))]
    assert r["dropped"] == sum(1 for e in flat if not 0 <= e < E)
