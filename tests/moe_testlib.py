"""Shared plumbing for the GPU parity tests: build both sides from the same seeded
draws and compare with the tolerances of the method.

The CUDA side quantises its FP32 experts with libmoe's quantiser; the oracle
side quantises the same FP32 draws with the oracle quantiser, and the two code
sets are asserted bit-identical before any forward is compared.  No input or
expected value of the oracle comes from the CUDA path.
"""

from __future__ import annotations

import numpy as np
import torch

from block_quantised_moe_gb300 import synth

# Tolerances of the fused MoE output against the FP32 oracle (BF16 output,
# FP32 accumulation in a different order): normwise and per element.
NORM_TOL = 1e-2
ELEM_TOL = 3e-2


class RefArray(np.ndarray):
    """Oracle output carrying ``env``: the per-element envelope of equally valid
    re-quantisation decisions (see requant_envelope); zero for BF16 activations."""

    env = None


def check_close(y: np.ndarray, y_ref: np.ndarray, what: str = "", env=None) -> dict:
    env = getattr(y_ref, "env", None) if env is None else env
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    den = np.linalg.norm(y_ref)
    norm_err = np.linalg.norm(y - y_ref) / den if den > 0 else np.linalg.norm(y)
    rms = np.sqrt(np.mean(y_ref ** 2)) if y_ref.size else 0.0
    diff = np.abs(y - y_ref)
    if env is not None:
        diff = np.maximum(diff - np.asarray(env, dtype=np.float64), 0.0)
    elem = diff / (np.abs(y_ref) + rms + 1e-30)
    worst = float(elem.max()) if elem.size else 0.0
    assert norm_err <= NORM_TOL, f"{what}: normwise error {norm_err:.3e} > {NORM_TOL}"
    assert worst <= ELEM_TOL, f"{what}: element error {worst:.3e} > {ELEM_TOL}"
    return dict(norm=float(norm_err), elem=worst)


_ORACLE_EXPERT_CACHE: dict = {}
# experts with at least this many weight elements are quantised in the oracle pool
_POOL_MIN_ELEMS = 4 << 20


def oracle_expert(E, H, I, wfmt, act, e, seed=0):
    """Oracle-quantised expert e: (codes13, scales13, g13, codes2, scales2, g2) as numpy."""
    key = (E, H, I, wfmt, act, e, seed)
    if key not in _ORACLE_EXPERT_CACHE:
        prefetch_oracle_experts(E, H, I, wfmt, act, [e], seed)
    return _ORACLE_EXPERT_CACHE[key]


def prefetch_oracle_experts(E, H, I, wfmt, act, experts, seed=0):
    """Quantise the listed experts with the oracle quantiser (in the worker pool
    for large experts), from the same seeded FP32 draws as the GPU layer."""
    import oracle_pool
    gated = act == "silu"
    missing = [int(e) for e in experts if (E, H, I, wfmt, act, int(e), seed) not in _ORACLE_EXPERT_CACHE]
    if not missing:
        return
    if (3 if gated else 2) * H * I < _POOL_MIN_ELEMS or len(missing) == 1:
        for e in missing:
            w13, w2 = synth.make_expert_weights(e, H, I, gated, seed, device="cuda")
            _ORACLE_EXPERT_CACHE[(E, H, I, wfmt, act, e, seed)] = oracle_pool.quantize_expert(
                [m.cpu().numpy() for m in w13], w2.cpu().numpy(), wfmt)
        return
    ex = oracle_pool.pool()
    inflight = {}
    todo = list(missing)
    while todo or inflight:
        while todo and len(inflight) < 2 * oracle_pool.workers():
            e = todo.pop(0)
            w13, w2 = synth.make_expert_weights(e, H, I, gated, seed, device="cuda")
            fut = ex.submit(oracle_pool.quantize_expert, [m.cpu().numpy() for m in w13], w2.cpu().numpy(), wfmt)
            inflight[fut] = e
        import concurrent.futures as cf
        done, _ = cf.wait(list(inflight), return_when=cf.FIRST_COMPLETED)
        for fut in done:
            e = inflight.pop(fut)
            _ORACLE_EXPERT_CACHE[(E, H, I, wfmt, act, e, seed)] = fut.result()


def oracle_layer_for(ck, H, I, experts, seed=0, check_codes=True):
    """Oracle QuantLayer over the listed experts (compact index space), after
    checking that libmoe's quantiser produced the same bytes for them."""
    from oracle import moe
    E = ck.num_experts
    wfmt, act = ck.wfmt, ck.act
    prefetch_oracle_experts(E, H, I, wfmt, act, experts, seed)
    parts = [oracle_expert(E, H, I, wfmt, act, int(e), seed) for e in experts]
    if check_codes:
        for e, (c13, s13, g13, c2, s2, g2) in zip(experts, parts):
            e = int(e)
            assert np.array_equal(ck.w13_codes[e].cpu().numpy(), c13), f"W13 codes of expert {e}"
            assert np.array_equal(ck.w13_scales[e].cpu().numpy(), s13), f"W13 scales of expert {e}"
            assert np.array_equal(ck.w2_codes[e].cpu().numpy(), c2), f"W2 codes of expert {e}"
            assert np.array_equal(ck.w2_scales[e].cpu().numpy(), s2), f"W2 scales of expert {e}"
            if wfmt == "nvfp4":
                assert np.array_equal(ck.w13_global[e].cpu().numpy(), np.array(g13, np.float32))
                assert ck.w2_global[e].item() == np.float32(g2)
    nv = wfmt == "nvfp4"
    return moe.QuantLayer(
        wfmt=wfmt, act=act,
        w13_codes=np.stack([p[0] for p in parts]), w13_scales=np.stack([p[1] for p in parts]),
        w13_global=np.array([p[2] for p in parts], np.float32) if nv else None,
        w2_codes=np.stack([p[3] for p in parts]), w2_scales=np.stack([p[4] for p in parts]),
        w2_global=np.array([p[5] for p in parts], np.float32) if nv else None)


def oracle_forward(ck, H, I, x, ids, w, afmt, tokens=None, seed=0):
    """Oracle y for the given token rows (all by default), in FP32, as a RefArray
    whose ``env`` is the re-quantisation envelope.  Large layers run in the
    worker pool, a chunk of tokens per job (tokens are independent in the
    oracle's definition)."""
    from oracle import moe
    import oracle_pool
    import requant_envelope
    x = x.float().cpu().numpy()
    ids = ids.cpu().numpy()
    w = w.cpu().numpy()
    if tokens is not None:
        x, ids, w = x[tokens], ids[tokens], w[tokens]
    E = ck.num_experts
    valid = (ids >= 0) & (ids < E)
    used = np.unique(ids[valid])
    prefetch_oracle_experts(E, H, I, ck.wfmt, ck.act, used, seed)
    L = oracle_layer_for(ck, H, I, used, seed)
    remap = np.full(E, -1, np.int64)
    remap[used] = np.arange(len(used))
    ids_c = np.where(valid, remap[np.clip(ids, 0, E - 1)], -1)
    T = x.shape[0]
    big = H * I >= _POOL_MIN_ELEMS // 2 and T > 1
    if not big:
        y, env = requant_envelope.forward_with_envelope(x, ids_c, w, L, afmt)
    else:
        n = min(T, oracle_pool.workers())
        chunks = np.array_split(np.arange(T), n)
        futs = []
        for ch in chunks:
            sub = ids_c[ch]
            u = np.unique(sub[sub >= 0])
            rm = np.full(len(used), -1, np.int64)
            rm[u] = np.arange(len(u))
            sub_c = np.where(sub >= 0, rm[np.clip(sub, 0, None)], -1)
            Lc = moe.QuantLayer(
                wfmt=L.wfmt, act=L.act, w13_codes=L.w13_codes[u], w13_scales=L.w13_scales[u],
                w13_global=None if L.w13_global is None else L.w13_global[u],
                w2_codes=L.w2_codes[u], w2_scales=L.w2_scales[u],
                w2_global=None if L.w2_global is None else L.w2_global[u])
            futs.append(oracle_pool.pool().submit(oracle_pool.forward_tokens, x[ch], sub_c, w[ch], Lc, afmt))
        res = [f.result() for f in futs]
        y = np.concatenate([r[0] for r in res], axis=0)
        env = np.concatenate([r[1] for r in res], axis=0)
    out = np.asarray(y, dtype=np.float32).view(RefArray)
    out.env = env
    return out


def make_inputs(cfg, T, seed=0, device="cuda"):
    x = synth.make_x(T, cfg["H"], seed, device="cpu").to(device)
    ids, w = synth.make_routing(T, cfg["E"], cfg["K"], seed, zipf=cfg["zipf"])
    return x, ids.to(device), w.to(device)


def sample_tokens(T, n, seed=0):
    if T <= n:
        return np.arange(T)
    rng = np.random.default_rng(seed + T)
    return np.sort(rng.choice(T, size=n, replace=False))
