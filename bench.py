#!/usr/bin/env python
"""MoE-layer throughput of libmoe on GB300, one JSON line on rank 0.

Headline workload: the prefill layer E=256 experts, hidden 7168, intermediate
2048, top-8, T=8192 tokens, NVFP4 weights with BF16 activations (W4A16) and
gated SiLU -- the largest single-GPU configuration of this op.  A step is one
full forward of the layer (routing, GEMM1 + SiLU, GEMM2 x topk weight,
combine) through the C ABI over one batch of seeded synthetic input.

``value`` is tokens/s with inputs resident in HBM, timed with CUDA events on
the launching stream over replays of CUDA graphs of the forward; ``e2e`` is the
same through ``moe_run_host`` with pinned host buffers (H2D of x / ids /
weights and D2H of the output inside the timed loop).  ``roofline`` is for the
dominant kernel, from per-stage CUDA events recorded by ``moe_run_timed``
inside the timed region.  ``cpu_baseline`` times the CPU oracle on a bounded
sample.  ``rows`` carries the other workloads (W4A4 prefill, the decode
layers, MXFP4 x MXFP8), each with its own step time and roofline.  Steps rotate
over R layer replicas and routing draws whose touched bytes together exceed L2
several times over, so every step streams its experts from HBM.
``--impl reference`` times only the oracle (the reference arm).  Multi-GPU
runs (torchrun) are independent replicas: one layer per rank, no collective on
the data path, weak scaling.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = ("prefill_w4a16_e256_h7168_i2048_k8", 8192)
# the other workloads of the op, reported under "rows"
ROWS = [("prefill_w4a4_e256_h7168_i2048_k8", 8192)] + \
    [("decode_e128_h2048_i768_k8", t) for t in (1, 4, 16, 64)] + \
    [("decode_e128_h2048_i768_k8", t, "single-launch") for t in (1, 64)] + \
    [("decode_zipf_e256_h7168_i2048_k8", t) for t in (1, 8, 32, 128)] + \
    [("mxfp4_mxfp8_relu2_e128_h4096_i1024_k4", t) for t in (1, 64, 4096)] + \
    [("mxfp4_mxfp8_relu2_e128_h4096_i1024_k4", 1, "single-launch")]
L2_BYTES = 126.5e6
# committed ncu summaries (profiles/) per (workload, T), else per workload
PROFILES = {
    "prefill_w4a16_e256_h7168_i2048_k8": "profiles/k_grouped_tc2_prefill_e32_h7168_t2048.md",
    "prefill_w4a4_e256_h7168_i2048_k8": "profiles/k_grouped_fp4_prefill_e32_h7168_t2048.md",
    "decode_e128_h2048_i768_k8": "profiles/k_grouped_mma_decode_e128_h2048_t64.md",
    ("decode_e128_h2048_i768_k8", 1): "profiles/k_grouped_mma_decode_e128_h2048_t1.md",
    ("decode_zipf_e256_h7168_i2048_k8", 1): "profiles/k_grouped_mma_zipf_e256_h7168_t1.md",
    ("decode_zipf_e256_h7168_i2048_k8", 128): "profiles/k_grouped_mma_zipf_e256_h7168_t128.md",
    ("mxfp4_mxfp8_relu2_e128_h4096_i1024_k4", 1): "profiles/k_grouped_mma_mxfp4_mxfp8_e128_h4096_t1.md",
    ("mxfp4_mxfp8_relu2_e128_h4096_i1024_k4", 64): "profiles/k_grouped_mma_mxfp4_mxfp8_e128_h4096_t64.md",
    ("mxfp4_mxfp8_relu2_e128_h4096_i1024_k4", 4096): "profiles/k_grouped_tc2_mxfp4_mxfp8_e128_h4096_t4096.md",
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=None, help="run this workload alone as the headline")
    ap.add_argument("--tokens", type=int, default=None)
    ap.add_argument("--rows", default=None,
                    help="'all' (default with the headline), 'none', or workload:T pairs, comma separated")
    ap.add_argument("--row-steps", type=int, default=None, help="timed steps per extra row (default: --steps)")
    ap.add_argument("--max-replicas", type=int, default=16)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--experts", type=int, default=None,
                    help="override the workload's expert count (small captures for ncu)")
    return ap.parse_args()


# ------------------------------------------------------------- distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    """The largest of the ranks' values (the slowest rank's time), on every rank."""
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, seconds_max):
    """Whole-job units per second: every rank's units over the slowest rank's time
    (independent replicas, so the work grows with the number of ranks)."""
    return world * units_per_rank / seconds_max


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """SM clock and clock-event reasons sampled through NVML (read-only) while running."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting"}

    def __init__(self, interval=0.002):
        self.samples, self.reasons, self.max_mhz = [], 0, None
        self.interval, self._stop = interval, threading.Event()
        self.nvml = self.handle = None
        try:
            nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if nvml.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            p = torch.cuda.get_device_properties(torch.cuda.current_device())
            bus = getattr(p, "pci_bus_id", None)
            ok = -1
            if bus is not None:
                busid = f"{getattr(p, 'pci_domain_id', 0):08x}:{bus:02x}:{getattr(p, 'pci_device_id', 0):02x}.0"
                ok = nvml.nvmlDeviceGetHandleByPciBusId_v2(busid.encode(), ctypes.byref(h))
            if ok != 0:
                ok = nvml.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h))
            if ok != 0:
                return
            mx = ctypes.c_uint()
            if nvml.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self.nvml, self.handle = nvml, h
        except OSError:
            pass

    def _run(self):
        mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(mhz)) == 0:
                self.samples.append(mhz.value)
            if self.nvml.nvmlDeviceGetCurrentClocksEventReasons(self.handle, ctypes.byref(rs)) == 0:
                self.reasons |= rs.value
            time.sleep(self.interval)

    def __enter__(self):
        if self.nvml is not None:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self.nvml is not None:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "note": "NVML unavailable"}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": [n for b, n in self.REASONS.items() if self.reasons & b],
                "samples": len(self.samples)}


# ------------------------------------------------------------------ helpers

def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def tensor_peak(cfg, afmt, pairs):
    """Dense tensor peak (TFLOP/s) of the MMA kind the large-batch GEMMs run on.

    FP16/BF16 operands (kind::f16: the register-dequant kernel and the W4A16 and
    MXFP4 x BF16 tcgen05 kernels) take the measured cuBLAS BF16 figure, sustained
    since the GEMMs run inside a long step; NVFP4 x NVFP4 batches of 1024+ pairs
    run on the block-scaled FP4 kind and take that figure x 6 (13.5 / 2.25
    PFLOP/s nominal), MXFP4 x MXFP8 batches of 1024+ pairs on the block-scaled
    FP8 kind, x 2 (4.5 / 2.25)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16, src = float(json.load(f)["bf16_tflops_sustained"]), "measured"
    except (OSError, KeyError, ValueError):
        bf16, src = 1700.0, "fallback"
    if cfg["wfmt"] == "nvfp4" and afmt == "nvfp4" and pairs >= 1024:
        return bf16 * 13.5 / 2.25, f"{src} bf16 sustained x 13.5/2.25 (fp4)"
    if cfg["wfmt"] == "mxfp4" and afmt == "mxfp8" and pairs >= 1024:
        return bf16 * 4.5 / 2.25, f"{src} bf16 sustained x 4.5/2.25 (mx fp8)"
    return bf16, f"{src} bf16 sustained"


def expert_bytes(cfg):
    """Packed bytes of one expert: codes + block scales + globals."""
    H, I, wfmt, act = cfg["H"], cfg["I"], cfg["wfmt"], cfg["act"]
    n13 = 2 * I if act == "silu" else I
    bs = 16 if wfmt == "nvfp4" else 32
    per = lambda rows, K: rows * K // 2 + rows * K // bs  # noqa: E731
    g13 = 4 * (n13 // I) if wfmt == "nvfp4" else 0
    g2 = 4 if wfmt == "nvfp4" else 0
    return per(n13, H) + g13, per(H, I) + g2


def src_hash(kernel_src):
    """First 16 hex digits of the SHA-256 of a kernel's source file(s), concatenated."""
    files = [kernel_src] if isinstance(kernel_src, str) else list(kernel_src)
    d = hashlib.sha256()
    for f in files:
        d.update(open(os.path.join(ROOT, "block_quantised_moe_gb300", "csrc", os.path.basename(f)), "rb").read())
    return d.hexdigest()[:16]


def traffic_for(workload, stage):
    """ncu DRAM bytes (read + write) per launch of `stage`'s kernel on `workload`,
    recorded in profiles/traffic.json, or None: a record counts only while the
    kernel source it was measured on is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        recs = json.load(open(path))["records"]
    except (OSError, ValueError, KeyError):
        return None
    for rec in recs:
        if rec.get("workload") != workload or stage not in rec.get("per_launch", {}):
            continue
        src = rec.get("kernel_source")
        if src and rec.get("src_sha256_16") == src_hash(src):
            return rec["per_launch"][stage]
    return None


# --------------------------------------------------------------- oracle arm

def oracle_prepare(cfg, x, ids, w, n_pairs, seed=0):
    """CPU oracle on the first n_pairs (token, slot) pairs of a batch.

    Returns (forward callable, tokens-equivalent of the sample, description).
    Pairs outside the sample get an out-of-range id, which the oracle skips, so
    its work is proportional to the sample.  The oracle's experts are quantised
    here (untimed) from the same seeded FP32 draws the GPU layer was built from.
    """
    from oracle import moe
    from block_quantised_moe_gb300 import synth
    T, K = ids.shape
    E, H, I = cfg["E"], cfg["H"], cfg["I"]
    flat = np.full(T * K, -1, dtype=np.int64)
    flat[:n_pairs] = ids.reshape(-1)[:n_pairs]
    ids_s = flat.reshape(T, K)
    toks = np.unique(np.nonzero(ids_s >= 0)[0])
    used = np.unique(ids_s[ids_s >= 0])
    remap = np.full(E, -1)
    remap[used] = np.arange(len(used))
    ids_c = np.where(ids_s >= 0, remap[np.clip(ids_s, 0, E - 1)], -1)[toks]
    gated = cfg["act"] == "silu"
    w13s, w2s = [], []
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    for e in used:
        a, b = synth.make_expert_weights(int(e), H, I, gated, seed, device=dev)
        w13s.append([m.cpu().numpy() for m in a]), w2s.append(b.cpu().numpy())
    L = moe.quantize_layer(w13s, w2s, cfg["wfmt"], cfg["act"])
    xs, ws = x[toks], w[toks]
    afmt = cfg["afmt"]

    def forward():
        return moe.moe_forward(xs, ids_c, ws, L, afmt)

    desc = f"{n_pairs} (token, slot) pairs of a {T}x{K} batch ({len(toks)} tokens, {len(used)} experts)"
    return forward, n_pairs / K, desc


def time_repeated(fn, min_seconds):
    """Mean seconds per call over repeated calls lasting at least min_seconds."""
    n, t0 = 0, time.perf_counter()
    while True:
        fn()
        n += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            return el / n, n


def workload_name(name, T, E_override=None):
    return f"{name} T={T}" + (f" E={E_override}" if E_override else "")


def run_reference(args, cfg, world, rank):
    if rank != 0:
        return
    from block_quantised_moe_gb300 import synth
    name = args.config or HEADLINE[0]
    T = args.tokens or (HEADLINE[1] if name == HEADLINE[0] else synth.CONFIGS[name]["tokens"][-1])
    K = cfg["K"]
    x = synth.make_x(T, cfg["H"], 0).float().numpy()
    ids, w = synth.make_routing(T, cfg["E"], K, 0, zipf=cfg["zipf"])
    ids, w = ids.numpy(), w.numpy()
    # one (token, slot) pair per step keeps any --steps run within minutes
    fwd, tok, desc = oracle_prepare(cfg, x, ids, w, 1)
    for _ in range(args.warmup):
        fwd()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fwd()
    total = time.perf_counter() - t0
    value = args.steps * tok / total
    cores = len(os.sched_getaffinity(0))
    line = {
        "impl": "reference", "metric": "moe_layer_tokens_per_s", "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_name(name, T), "sample_per_step": desc},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: {desc}; oracle forward only (weights quantised untimed)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm

def replicas_for(touched_bytes, packed_bytes, max_replicas):
    """Layer replicas (each with its own routing draw) so that a replica's
    touched experts come back only after several L2 capacities of other bytes;
    at most 64 GB of copies."""
    if touched_bytes >= 3 * L2_BYTES:
        return 1
    want = math.ceil(3 * L2_BYTES / max(touched_bytes, 1.0)) + 1
    cap = max(1, int(64e9 // max(packed_bytes, 1)))
    return int(max(1, min(want, max_replicas, cap)))


class Layers:
    """Packed layers shared by the workloads (a layer does not depend on T)."""

    def __init__(self):
        self.cache = {}

    def get(self, cfg, need_fp4_tiles):
        from block_quantised_moe_gb300 import layer
        key = (cfg["E"], cfg["H"], cfg["I"], cfg["wfmt"], cfg["act"])
        ent = self.cache.get(key)
        if ent is None or (need_fp4_tiles and not ent.fp4_tiles):
            # NVFP4 layers of the big shape carry the FP4 tiles too, so that the
            # W4A16, W4A4 and decode workloads share one packed buffer
            tiles = cfg["wfmt"] == "nvfp4" and (need_fp4_tiles or cfg["H"] % 256 == 0 and cfg["I"] % 256 == 0
                                               and cfg["E"] >= 256)
            self.cache.pop(key, None)
            torch.cuda.empty_cache()
            ck = layer.make_experts_gpu(cfg["E"], cfg["H"], cfg["I"], cfg["wfmt"], cfg["act"], seed=0)
            ent = layer.PackedLayer(ck, cfg["H"], cfg["I"], fp4_tiles=tiles)
            ent.fp4_tiles = tiles
            del ck
            self.cache[key] = ent
        return ent


def algorithmic(cfg, T, touched):
    """Algorithmic HBM bytes of the layer and of each kernel, and FLOPs, per step."""
    E, H, I, K = cfg["E"], cfg["H"], cfg["I"], cfg["K"]
    b13, b2 = expert_bytes(cfg)
    x_bytes, out_bytes, route_bytes = T * H * 2, T * H * 2, T * K * 8
    layer_bytes = touched * (b13 + b2) + x_bytes + out_bytes + route_bytes
    kernel_bytes = {"gemm1": touched * b13 + x_bytes, "gemm2": touched * b2 + T * K * 4,
                    "combine": out_bytes, "route": T * K * 4}
    n13 = 2 * I if cfg["act"] == "silu" else I
    kernel_flops = {"gemm1": 2.0 * T * K * n13 * H, "gemm2": 2.0 * T * K * H * I}
    flops = kernel_flops["gemm1"] + kernel_flops["gemm2"]
    return layer_bytes, kernel_bytes, kernel_flops, flops


def roofline_of(stage_ms, kernel_bytes, kernel_flops, cfg, afmt, pairs):
    """Dominant stage, its bound and achieved / peak (see the roofline conventions)."""
    from block_quantised_moe_gb300 import abi
    names = abi.STAGES
    dom = int(np.argmax(stage_ms))
    dom_name = names[dom]
    hbm, peak_kind = peaks()
    tc_peak, tc_kind = tensor_peak(cfg, afmt, pairs)
    dom_bytes = kernel_bytes.get(dom_name, 0.0)
    dom_flops = kernel_flops.get(dom_name, 0.0)
    dom_s = stage_ms[dom] * 1e-3
    if dom_flops / (tc_peak * 1e12) > dom_bytes / (hbm * 1e9):
        roof = {"kernel": dom_name, "bound": "tensor", "achieved": dom_flops / dom_s / 1e12 if dom_s > 0 else 0.0,
                "peak": tc_peak, "peak_kind": tc_kind, "unit": "TFLOP/s"}
        roof["frac"] = roof["achieved"] / tc_peak
        # the same kernel against the byte floor, for context
        roof["hbm_frac"] = dom_bytes / dom_s / 1e9 / hbm if dom_s > 0 else 0.0
    else:
        roof = {"kernel": dom_name, "bound": "hbm", "achieved": dom_bytes / dom_s / 1e9 if dom_s > 0 else 0.0,
                "peak": hbm, "peak_kind": peak_kind, "unit": "GB/s"}
        roof["frac"] = roof["achieved"] / hbm
    roof.update(algorithmic_bytes=dom_bytes, algorithmic_flops=dom_flops)
    return roof


def measure(name, T, args, world, rank, layers, steps, headline=False, variant=None):
    """Time `steps` forwards of workload `name` at T tokens; returns the row."""
    from block_quantised_moe_gb300 import abi, layer, synth
    cfg = dict(synth.CONFIGS[name])
    if args.experts:
        cfg["E"] = args.experts
    E, H, I, K = cfg["E"], cfg["H"], cfg["I"], cfg["K"]
    afmt = cfg["afmt"]
    fp4 = cfg["wfmt"] == "nvfp4" and afmt == "nvfp4"
    packed0 = layers.get(cfg, fp4)
    plan = layer.Plan(packed0, K, T, afmt)
    if variant == "single-launch":
        abi.moe_plan_set_option(plan.handle, abi.MOE_OPT_SINGLE_LAUNCH, 1)
    seed_base = 1000 * rank
    # routing draws first: the replica count depends on the touched bytes
    b13, b2 = expert_bytes(cfg)
    draws = []
    for r in range(args.max_replicas):
        ids, w = synth.make_routing(T, E, K, seed_base + r, zipf=cfg["zipf"])
        draws.append((ids, w, len(np.unique(ids.numpy()))))
    R = replicas_for(np.mean([d[2] for d in draws]) * (b13 + b2), packed0.packed.numel(), args.max_replicas)
    R = max(1, min(R, steps))
    packed = [packed0.packed] + [packed0.packed.clone() for _ in range(R - 1)]
    xs, idss, ws, outs, binds, touched = [], [], [], [], [], []
    for r in range(R):
        x = synth.make_x(T, H, seed_base + r).cuda()
        ids, w, tch = draws[r]
        ids, w = ids.cuda(), w.cuda()
        out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
        xs.append(x), idss.append(ids), ws.append(w), outs.append(out), touched.append(tch)
        binds.append(plan.bind(x, ids, w, out, packed=packed[r]))
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()

    # The timed steps replay CUDA graphs of forwards in replica rotation: one
    # graph of L = min(steps, 64) forwards, replayed steps // L times, and one
    # of the remaining steps % L, so exactly `steps` forwards run, with no
    # instrumentation.  Per-stage times come from a second loop of the same
    # forwards in which every forward records stage events (moe_run_timed,
    # external event nodes); events split the programmatic overlap between the
    # stages, so stage times slightly overstate kernel times.
    n_ev = abi.MOE_NUM_STAGES + 1
    L = max(1, min(steps, 64))
    n_rep, rem = divmod(steps, L)
    for i in range(args.warmup):
        binds[i % R].run(stream)
    torch.cuda.synchronize()
    launches_per_fwd = abi.moe_launch_count(binds[0].handle)
    cap = torch.cuda.Stream()

    def capture(n, first, ev_sets=None):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            g.capture_begin()
            for i in range(n):
                b = binds[(first + i) % R]
                if ev_sets is not None:
                    abi.moe_run_timed(b.handle, [e.cuda_event for e in ev_sets[i]], cap)
                else:
                    b.run(cap)
            g.capture_end()
        return g

    g_main = capture(L, 0)
    g_rem = capture(rem, (n_rep * L) % R) if rem else None
    ev_sets = []
    for _ in range(L):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
        for e in evs:
            e.record(stream)  # creates the handles
        ev_sets.append(evs)
    g_ev = capture(L, 0, ev_sets)
    torch.cuda.synchronize()
    for g in (g_main, g_rem, g_ev):  # upload and warm every graph
        if g is not None:
            g.replay()
    torch.cuda.synchronize()
    barrier(world)

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler() as clk:
        torch.cuda.synchronize()
        barrier(world)
        start.record(stream)
        for c in range(n_rep):
            g_main.replay()
        if g_rem is not None:
            g_rem.replay()
        end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        # stage-timing loop: the same L forwards, each with its stage events
        g_ev.replay()
        torch.cuda.synchronize()
    ms = max_over_ranks(start.elapsed_time(end), world)
    value = job_throughput(T * steps, world, ms / 1e3)

    used = list(range(L))
    stage_ms = np.zeros(abi.MOE_NUM_STAGES)
    for i in used:
        evs = ev_sets[i]
        for s_ in range(abi.MOE_NUM_STAGES):
            stage_ms[s_] += evs[s_].elapsed_time(evs[s_ + 1])
    stage_ms /= len(used)
    # touched experts of the forwards whose events are used
    tch_ev = float(np.mean([touched[i % R] for i in used]))
    layer_bytes, kernel_bytes, kernel_flops, flops = algorithmic(cfg, T, tch_ev)
    layer_bytes_all, _, _, _ = algorithmic(cfg, T, float(np.mean(touched)))
    roof = roofline_of(stage_ms, kernel_bytes, kernel_flops, cfg, afmt, T * K)
    step_s = ms / steps * 1e-3
    hbm, hbm_kind = peaks()
    if launches_per_fwd == 1:
        # the single-launch forward: its one kernel is the dominant one; its
        # duration per launch is at most the step time of the replayed graphs
        roof = {"kernel": "single_launch_forward", "bound": "hbm", "achieved": layer_bytes / step_s / 1e9,
                "peak": hbm, "peak_kind": hbm_kind, "unit": "GB/s", "frac": layer_bytes / step_s / 1e9 / hbm,
                "algorithmic_bytes": layer_bytes, "algorithmic_flops": flops,
                "duration": "step time of the uninstrumented graph replays (an upper bound on the kernel's)"}
    row = {
        "workload": workload_name(name, T, args.experts) + (f" {variant}" if variant else ""), "value": value,
        "unit": "tokens/s",
        "ms_per_step": ms / steps, "steps": steps,
        "config": {"experts": E, "hidden": H, "intermediate": I, "top_k": K, "weights": cfg["wfmt"],
                   "activations": afmt, "act": cfg["act"], "tokens": T,
                   "l2": f"{R} layer replica(s) x {packed0.packed.numel() / 1e6:.0f} MB, each with its own "
                         f"routing draw, rotated per step; {tch_ev:.1f} touched experts x "
                         f"{(b13 + b2) / 1e6:.1f} MB per step"
                         + ("; inputs larger than L2" if tch_ev * (b13 + b2) > L2_BYTES else ""),
                   "touched_experts_mean": float(np.mean(touched))},
        "hbm_gbs_layer": layer_bytes_all / step_s / 1e9,
        "layer_roofline_frac": layer_bytes_all / step_s / 1e9 / hbm,
        "tflops": flops / step_s / 1e12,
        ("stage_us_per_stage_launches" if launches_per_fwd == 1 else "stage_us"):
            {n: round(1e3 * v, 3) for n, v in zip(abi.STAGES, stage_ms)},
        "roofline": roof,
        "gpu_launches": steps * launches_per_fwd,
        "timing": f"CUDA graph replays of {steps} forwards over {R} layer replica(s), uninstrumented; "
                  f"stage events from a second replay of {len(used)} instrumented forwards right after",
        "clocks": clk.summary(),
    }
    prof = PROFILES.get((name, T), PROFILES.get(name))
    if prof and os.path.exists(os.path.join(ROOT, prof)):
        row["roofline"]["profile"] = prof
    row["roofline"]["traffic"] = traffic_for(workload_name(name, T, args.experts), roof["kernel"])

    if headline:
        # end to end through moe_run_host: pinned host buffers, copies inside the loop
        xh = xs[0].cpu().pin_memory()
        ih = idss[0].cpu().pin_memory()
        wh = ws[0].cpu().pin_memory()
        oh = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
        n_e2e = max(1, min(args.e2e_steps, steps))
        for _ in range(3):
            abi.moe_run_host(binds[0].handle, xh, ih, wh, oh, stream)
        barrier(world)
        t0 = time.perf_counter()
        for i in range(n_e2e):
            abi.moe_run_host(binds[i % R].handle, xh, ih, wh, oh, stream)
        e2e_s = max_over_ranks(time.perf_counter() - t0, world)
        row["e2e"] = {"value": job_throughput(T * n_e2e, world, e2e_s), "unit": "tokens/s",
                      "h2d_bytes_per_step": T * H * 2 + T * K * 8, "d2h_bytes_per_step": T * H * 2,
                      "steps": n_e2e}
        row["_sample"] = (cfg, xs[0], idss[0], ws[0])
    del g_main, g_rem, g_ev, binds, packed, plan
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return row


def parse_rows(args):
    from block_quantised_moe_gb300 import synth
    spec = args.rows if args.rows is not None else ("none" if args.config else "all")
    if spec == "none":
        return []
    if spec == "all":
        return list(ROWS)
    out = []
    for item in spec.split(","):
        parts = item.split(":")
        assert parts[0] in synth.CONFIGS, parts[0]
        out.append((parts[0], int(parts[1])) + tuple(parts[2:]))
    return out


def main():
    args = parse()
    from block_quantised_moe_gb300 import synth
    name = args.config or HEADLINE[0]
    cfg = dict(synth.CONFIGS[name])
    if args.experts:
        cfg["E"] = args.experts
    T = args.tokens or (HEADLINE[1] if name == HEADLINE[0] else cfg["tokens"][-1])
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, cfg, world, rank)
        return

    from block_quantised_moe_gb300 import build
    if local == 0:
        build.build()
    barrier(world)

    layers = Layers()
    head = measure(name, T, args, world, rank, layers, args.steps, headline=True)
    cfg_s, x_s, ids_s, w_s = head.pop("_sample")
    rows = {}
    # the extra workloads run at N=1 only (multi-GPU runs time the headline)
    if world == 1:
        for row_spec in parse_rows(args):
            n, t = row_spec[0], row_spec[1]
            variant = row_spec[2] if len(row_spec) > 2 else None
            if (n, t) == (name, T) and variant is None:
                continue
            r = measure(n, t, args, world, rank, layers, args.row_steps or args.steps, variant=variant)
            rows[r.pop("workload")] = r
    line = {
        "metric": "moe_layer_tokens_per_s", "value": head["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": dict({"workload": head["workload"], "parallelism": f"replicas x{world}",
                        "mma_operands": "fp16 (fp4 weights dequantised in shared memory) x fp16 activations, "
                                        "f32 accumulate" if cfg["afmt"] == "bf16" else cfg["afmt"]},
                       **head["config"]),
        "hbm_gbs_layer": head["hbm_gbs_layer"], "layer_roofline_frac": head["layer_roofline_frac"],
        "tflops": head["tflops"], "stage_us": head["stage_us"], "roofline": head["roofline"],
        "gpu_launches": head["gpu_launches"], "timing": head["timing"], "e2e": head["e2e"],
        "clocks": head["clocks"], "rows": rows,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        x_np = x_s.float().cpu().numpy()
        ids_np, w_np = ids_s.cpu().numpy(), w_s.cpu().numpy()
        # a couple of (token, slot) pairs, forward repeated for about cpu_budget_s
        n_pairs = 2 if cfg_s["H"] * cfg_s["I"] > 4e6 else min(T * cfg_s["K"], 2 * cfg_s["K"])
        fwd, tok, desc = oracle_prepare(cfg_s, x_np, ids_np, w_np, n_pairs)
        dt, n = time_repeated(fwd, args.cpu_budget_s)
        line["cpu_baseline"] = {"value": tok / dt, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
                                "kind": "oracle",
                                "sample": f"{desc} of {head['workload']}; forward only, mean of {n} calls"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
