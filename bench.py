#!/usr/bin/env python
"""MoE-layer throughput of libmoe on GB300, one JSON line on rank 0.

Workload: the decode layer E=128 experts, hidden 2048, intermediate 768, top-8,
NVFP4 weights with BF16 activations and gated SiLU, at T tokens per step
(default 64; 1, 4 and 16 are the other decode batch sizes of this layer).  A
step is one full forward of the layer (routing, GEMM1 + SiLU, GEMM2 x topk
weight, combine) through the C ABI over one batch of seeded synthetic input.
Steps rotate over R independent layer replicas and routing draws whose packed
weights together exceed L2, so every step streams its experts from HBM.

``value`` is tokens/s with inputs resident in HBM, timed with CUDA events on
the launching stream; ``e2e`` is the same through ``moe_run_host`` with pinned
host buffers (H2D of x / ids / weights and D2H of the output inside the timed
loop).  ``roofline`` is for the dominant kernel, from per-stage CUDA events
recorded by ``moe_run_timed`` inside the timed region.  ``cpu_baseline`` times
the CPU oracle on a bounded sample.  ``--impl reference`` times only the oracle
(the reference arm).  Multi-GPU runs (torchrun) are independent replicas: one
layer per rank, no collective on the data path, weak scaling.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_CONFIG = "decode_e128_h2048_i768_k8"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--tokens", type=int, default=64)
    ap.add_argument("--replicas", type=int, default=4)
    ap.add_argument("--e2e-steps", type=int, default=300)
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
    MXFP4 tcgen05 kernels) take the measured cuBLAS BF16 figure, sustained since
    the GEMMs run inside a long step; NVFP4 x NVFP4 batches of 1024+ pairs run on
    the block-scaled FP4 kind and take that figure x 6 (13.5 / 2.25 PFLOP/s
    nominal)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16, src = float(json.load(f)["bf16_tflops_sustained"]), "measured"
    except (OSError, KeyError, ValueError):
        bf16, src = 1700.0, "fallback"
    if cfg["wfmt"] == "nvfp4" and afmt == "nvfp4" and pairs >= 1024:
        return bf16 * 13.5 / 2.25, f"{src} bf16 sustained x 13.5/2.25 (fp4)"
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


def traffic_record(kernel_src):
    """ncu DRAM bytes per launch recorded in profiles/, valid only for the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path))
    except (OSError, ValueError):
        return None, None
    src = open(os.path.join(ROOT, "block_quantised_moe_gb300", "csrc", kernel_src), "rb").read()
    return rec, hashlib.sha256(src).hexdigest()[:16]


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
    for e in used:
        a, b = synth.make_expert_weights(int(e), H, I, gated, seed, device="cuda")
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


def run_reference(args, cfg, world, rank):
    if rank != 0:
        return
    from block_quantised_moe_gb300 import synth
    T, K = args.tokens, cfg["K"]
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
        "config": {"workload": f"{args.config} T={T}", "sample_per_step": desc},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: {desc}; oracle forward only (weights quantised untimed)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm

def main():
    args = parse()
    from block_quantised_moe_gb300 import synth
    cfg = dict(synth.CONFIGS[args.config])
    if args.experts:
        cfg["E"] = args.experts
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, cfg, world, rank)
        return

    from block_quantised_moe_gb300 import build
    if local == 0:
        build.build()
    barrier(world)
    from block_quantised_moe_gb300 import abi, layer

    E, H, I, K, T = cfg["E"], cfg["H"], cfg["I"], cfg["K"], args.tokens
    afmt = cfg["afmt"]
    R = max(1, args.replicas)
    seed_base = 1000 * rank
    ck = layer.make_experts_gpu(E, H, I, cfg["wfmt"], cfg["act"], seed=0)
    # W4A4 layers also carry the FP4 tiles of the block-scaled tensor-core kernel
    packed0 = layer.PackedLayer(ck, H, I, fp4_tiles=cfg["wfmt"] == "nvfp4" and afmt == "nvfp4")
    del ck
    packed = [packed0.packed] + [packed0.packed.clone() for _ in range(R - 1)]
    plan = layer.Plan(packed0, K, T, afmt)
    xs, idss, ws, outs, binds, touched = [], [], [], [], [], []
    for r in range(R):
        x = synth.make_x(T, H, seed_base + r).cuda()
        ids, w = synth.make_routing(T, E, K, seed_base + r, zipf=cfg["zipf"])
        touched.append(len(np.unique(ids.numpy())))
        ids, w = ids.cuda(), w.cuda()
        out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
        xs.append(x), idss.append(ids), ws.append(w), outs.append(out)
        binds.append(plan.bind(x, ids, w, out, packed=packed[r]))
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()

    # The timed steps replay CUDA graphs of L = 4R forwards (replicas in
    # rotation, so every step streams a different layer copy).  The first
    # forward of each of the NG graphs records per-stage events (external event
    # nodes), so after the timed loop each event set holds the stage times of
    # its graph's last replay inside the timed region.
    n_ev = abi.MOE_NUM_STAGES + 1
    L, NG = 4 * R, 8
    ev_sets = []
    for _ in range(NG):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
        for e in evs:
            e.record(stream)  # creates the handles
        ev_sets.append(evs)
    for i in range(args.warmup):
        binds[i % R].run(stream)
    torch.cuda.synchronize()
    launches_per_fwd = abi.moe_launch_count(binds[0].handle)
    cap = torch.cuda.Stream()
    graphs = []
    with torch.cuda.stream(cap):
        for j in range(NG):
            g = torch.cuda.CUDAGraph()
            g.capture_begin()
            for i in range(L):
                if i == 0:
                    abi.moe_run_timed(binds[0].handle, [e.cuda_event for e in ev_sets[j]], cap)
                else:
                    binds[i % R].run(cap)
            g.capture_end()
            graphs.append(g)
    torch.cuda.synchronize()
    for g in graphs:  # upload and warm every graph
        g.replay()
    torch.cuda.synchronize()
    barrier(world)

    n_rep, rem = divmod(args.steps, L)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler() as clk:
        torch.cuda.synchronize()
        barrier(world)
        start.record(stream)
        for c in range(n_rep):
            graphs[c % NG].replay()
        for i in range(rem):
            binds[i % R].run(stream)
        end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms = max_over_ranks(start.elapsed_time(end), world)
    value = job_throughput(T * args.steps, world, ms / 1e3)

    used = ev_sets[:max(1, min(NG, n_rep))]
    stage_ms = np.zeros(abi.MOE_NUM_STAGES)
    for evs in used:
        for s_ in range(abi.MOE_NUM_STAGES):
            stage_ms[s_] += evs[s_].elapsed_time(evs[s_ + 1])
    stage_ms /= len(used)

    # algorithmic bytes (HBM) of the whole layer and of each kernel, per step
    b13, b2 = expert_bytes(cfg)
    tch = float(np.mean(touched))
    x_bytes, out_bytes, route_bytes = T * H * 2, T * H * 2, T * K * 8
    layer_bytes = tch * (b13 + b2) + x_bytes + out_bytes + route_bytes
    kernel_bytes = {"gemm1": tch * b13 + x_bytes, "gemm2": tch * b2 + T * K * 4,
                    "combine": out_bytes, "route": T * K * 4}
    flops = 2 * T * K * (3 if cfg["act"] == "silu" else 2) * H * I
    n13 = 2 * I if cfg["act"] == "silu" else I
    kernel_flops = {"gemm1": 2.0 * T * K * n13 * H, "gemm2": 2.0 * T * K * H * I}
    names = abi.STAGES
    dom = int(np.argmax(stage_ms))
    dom_name = names[dom]
    hbm, peak_kind = peaks()
    tc_peak, tc_kind = tensor_peak(cfg, afmt, T * K)
    dom_bytes = kernel_bytes.get(dom_name, 0.0)
    dom_flops = kernel_flops.get(dom_name, 0.0)
    dom_s = stage_ms[dom] * 1e-3
    # the kernel's bound is the larger of its two floors: bytes at the HBM peak, FLOPs at the tensor peak
    if dom_flops / (tc_peak * 1e12) > dom_bytes / (hbm * 1e9):
        roof = {"kernel": dom_name, "bound": "tensor", "achieved": dom_flops / dom_s / 1e12 if dom_s > 0 else 0.0,
                "peak": tc_peak, "peak_kind": tc_kind, "unit": "TFLOP/s"}
        roof["frac"] = roof["achieved"] / tc_peak
    else:
        roof = {"kernel": dom_name, "bound": "hbm", "achieved": dom_bytes / dom_s / 1e9 if dom_s > 0 else 0.0,
                "peak": hbm, "peak_kind": peak_kind, "unit": "GB/s"}
        roof["frac"] = roof["achieved"] / hbm
    rec, src_hash = traffic_record("k_grouped_mma.cu")
    traffic = None
    if rec and rec.get("src_sha256_16") == src_hash and rec.get("workload") == f"{args.config} T={T}":
        traffic = rec.get("per_launch", {}).get(dom_name)

    # end to end through moe_run_host: pinned host buffers, copies inside the loop
    xh = xs[0].cpu().pin_memory()
    ih = idss[0].cpu().pin_memory()
    wh = ws[0].cpu().pin_memory()
    oh = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
    n_e2e = max(1, min(args.e2e_steps, args.steps))
    for _ in range(3):
        abi.moe_run_host(binds[0].handle, xh, ih, wh, oh, stream)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(n_e2e):
        abi.moe_run_host(binds[i % R].handle, xh, ih, wh, oh, stream)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e_value = job_throughput(T * n_e2e, world, e2e_s)

    line = {
        "metric": "moe_layer_tokens_per_s", "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"{args.config} T={T}" + (f" E={E}" if args.experts else ""), "experts": E, "hidden": H, "intermediate": I,
                   "top_k": K, "weights": cfg["wfmt"], "activations": afmt, "act": cfg["act"],
                   "tokens": T, "parallelism": f"replicas x{world}",
                   "l2": f"{R} layer replicas x {packed0.packed.numel() / 1e6:.0f} MB rotated per step (> L2)",
                   "touched_experts_mean": tch},
        "hbm_gbs_layer": layer_bytes / (ms / args.steps * 1e-3) / 1e9,
        "tflops": flops / (ms / args.steps * 1e-3) / 1e12,
        "stage_us": {n: round(1e3 * v, 3) for n, v in zip(names, stage_ms)},
        "roofline": dict(roof, traffic=traffic, algorithmic_bytes=dom_bytes, algorithmic_flops=dom_flops),
        "layer_roofline_frac": layer_bytes / (ms / args.steps * 1e-3) / 1e9 / hbm,
        "gpu_launches": args.steps * launches_per_fwd,
        "timing": f"CUDA graphs of {L} forwards replayed; stage events from the last replay of each of "
                  f"{len(used)} graphs",
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": T * H * 2 + T * K * 8,
                "d2h_bytes_per_step": T * H * 2, "steps": n_e2e},
        "clocks": clk.summary(),
    }

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        x_np = xs[0].float().cpu().numpy()
        ids_np, w_np = idss[0].cpu().numpy(), ws[0].cpu().numpy()
        # two tokens' pairs, forward repeated for about cpu_budget_s
        fwd, tok, desc = oracle_prepare(cfg, x_np, ids_np, w_np, min(T * K, 2 * K))
        dt, n = time_repeated(fwd, args.cpu_budget_s)
        line["cpu_baseline"] = {"value": tok / dt, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
                                "kind": "oracle",
                                "sample": f"{desc} of {args.config} T={T}; forward only, mean of {n} calls"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
