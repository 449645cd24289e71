"""Tensor parallelism over the intermediate dimension, on the CPU with two gloo
ranks: each rank runs the oracle on its slice of every expert (the slicing of
block_quantised_moe_gb300.tp, the same code that slices the device tensors),
and the rank-ordered all-reduce of the partials must give the unsharded
layer's output, the same bytes on both ranks.  With BF16 activations only the
order of the FP32 additions differs; with MXFP8 activations h's per-32-element
re-quantisation is also the same on every slice boundary that is a multiple of 64.
"""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

E, H, I, K, T = 4, 128, 256, 2, 12


def _layer_arrays(wfmt, act):
    from block_quantised_moe_gb300 import synth
    d = synth.make_random_codes(E, H, I, wfmt, act == "silu", seed=5)
    return {k: (None if v is None else v.numpy()) for k, v in d.items()}


def _oracle_layer(d, wfmt, act):
    from oracle import moe
    return moe.QuantLayer(wfmt=wfmt, act=act, **d)


def _inputs():
    from block_quantised_moe_gb300 import synth
    x = synth.make_x(T, H, 3).float().numpy()
    ids, w = synth.make_routing(T, E, K, 3)
    return x, ids.numpy(), w.numpy()


def test_shard_bounds_and_shapes():
    from block_quantised_moe_gb300 import tp
    assert tp.shard_bounds(256, 1, 2) == (128, 256)
    with pytest.raises(ValueError):
        tp.shard_bounds(192, 0, 2)  # 96-wide slices are not a multiple of 64
    d = _layer_arrays("nvfp4", "silu")
    s = tp.shard_arrays(d, I, True, 1, 2)
    assert s["w13_codes"].shape == (E, I, H // 2)         # its half of the gate rows, then of the up rows
    assert np.array_equal(s["w13_codes"][:, :I // 2], d["w13_codes"][:, I // 2:I])
    assert np.array_equal(s["w13_codes"][:, I // 2:], d["w13_codes"][:, I + I // 2:])
    assert s["w2_codes"].shape == (E, H, I // 4)            # its half of W2's columns, two codes per byte
    assert np.array_equal(s["w2_scales"], d["w2_scales"][:, :, (I // 2) // 16:])
    assert np.array_equal(s["w13_global"], d["w13_global"])  # whole-matrix scales are kept


def _rank_main(rank, world, port, wfmt, act, afmt, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from block_quantised_moe_gb300 import tp
        from oracle import moe
        d = _layer_arrays(wfmt, act)
        x, ids, w = _inputs()
        part = moe.moe_forward(x, ids, w, _oracle_layer(tp.shard_arrays(d, I, act == "silu", rank, world), wfmt, act),
                               afmt)
        y = tp.ordered_all_reduce(torch.from_numpy(np.ascontiguousarray(part, dtype=np.float32)))
        out.put((rank, y.numpy().tobytes()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("wfmt,act,afmt", [("nvfp4", "silu", "bf16"), ("mxfp4", "relu2", "mxfp8"),
                                           ("mxfp4", "silu", "bf16")])
def test_two_gloo_ranks_sum_to_the_unsharded_layer(wfmt, act, afmt):
    from oracle import moe
    world = 2
    port = None
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, wfmt, act, afmt, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert got[0][1] == got[1][1]  # the rank-ordered sum: the same bytes on every rank
    y = np.frombuffer(got[0][1], dtype=np.float32).reshape(T, H)
    x, ids, w = _inputs()
    ref = moe.moe_forward(x, ids, w, _oracle_layer(_layer_arrays(wfmt, act), wfmt, act), afmt)
    err = np.linalg.norm(y.astype(np.float64) - ref) / np.linalg.norm(ref)
    assert err < 1e-5, err
