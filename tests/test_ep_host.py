"""Expert parallelism on the CPU with two gloo ranks: each rank runs the oracle on
its range of experts with the router's ids in its own numbering (the slicing
and id mapping of block_quantised_moe_gb300.ep, the same code that prepares the
device tensors; other ranks' pairs get id -1 and are skipped), and the
rank-ordered all-reduce of the partials must give the unsharded layer's output,
the same bytes on both ranks.  Every activation format qualifies, NVFP4
included: each (token, slot) pair's h row lives on one rank.
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
    d = synth.make_random_codes(E, H, I, wfmt, act == "silu", seed=9)
    return {k: (None if v is None else v.numpy()) for k, v in d.items()}


def _oracle_layer(d, wfmt, act):
    from oracle import moe
    return moe.QuantLayer(wfmt=wfmt, act=act, **d)


def _inputs():
    from block_quantised_moe_gb300 import synth
    x = synth.make_x(T, H, 4).float().numpy()
    ids, w = synth.make_routing(T, E, K, 4)
    return x, ids.numpy(), w.numpy()


def test_expert_bounds_slicing_and_ids():
    from block_quantised_moe_gb300 import ep
    assert ep.expert_bounds(256, 3, 4) == (192, 256)
    with pytest.raises(ValueError):
        ep.expert_bounds(6, 0, 4)  # 6 experts do not split into 4 equal ranges
    d = _layer_arrays("nvfp4", "silu")
    s = ep.shard_expert_arrays(d, E, 1, 2)
    for k in ("w13_codes", "w13_scales", "w13_global", "w2_codes", "w2_scales", "w2_global"):
        assert np.array_equal(s[k], d[k][2:4]), k  # experts 2 and 3, every array
    m = ep.shard_expert_arrays(_layer_arrays("mxfp4", "relu2"), E, 0, 2)
    assert m["w13_global"] is None and m["w2_codes"].shape == (2, H, I // 2)
    ids = np.array([[0, 3], [2, 1], [-1, 2], [4, 2]], dtype=np.int32)
    want = np.array([[-1, 1], [0, -1], [-1, 0], [-1, 0]], dtype=np.int32)
    assert np.array_equal(ep.local_ids(ids, 2, 4), want)  # out-of-range ids stay dropped
    got = ep.local_ids(torch.from_numpy(ids).to(torch.int64), 2, 4)
    assert got.dtype == torch.int32 and np.array_equal(got.numpy(), want)


def _rank_main(rank, world, port, wfmt, act, afmt, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from block_quantised_moe_gb300 import ep, tp
        from oracle import moe
        d = _layer_arrays(wfmt, act)
        x, ids, w = _inputs()
        e0, e1 = ep.expert_bounds(E, rank, world)
        part = moe.moe_forward(x, ep.local_ids(ids, e0, e1), w,
                               _oracle_layer(ep.shard_expert_arrays(d, E, rank, world), wfmt, act), afmt)
        y = tp.ordered_all_reduce(torch.from_numpy(np.ascontiguousarray(part, dtype=np.float32)))
        out.put((rank, y.numpy().tobytes()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("wfmt,act,afmt", [("nvfp4", "silu", "bf16"), ("nvfp4", "silu", "nvfp4"),
                                           ("mxfp4", "relu2", "mxfp8")])
def test_two_gloo_ranks_sum_to_the_unsharded_layer(wfmt, act, afmt):
    from oracle import moe
    world = 2
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
