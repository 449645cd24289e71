"""The single-launch decode forward (the pages' unified persistent-grid path).

Decode plans run their whole forward as one cooperative launch whose phases
(routing and activation staging, GEMM1, the h re-quantiser, GEMM2, the combine)
are separated by bounded grid barriers.  It runs the same arithmetic in the
same order as the one-launch-per-stage forward, so the two must agree bit for
bit; the oracle comparisons of the other test files run on it too, since it is
the default for these plans.  A barrier whose arrival is withheld must give up
within its bound, report a timeout and leave the context usable.
"""

import numpy as np
import pytest
import torch

from block_quantised_moe_gb300 import synth
import moe_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from block_quantised_moe_gb300 import build
    build.build()
    from block_quantised_moe_gb300 import abi, layer
    return abi, layer


def _forward(lib, packed, x, ids, w, K, afmt, single, max_tokens=None):
    abi, layer = lib
    T = x.shape[0]
    plan = layer.Plan(packed, K, max_tokens or T, afmt)
    abi.moe_plan_set_option(plan.handle, abi.MOE_OPT_SINGLE_LAUNCH, 1 if single else 0)
    out = torch.full((T, packed.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    b = plan.bind(x, ids, w, out)
    b.run()
    rc, st = b.device_status()
    torch.cuda.synchronize()
    assert rc == abi.MOE_OK
    return out, abi.moe_launch_count(b.handle), st, (plan, b)


MODES = [("nvfp4", "silu", "bf16"), ("nvfp4", "silu", "nvfp4"), ("nvfp4", "silu", "mxfp8"),
         ("nvfp4", "relu2", "bf16"), ("nvfp4", "relu2", "nvfp4"), ("mxfp4", "relu2", "mxfp8"),
         ("mxfp4", "relu2", "bf16"), ("mxfp4", "silu", "mxfp8")]


@pytest.mark.parametrize("wfmt,act,afmt", MODES)
@pytest.mark.parametrize("T", [1, 16, 40])
def test_single_launch_matches_per_stage_launches_bit_for_bit(lib, wfmt, act, afmt, T):
    abi, layer = lib
    cfg = dict(E=8, H=256, I=512, K=2, zipf=None)
    ck = layer.make_experts_gpu(cfg["E"], cfg["H"], cfg["I"], wfmt, act)
    packed = layer.PackedLayer(ck, cfg["H"], cfg["I"])
    x, ids, w = tl.make_inputs(cfg, T, seed=100 + T)
    one, n1, st1, _ = _forward(lib, packed, x, ids, w, cfg["K"], afmt, True, max_tokens=64)
    many, n2, st2, _ = _forward(lib, packed, x, ids, w, cfg["K"], afmt, False, max_tokens=64)
    assert n1 == 1 and n2 > 1
    assert st1 == st2
    assert torch.equal(one, many), f"{wfmt}/{act}/{afmt} T={T}: single launch differs"
    tl.check_close(one.float().cpu().numpy(), tl.oracle_forward(ck, cfg["H"], cfg["I"], x, ids, w, afmt),
                   f"single launch {wfmt}/{act}/{afmt} T={T}")


@pytest.mark.parametrize("name,T", [("decode_e128_h2048_i768_k8", 1), ("decode_e128_h2048_i768_k8", 64),
                                    ("mxfp4_mxfp8_relu2_e128_h4096_i1024_k4", 1),
                                    ("mxfp4_mxfp8_relu2_e128_h4096_i1024_k4", 64)])
def test_single_launch_on_the_decode_layers(lib, name, T):
    abi, layer = lib
    cfg = synth.CONFIGS[name]
    ck = layer.make_experts_gpu(cfg["E"], cfg["H"], cfg["I"], cfg["wfmt"], cfg["act"])
    packed = layer.PackedLayer(ck, cfg["H"], cfg["I"])
    x, ids, w = tl.make_inputs(cfg, T, seed=3)
    ids[0, 0] = cfg["E"] + 1  # one dropped pair, counted by both paths
    one, n1, st1, _ = _forward(lib, packed, x, ids, w, cfg["K"], cfg["afmt"], True)
    many, _, st2, _ = _forward(lib, packed, x, ids, w, cfg["K"], cfg["afmt"], False)
    assert n1 == 1
    assert st1 == st2 == [1, 1, 0, 0]
    assert torch.equal(one, many)


def test_withheld_grid_barrier_arrival_times_out_and_the_next_forward_is_correct(lib):
    abi, layer = lib
    cfg = synth.CONFIGS["decode_e128_h2048_i768_k8"]
    ck = layer.make_experts_gpu(cfg["E"], cfg["H"], cfg["I"], cfg["wfmt"], cfg["act"])
    packed = layer.PackedLayer(ck, cfg["H"], cfg["I"])
    T = 16
    x, ids, w = tl.make_inputs(cfg, T, seed=9)
    plan = layer.Plan(packed, cfg["K"], T, cfg["afmt"])
    abi.moe_plan_set_option(plan.handle, abi.MOE_OPT_SINGLE_LAUNCH, 1)
    out = torch.empty(T, cfg["H"], dtype=torch.bfloat16, device="cuda")
    b = plan.bind(x, ids, w, out)
    rc, st = abi.moe_selftest_grid_barrier_timeout(b.handle)
    assert rc == abi.MOE_ERR_TIMEOUT
    assert st[0] & 2
    b.run()
    rc, st = b.device_status()
    torch.cuda.synchronize()
    assert rc == abi.MOE_OK and st == [0, 0, 0, 0]
    tl.check_close(out.float().cpu().numpy(),
                   tl.oracle_forward(ck, cfg["H"], cfg["I"], x, ids, w, cfg["afmt"]), "after the barrier timeout")
