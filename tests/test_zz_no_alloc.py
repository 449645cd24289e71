"""moe_run_no_alloc: the forward for callers that cannot allocate device memory
(plugin interfaces that pass no workspace, applications whose pool owns the
device).  It must give what moe_bind + moe_run give, call after call, while its
scratch is the library's own static device array.  Collected last on purpose."""

import pytest
import torch

from block_quantised_moe_gb300 import synth
import moe_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    from block_quantised_moe_gb300 import build
    build.build()
    from block_quantised_moe_gb300 import abi, layer
    cfg = synth.CONFIGS["decode_e128_h2048_i768_k8"]
    ck = layer.make_experts_gpu(cfg["E"], cfg["H"], cfg["I"], cfg["wfmt"], cfg["act"])
    packed = layer.PackedLayer(ck, cfg["H"], cfg["I"])
    packed.ck = ck
    return abi, layer, cfg, packed


def packed_ck(setup):
    return setup[3].ck


def test_no_alloc_matches_moe_run_on_two_calls_in_a_row(setup):
    abi, layer, cfg, packed = setup
    T = 16
    plan = layer.Plan(packed, cfg["K"], T, cfg["afmt"])
    assert plan.scratch_bytes <= abi.MOE_NO_ALLOC_SCRATCH_BYTES
    for call, seed in enumerate((11, 12)):  # different inputs: stale scratch must not leak into call 2
        x, ids, w = tl.make_inputs(cfg, T, seed=seed)
        if call == 1:
            ids[0, 0] = cfg["E"] + 3  # one out-of-range id: dropped and counted in the status word
        ref = torch.empty(T, cfg["H"], dtype=torch.bfloat16, device="cuda")
        b = plan.bind(x, ids, w, ref)
        b.run()
        rc_ref, st_ref = b.device_status()
        got = torch.full((T, cfg["H"]), float("nan"), dtype=torch.bfloat16, device="cuda")
        abi.moe_run_no_alloc(plan.handle, packed.packed, x, ids, w, T, got)
        rc, st = abi.moe_no_alloc_device_status(plan.handle)
        torch.cuda.synchronize()
        # same plan, kernels, launch order and inputs: the outputs are bit-identical
        assert torch.equal(got, ref), f"no-alloc call {call + 1} differs from moe_run"
        assert rc == abi.MOE_OK and rc_ref == abi.MOE_OK
        assert st == st_ref == ([0, 0, 0, 0] if call == 0 else [1, 1, 0, 0])
        # and both agree with the oracle
        tl.check_close(got.float().cpu().numpy(),
                       tl.oracle_forward(packed_ck(setup), cfg["H"], cfg["I"], x, ids, w, cfg["afmt"]),
                       f"no-alloc call {call + 1}")


def test_no_alloc_rejects_plans_beyond_its_scratch(setup):
    abi, layer, cfg, packed = setup
    big, nbytes, _ = abi.moe_plan(packed.wplan, cfg["K"], 4096, cfg["afmt"])
    assert nbytes > abi.MOE_NO_ALLOC_SCRATCH_BYTES
    x = torch.zeros(1, cfg["H"], dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros(1, cfg["K"], dtype=torch.int32, device="cuda")
    w = torch.zeros(1, cfg["K"], device="cuda")
    out = torch.empty_like(x)
    with pytest.raises(abi.MoeError) as ei:
        abi.moe_run_no_alloc(big, packed.packed, x, ids, w, 1, out)
    assert ei.value.status == abi.MOE_ERR_CAPACITY
    abi.moe_destroy_plan(big)
