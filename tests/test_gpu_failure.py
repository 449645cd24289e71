"""Failure detection without a GPU fault.

Every device-side wait of the library is bounded.  A wait that nothing
completes gives up after about two seconds, records the timeout in the device
status word and lets its kernel return, so the context stays usable.  The test
makes one such wait run out (an mbarrier that nothing arrives on), checks the
status the host reads back, then runs a forward on the same context and checks
it against the oracle.
"""

import time

import pytest
import torch

from block_quantised_moe_gb300 import synth
import moe_testlib as tl

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_the_context_stays_usable():
    from block_quantised_moe_gb300 import build
    build.build()
    from block_quantised_moe_gb300 import abi, layer
    status_dev = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    rc, st = abi.moe_selftest_wait_timeout(status_dev)
    waited = time.perf_counter() - t0
    assert rc == abi.MOE_ERR_TIMEOUT
    assert st == [2, 0, 0, 0]  # timeout bit only; the word was cleared first
    assert 1.0 < waited < 60.0

    cfg = synth.CONFIGS["tiny_e8_h256_i512_k2"]
    E, H, I, K = cfg["E"], cfg["H"], cfg["I"], cfg["K"]
    ck = layer.make_experts_gpu(E, H, I, cfg["wfmt"], cfg["act"])
    packed = layer.PackedLayer(ck, H, I)
    x, ids, w = tl.make_inputs(cfg, 16)
    plan = layer.Plan(packed, K, 16, cfg["afmt"])
    out = torch.empty(16, H, dtype=torch.bfloat16, device="cuda")
    b = plan.bind(x, ids, w, out)
    b.run()
    torch.cuda.synchronize()
    assert b.device_status()[0] == abi.MOE_OK
    tl.check_close(out.float().cpu().numpy(), tl.oracle_forward(ck, H, I, x, ids, w, cfg["afmt"]), "after timeout")
