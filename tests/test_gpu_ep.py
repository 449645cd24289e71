"""Expert parallelism on one GPU, with the ranks run one after the other (no
kernel of one rank waits on another's): each rank's range of experts runs
through the C ABI with the router's ids in its own numbering (other ranks'
pairs dropped) and an FP32 output (MOE_OPT_OUT_F32); the partials are added in
rank order and the sum is compared with the oracle's unsharded layer -- on the
register-dequant kernel (a decode batch) and on the tcgen05 kernels (1200
pairs).  The collective (block_quantised_moe_gb300.tp.ordered_all_reduce) is
covered by two gloo ranks on the CPU (tests/test_ep_host.py)."""

import pytest
import torch

from block_quantised_moe_gb300 import synth
import moe_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wfmt,act,afmt", [("nvfp4", "silu", "bf16"), ("nvfp4", "silu", "nvfp4"),
                                           ("mxfp4", "relu2", "mxfp8")])
@pytest.mark.parametrize("T", [8, 600])
def test_expert_ranges_sum_to_the_layer(wfmt, act, afmt, T):
    from block_quantised_moe_gb300 import build
    build.build()
    from block_quantised_moe_gb300 import ep, layer
    cfg = dict(synth.CONFIGS["tiny_e8_h256_i512_k2"])
    E, H, I, K = cfg["E"], cfg["H"], cfg["I"], cfg["K"]
    ck = layer.make_experts_gpu(E, H, I, wfmt, act)
    x, ids, w = tl.make_inputs(cfg, T, seed=13)
    world = 2
    ranks = [ep.EPLayer(ck, H, I, r, world, K, T, afmt) for r in range(world)]
    parts = [r.partial(x, ids, w) for r in ranks]
    torch.cuda.synchronize()
    y = parts[0].clone()
    for p in parts[1:]:
        y += p
    y_ref = tl.oracle_forward(ck, H, I, x, ids, w, afmt)
    tl.check_close(y.to(torch.bfloat16).float().cpu().numpy(), y_ref, f"ep {wfmt}/{act}/{afmt} T={T}")
