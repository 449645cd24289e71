"""The first contraction on its own: GEMM1's output h (before any
re-quantisation), read back in expert-sorted slot order, against the oracle's
step 3 for every routed (token, slot) pair.  Small batches run on the
register-dequant kernel, batches of 1024+ pairs with 32+ pairs per expert on
the tcgen05 kernel.  Operands are exact on both sides (x^ and the weights are
representable in the 16-bit MMA operands), so only the order of the FP32 sums
and the SiLU's exp differ: the bar is far tighter than the layer output's."""

import numpy as np
import pytest

from block_quantised_moe_gb300 import synth
import moe_testlib as tl

pytestmark = pytest.mark.gpu

CASES = [  # E, H, I, K, weights, activation, activations, T
    (16, 512, 256, 4, "nvfp4", "silu", "bf16", 16),
    (16, 512, 256, 4, "nvfp4", "relu2", "nvfp4", 16),
    (8, 256, 512, 2, "nvfp4", "silu", "bf16", 600),
    (8, 256, 512, 2, "mxfp4", "relu2", "mxfp8", 600),
    (8, 7168, 2048, 4, "nvfp4", "silu", "bf16", 256),   # full-length K on the tcgen05 kernel
    (8, 4096, 1024, 4, "mxfp4", "relu2", "mxfp8", 256),
]


@pytest.mark.parametrize("E,H,I,K,wfmt,act,afmt,T", CASES)
def test_gemm1_hidden_matches_oracle(E, H, I, K, wfmt, act, afmt, T):
    import torch
    from block_quantised_moe_gb300 import build
    build.build()
    from block_quantised_moe_gb300 import layer
    from oracle import moe, quant
    ck = layer.make_experts_gpu(E, H, I, wfmt, act)
    packed = layer.PackedLayer(ck, H, I)
    cfg = dict(synth.CONFIGS["tiny_e8_h256_i512_k2"], E=E, H=H, I=I, K=K)
    x, ids, w = tl.make_inputs(cfg, T, seed=3)
    plan = layer.Plan(packed, K, T, afmt)
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    b = plan.bind(x, ids, w, out)
    b.run()
    torch.cuda.synchronize()
    h = b.hidden()
    sorted_pair = b.routing()["sorted_pair"]
    assert h.shape[0] == sorted_pair.shape[0]

    ids_np = ids.cpu().numpy()
    xh = quant.qdq_rows(x.float().cpu().numpy(), afmt)
    used = np.unique(ids_np)
    L = tl.oracle_layer_for(ck, H, I, used)
    got, want = [], []
    for ce, e in enumerate(used):
        slots = np.nonzero([p >= 0 and ids_np[p // K, p % K] == e for p in sorted_pair])[0]
        toks = sorted_pair[slots] // K
        got.append(h[slots])
        want.append(moe.expert_hidden(L, ce, xh[toks]))
    got, want = np.concatenate(got).astype(np.float64), np.concatenate(want).astype(np.float64)
    assert got.shape[0] == T * K  # every pair has its row
    rms = np.sqrt(np.mean(want ** 2))
    assert np.linalg.norm(got - want) / np.linalg.norm(want) <= 1e-4
    assert np.max(np.abs(got - want) / (np.abs(want) + rms)) <= 1e-3
