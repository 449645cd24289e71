"""bench.py's host arithmetic: the algorithmic bytes behind the roofline, the
tensor peak it divides by, and the rule that ncu traffic is reported only for
the kernel source it was measured on."""

import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from block_quantised_moe_gb300 import synth  # noqa: E402


@pytest.mark.parametrize("name", sorted(synth.CONFIGS))
def test_expert_bytes_match_the_packed_format(name):
    cfg = synth.CONFIGS[name]
    H, I = cfg["H"], cfg["I"]
    b13, b2 = bench.expert_bytes(cfg)
    if cfg["wfmt"] == "nvfp4":
        # E2M1 codes (1/2 B) + one E4M3 scale per 16 (1/16 B) = 0.5625 B per
        # element, plus an FP32 global per matrix (gate and up, or w1; down)
        per_elem, g13 = 0.5625, (8 if cfg["act"] == "silu" else 4)
        g2 = 4
    else:
        # E2M1 codes + one E8M0 scale per 32: 0.53125 B per element, no globals
        per_elem, g13, g2 = 0.53125, 0, 0
    n13 = 2 * I if cfg["act"] == "silu" else I
    assert b13 == n13 * H * per_elem + g13
    assert b2 == H * I * per_elem + g2


def test_gated_nvfp4_expert_is_three_matrices():
    cfg = synth.CONFIGS["decode_e128_h2048_i768_k8"]
    b13, b2 = bench.expert_bytes(cfg)
    assert b13 + b2 == 3 * 2048 * 768 * 0.5625 + 12


def test_tensor_peak_follows_the_mma_kind():
    w4a4 = synth.CONFIGS["prefill_w4a4_e256_h7168_i2048_k8"]
    w4a16 = synth.CONFIGS["prefill_w4a16_e256_h7168_i2048_k8"]
    f16, _ = bench.tensor_peak(w4a16, w4a16["afmt"], 65536)
    fp4, kind = bench.tensor_peak(w4a4, w4a4["afmt"], 65536)
    assert fp4 == pytest.approx(f16 * 6) and "fp4" in kind
    # below 1024 pairs every expert runs on the register-dequant (FP16 MMA) kernel
    small, _ = bench.tensor_peak(w4a4, w4a4["afmt"], 1000)
    assert small == pytest.approx(f16)
    # MXFP4 weights with MXFP8 activations: the block-scaled FP8 kind, twice the FP16 rate
    mx = synth.CONFIGS["mxfp4_mxfp8_relu2_e128_h4096_i1024_k4"]
    fp8, kind = bench.tensor_peak(mx, mx["afmt"], 16384)
    assert fp8 == pytest.approx(f16 * 2) and "fp8" in kind


def test_traffic_is_reported_only_for_the_measured_source(tmp_path, monkeypatch):
    # a record counts only while its kernel source hashes to what it was measured on
    src = "k_grouped_mma.cu"
    good = bench.src_hash(src)
    prof = tmp_path / "profiles"
    prof.mkdir()
    rec = {"workload": "w T=1", "kernel_source": [src],
           "per_launch": {"gemm1": 123.0}, "command": "ncu --metrics dram__bytes_read.sum"}
    for sha, want in ((good, 123.0), ("0" * 16, None)):
        (prof / "traffic.json").write_text(json.dumps({"records": [dict(rec, src_sha256_16=sha)]}))
        monkeypatch.setattr(bench, "ROOT", str(tmp_path))
        # src_hash reads the real source tree
        monkeypatch.setattr(bench, "src_hash", lambda s, _h=good: _h)
        assert bench.traffic_for("w T=1", "gemm1") == want
        assert bench.traffic_for("other T=1", "gemm1") is None
        assert bench.traffic_for("w T=1", "gemm2") is None


def test_committed_traffic_records_name_their_command():
    stored = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for rec in stored["records"]:
        assert rec["command"].startswith("ncu ")
        assert set(rec["per_launch"]) <= {"gemm1", "gemm2", "combine", "route", "quant_x", "quant_h"}
