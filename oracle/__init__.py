"""CPU oracle for the block-quantised fused MoE layer.

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow, obviously correct
definition that the CUDA library is checked against.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import it.  It shares no code with the CUDA path
(``block_quantised_moe_gb300``) and neither imports the other; the only thing
both sides consume is the seeded input generator ``block_quantised_moe_gb300.synth``,
which holds none of the method's arithmetic.

What it computes (sources are cited per function):

* ``codecs``   E2M1 / E4M3 / E8M0 decode tables and round-to-nearest-even
               encoders (the NVFP4 / MXFP4 / MXFP8 element and scale formats).
* ``quant``    NVFP4 (16-element blocks, E4M3 scale, FP32 global scale) and
               MX (32-element blocks, E8M0 scale) quantisers and dequantisers.
* ``routing``  the expert-sorted, tile-padded pair list built from ``topk_ids``.
* ``moe``      the fused routed-expert FFN forward in FP32:
               y_t = sum_k w_tk * W2_e( act( W13_e x_t ) ).

Pins (tests that tie this code to something other than itself) live in
``tests/test_oracle_*.py``: exhaustive code tables against torch's float8 casts,
rounding ties, on-grid round trips, float64 brute force on tiny layers and the
invariants of the method (top-1 = single expert, zero weights, linearity in
``topk_weights``, permutation of the top-k slots, token independence).
Every oracle function has at least one such pin; none is "parity unpinned".
"""

from . import codecs, quant, routing, moe  # noqa: F401
