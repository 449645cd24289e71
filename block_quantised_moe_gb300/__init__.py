"""GB300-native fused routed-expert MoE FFN over FP4 block-quantised experts.

The compute lives in ``libmoe.so`` (hand-written CUDA for sm_103a behind a C
ABI, declared in ``include/moe.h``).  ``block_quantised_moe_gb300.abi`` is the
thin ctypes binding with the same function names; ``layer`` wraps it for torch
tensors (packed experts, plans, bindings); ``tp`` and ``ep`` split a layer
over ranks (intermediate features, or expert ranges) with a rank-ordered sum
of FP32 partials; ``synth`` holds the seeded synthetic input generators.
Importing this package does not load the library; importing ``abi`` does, and
raises if it has not been built.
"""
