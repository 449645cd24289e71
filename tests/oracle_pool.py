"""A process pool for the CPU oracle in the GPU parity tests (test infrastructure).

The full-size layers (hidden 7168, intermediate 2048) make the oracle slow:
quantising one expert takes seconds, and every oracle forward dequantises its
experts again.  Both jobs are independent per expert and per token (token
independence is one of the oracle's pinned invariants), so the tests farm them
out to worker processes.  Workers are started with ``spawn`` (never ``fork``:
the parent holds a CUDA context) and import only numpy and ``oracle``; the
FP32 weight draws are made in the parent and shipped as arrays.
"""

from __future__ import annotations

import os

_POOL = None


def _init():
    # one BLAS thread per worker: the pool itself is the parallelism
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"


def workers() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        n = os.cpu_count() or 2
    return max(1, min(16, n))


def pool():
    global _POOL
    if _POOL is None:
        import concurrent.futures as cf
        import multiprocessing as mp
        _POOL = cf.ProcessPoolExecutor(max_workers=workers(), mp_context=mp.get_context("spawn"),
                                       initializer=_init)
    return _POOL


# ----------------------------------------------------------- worker jobs

def quantize_expert(mats13, w2, wfmt):
    """Oracle quantisation of one expert: (codes13, scales13, [g13...], codes2, scales2, g2)."""
    import numpy as np
    from oracle import quant
    cs, ss, gs = [], [], []
    for m in mats13:
        c, s, g = quant.quantize_weight_matrix(m, wfmt)
        cs.append(c), ss.append(s), gs.append(g)
    c2, s2, g2 = quant.quantize_weight_matrix(w2, wfmt)
    return np.concatenate(cs), np.concatenate(ss), gs, c2, s2, g2


def forward_tokens(x, ids_c, w, layer, afmt):
    """Oracle forward of a chunk of token rows, with its re-quantisation envelope."""
    import requant_envelope
    return requant_envelope.forward_with_envelope(x, ids_c, w, layer, afmt)
