"""Expert routing reference: counting sort of (token, slot) pairs by expert (oracle).

Test infrastructure: see the package docstring for who may import this.

The fused MoE op takes ``topk_ids`` / ``topk_weights`` as inputs (b12x project
page, "Using it": ``fused_moe.bind(..., topk_weights=tw, topk_ids=ti)``) and
groups the pairs by expert before the two expert contractions.  The reading
used throughout this project:

* pair index p = t*K + k for token t and slot k;
* ``counts[e]``   number of pairs whose id is e;
* ``offsets``     exclusive prefix sum of counts rounded up to a multiple of
                  ``pad`` (the tile the grouped kernels work in), length E+1;
* ``sorted_pair`` pair indices grouped by expert, ascending p inside a group
                  (a stable sort), each group followed by -1 up to its padded
                  length;
* ``pair_pos[p]`` position of pair p in ``sorted_pair``;
* ids outside [0, E) are dropped: pair_pos = -1, counted in ``dropped``.
"""

from __future__ import annotations

import numpy as np


def route(topk_ids: np.ndarray, num_experts: int, pad: int) -> dict:
    ids = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    P = ids.shape[0]
    E = int(num_experts)
    counts = np.zeros(E, dtype=np.int32)
    for e in range(E):
        counts[e] = np.count_nonzero(ids == e)
    padded = (counts + pad - 1) // pad * pad
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(padded)
    sorted_pair = np.full(int(offsets[-1]), -1, dtype=np.int32)
    pair_pos = np.full(P, -1, dtype=np.int32)
    for e in range(E):
        ps = np.nonzero(ids == e)[0]  # ascending p: stable in p
        sorted_pair[offsets[e]:offsets[e] + len(ps)] = ps
        pair_pos[ps] = offsets[e] + np.arange(len(ps), dtype=np.int32)
    valid = (ids >= 0) & (ids < E)
    return dict(counts=counts, offsets=offsets, sorted_pair=sorted_pair,
                pair_pos=pair_pos, dropped=int(P - np.count_nonzero(valid)))
