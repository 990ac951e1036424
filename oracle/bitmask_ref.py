"""Bitmask scatter on the host: TEST INFRASTRUCTURE ONLY (the plain definition the GPU kernel is
checked against; only the tests, the smoke check and the benchmark's CPU leg use it).

"vLLM tour part 2" (pyshine.com/vllm-2), section "Grammar gates: structured output": the scheduler
sends grammar masks compacted to only the constrained requests, in scheduler order; the runner's
batch has its own order and per-request speculative offsets, so the runner rebuilds an index
mapping that walks both orderings, accounting for the spec-token offset of every request, and
places each request's rows at its rows of the batch. A request that is not constrained gets
all-ones rows (every token allowed).
"""
from __future__ import annotations

import numpy as np


def bitmask_scatter(compact: np.ndarray, constrained, cu_num_draft: np.ndarray, B: int, V: int) -> np.ndarray:
    """compact: int32 [R_c, W], the k_b + 1 rows of each constrained request back to back in
    scheduler order; constrained: the batch index of each constrained request, scheduler order.
    Returns the batch-order bitmask int32 [T, W], T = cu[B] + B.

    Readings (the pages are silent on malformed input): an id outside [0, B) owns no rows; a
    request listed twice takes the rows of its first listing (the second listing's rows are
    skipped over); rows a request would take beyond the end of `compact` allow nothing (zero
    words), which the verify reports as an empty mask row; a request whose offsets are malformed
    (cu[0] != 0, cu[b] < 0, cu[b+1] < cu[b] or cu[b+1] > cu[B], as the verify's BAD_OFFSETS) owns
    no rows and its output rows are left as they were (all ones here)."""
    W = (V + 31) // 32
    cu = np.asarray(cu_num_draft, dtype=np.int64)
    T = max(int(cu[B]), 0) + B
    out = np.full((T, W), -1, dtype=np.int32)
    R_c = int(compact.shape[0]) if compact is not None else 0
    off = 0
    placed = set()
    def malformed(b):
        return cu[0] != 0 or cu[b] < 0 or cu[b + 1] < cu[b] or cu[b + 1] > cu[B]

    for b in constrained:
        b = int(b)
        if b < 0 or b >= B or malformed(b):
            continue
        k = int(cu[b + 1] - cu[b])
        if b not in placed:
            placed.add(b)
            t0 = int(cu[b]) + b
            for j in range(k + 1):
                src = off + j
                out[t0 + j] = compact[src] if src < R_c else 0
        off += k + 1
    return out
