"""Request sharding for running one verify batch on several GPUs (one process per GPU).

Requests are independent in the verify step (each request's rows, drafts and draws are its
own), so a batch splits into contiguous request ranges with no exchange during the verify;
afterwards the counters add up and the per-request outputs concatenate in rank order.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np


def shard_bounds(cu_num_draft: Sequence[int], world: int) -> List[Tuple[int, int]]:
    """Contiguous request ranges [b0, b1), one per rank, balanced by logit rows (k_b + 1)."""
    cu = np.asarray(cu_num_draft, dtype=np.int64)
    B = cu.size - 1
    rows = np.diff(cu) + 1
    cum = np.concatenate([[0], np.cumsum(rows)])
    total = int(cum[-1])
    bounds = []
    b0 = 0
    for r in range(world):
        if r == world - 1:
            b1 = B
        else:
            target = total * (r + 1) / world
            b1 = int(np.searchsorted(cum, target, side="left"))
            b1 = max(b0, min(B, b1))
        bounds.append((b0, b1))
        b0 = b1
    return bounds


def merge_counters(per_rank: Sequence[Sequence[int]]) -> np.ndarray:
    return np.sum(np.asarray(per_rank, dtype=np.uint64), axis=0, dtype=np.uint64)


def merge_outputs(per_rank: Sequence[dict]) -> dict:
    """One batch's outputs from its shards' outputs, in rank order: per-row and per-request arrays
    concatenate (the shards are contiguous request ranges), counters and telemetry add up."""
    merged = {}
    for key in ("out_tokens", "out_num_accepted", "status"):
        merged[key] = np.concatenate([np.asarray(r[key]) for r in per_rank])
    merged["counters"] = merge_counters([r["counters"] for r in per_rank])
    if all(r.get("telemetry") is not None for r in per_rank):
        merged["telemetry"] = np.sum([np.asarray(r["telemetry"], dtype=np.uint64) for r in per_rank], axis=0,
                                     dtype=np.uint64)
    return merged
