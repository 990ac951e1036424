"""Hand-built verify batches for the tests (explicit arrays, no recipe)."""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from speculative_decoding_verification_specdec_gb300 import workloads as W


def rows_of(cu: np.ndarray, b: int, j: int) -> int:
    return int(cu[b]) + b + j


def batch(*, V: int, ks: Sequence[int], logits: np.ndarray, draft_ids: Sequence[int],
          temperature, q: Optional[np.ndarray] = None, has_q: Optional[Sequence[int]] = None,
          allowed: Optional[np.ndarray] = None, uniforms: Optional[np.ndarray] = None,
          noise: Optional[np.ndarray] = None, max_k: Optional[int] = None, seed: int = 0,
          dtype: str = W.F32, bitmask: Optional[np.ndarray] = None, name: str = "hand") -> W.Workload:
    ks = np.asarray(ks, dtype=np.int64)
    B = ks.size
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(ks)
    N = int(cu[-1])
    T = N + B
    logits = np.asarray(logits, dtype=np.float32).reshape(T, V)
    if dtype == W.BF16:
        lg = W.f32_to_bf16_bits(logits)
    else:
        lg = np.ascontiguousarray(logits)
    rng = np.random.default_rng([seed, 777])
    if uniforms is None:
        uniforms = W.uniforms_from_bits(rng.integers(0, 2 ** 32, size=T, dtype=np.uint32))
    if noise is None:
        noise = W.exp1_from_bits(rng.integers(0, 2 ** 32, size=(T, V), dtype=np.uint32))
    if bitmask is None and allowed is not None:
        bitmask = W.pack_mask_rows(np.asarray(allowed, dtype=bool).reshape(T, V))
    temps = np.broadcast_to(np.asarray(temperature, dtype=np.float32), (B,)).copy()
    return W.Workload(
        name=name, B=B, V=V, max_k=int(ks.max() if max_k is None and B else (max_k or 0)),
        logits_dtype=dtype, logits=lg, draft_ids=np.asarray(draft_ids, dtype=np.int32).reshape(N),
        draft_probs=None if q is None else np.ascontiguousarray(np.asarray(q, dtype=np.float32).reshape(N, V)),
        has_q=None if has_q is None else np.asarray(has_q, dtype=np.uint8),
        cu_num_draft=cu, bitmask=bitmask, temperature=temps,
        uniforms=np.asarray(uniforms, dtype=np.float32).reshape(T),
        exp_noise=np.ascontiguousarray(np.asarray(noise, dtype=np.float32).reshape(T, V)),
    )
