"""Seeded synthetic inputs for batched speculative-decoding verification.

This module only manufactures inputs. It holds none of the verification
arithmetic (no acceptance test, no residual, no counters); both the CUDA path
and the CPU oracle consume exactly the bytes produced here.

Layout of one batch (the verify step of the vLLM source tour, pyshine.com
"vllm-2", section "Verification: rejection sampling on the GPU": target logits
for every draft position plus one bonus position):

* B requests; request b has k_b = cu[b+1] - cu[b] drafts (ragged).
* draft d(b, j) = cu[b] + j, j in [0, k_b); N = cu[B] drafts in total.
* logit row t(b, j) = cu[b] + b + j, j in [0, k_b]; j = k_b is the bonus row;
  T = N + B rows in total.
* bitmask: int32 [T, ceil(V/32)], bit (i & 31) of word i >> 5, 1 = allowed
  (one mask row per speculative position plus the bonus, as in the tour's
  section "Grammar gates: structured output").
* uniforms: float32 [T]; exp_noise: float32 [T, V], Exp(1) samples > 0.

Random numbers the method consumes (uniforms, exponential noise) are drawn
here and passed in, so that both sides see the same values.

Every tensor has its own substream ``numpy.random.default_rng([seed, tag])``.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import os
from typing import Optional, Sequence, Tuple

import numpy as np

F32 = "f32"
BF16 = "bf16"

# One substream per tensor: default_rng([seed, tag]).
_TAGS = {
    "k": 1,
    "temperature": 2,
    "greedy_pick": 3,
    "q_pick": 4,
    "mask_pick": 5,
    "logits": 6,
    "draft_logit_noise": 7,
    "draft_sample": 8,
    "draft_argmax_pick": 9,
    "draft_uniform_id": 10,
    "forced_invalid": 11,
    "mask": 12,
    "uniforms": 13,
    "exp_noise": 14,
    "ngram_histories": 15,
    "top_k_top_p": 16,
}

_ROW_BLOCK = 64  # rows generated per block (one substream each) for the [T, V] tensors


def substream(seed: int, tag: str, block: Optional[int] = None) -> np.random.Generator:
    """Substream of one tensor; tensors generated in row blocks get one substream per block."""
    if block is None:
        return np.random.default_rng([int(seed), _TAGS[tag]])
    return np.random.default_rng([int(seed), _TAGS[tag], int(block)])


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _for_blocks(n: int, block: int, fn) -> None:
    """fn(block_index, r0, r1) over [0, n) in blocks, on a thread pool (results do not depend
    on the thread count: every block draws from its own substream)."""
    starts = list(range(0, n, block))
    if len(starts) <= 1 or _threads() == 1:
        for i, r0 in enumerate(starts):
            fn(i, r0, min(n, r0 + block))
        return
    with concurrent.futures.ThreadPoolExecutor(max_workers=_threads()) as ex:
        list(ex.map(lambda i: fn(i, starts[i], min(n, starts[i] + block)), range(len(starts))))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even), integer ops only."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((bits >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((bits + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def uniforms_from_bits(bits: np.ndarray) -> np.ndarray:
    """float32 in [0, 1): the top 24 bits of a uint32 times 2^-24 (exact in fp32)."""
    return (bits >> np.uint32(8)).astype(np.float32) * np.float32(2.0 ** -24)


def exp1_from_bits(bits: np.ndarray) -> np.ndarray:
    """Exp(1) samples: -log((top24 + 0.5) * 2^-24) in fp64, stored as fp32 (always > 0)."""
    v = ((bits >> np.uint32(8)).astype(np.float64) + 0.5) * (2.0 ** -24)
    return (-np.log(v)).astype(np.float32)


def pack_mask_rows(allowed: np.ndarray, pad_value: bool = False) -> np.ndarray:
    """Pack bool [rows, V] into int32 [rows, ceil(V/32)], LSB-first, 1 = allowed."""
    allowed = np.atleast_2d(allowed)
    rows, V = allowed.shape
    W = (V + 31) // 32
    padded = np.full((rows, W * 32), pad_value, dtype=bool)
    padded[:, :V] = allowed
    packed = np.packbits(padded.reshape(rows, W * 4, 8), axis=-1, bitorder="little")
    return np.ascontiguousarray(packed.reshape(rows, W * 4)).view("<u4").astype(np.uint32).view(np.int32)


def unpack_mask_rows(words: np.ndarray, V: int) -> np.ndarray:
    """Inverse of pack_mask_rows (bits >= V dropped)."""
    words = np.atleast_2d(np.asarray(words, dtype=np.int32))
    rows, W = words.shape
    b = np.unpackbits(words.view(np.uint32).astype("<u4").view(np.uint8).reshape(rows, W * 4),
                      axis=-1, bitorder="little").astype(bool)
    return b[:, :V]


@dataclasses.dataclass
class Workload:
    """One verify batch, host-resident (numpy)."""

    name: str
    B: int
    V: int
    max_k: int
    logits_dtype: str                    # "f32" or "bf16"
    logits: np.ndarray                   # [T, V] float32, or uint16 bf16 bits
    draft_ids: np.ndarray                # [N] int32
    draft_probs: Optional[np.ndarray]    # [N, V] float32 or None
    has_q: Optional[np.ndarray]          # [B] uint8 or None
    cu_num_draft: np.ndarray             # [B+1] int32
    bitmask: Optional[np.ndarray]        # [T, W] int32 or None
    temperature: np.ndarray              # [B] float32
    uniforms: np.ndarray                 # [T] float32
    exp_noise: np.ndarray                # [T, V] float32
    description: str = ""
    top_k: Optional[np.ndarray] = None   # [B] int32 or None (<= 0: no top-k)
    top_p: Optional[np.ndarray] = None   # [B] float32 or None (>= 1: no top-p)

    @property
    def N(self) -> int:
        return int(self.cu_num_draft[-1])

    @property
    def T(self) -> int:
        return self.N + self.B

    @property
    def W(self) -> int:
        return (self.V + 31) // 32

    @property
    def k(self) -> np.ndarray:
        return np.diff(self.cu_num_draft).astype(np.int64)

    def row(self, b: int, j: int) -> int:
        return int(self.cu_num_draft[b]) + b + j

    def logits_f32(self, rows=slice(None)) -> np.ndarray:
        if self.logits_dtype == BF16:
            return bf16_bits_to_f32(self.logits[rows])
        return self.logits[rows]

    def nbytes(self) -> int:
        tot = 0
        for a in (self.logits, self.draft_ids, self.draft_probs, self.has_q, self.cu_num_draft,
                  self.bitmask, self.temperature, self.uniforms, self.exp_noise):
            if a is not None:
                tot += a.nbytes
        return tot

    def subset(self, requests: Sequence[int], name: Optional[str] = None) -> "Workload":
        """The batch made of the listed requests only, rows and drafts copied in that order."""
        requests = [int(b) for b in requests]
        k = self.k
        rows, drafts = [], []
        cu = [0]
        for b in requests:
            rows.extend(range(self.row(b, 0), self.row(b, int(k[b])) + 1))
            drafts.extend(range(int(self.cu_num_draft[b]), int(self.cu_num_draft[b + 1])))
            cu.append(cu[-1] + int(k[b]))
        rows = np.asarray(rows, dtype=np.int64)
        drafts = np.asarray(drafts, dtype=np.int64)
        sel = np.asarray(requests, dtype=np.int64)
        return Workload(
            name=name or f"{self.name}[subset {len(requests)}]",
            B=len(requests), V=self.V, max_k=self.max_k, logits_dtype=self.logits_dtype,
            logits=np.ascontiguousarray(self.logits[rows]),
            draft_ids=np.ascontiguousarray(self.draft_ids[drafts]),
            draft_probs=None if self.draft_probs is None else np.ascontiguousarray(self.draft_probs[drafts]),
            has_q=None if self.has_q is None else np.ascontiguousarray(self.has_q[sel]),
            cu_num_draft=np.asarray(cu, dtype=np.int32),
            bitmask=None if self.bitmask is None else np.ascontiguousarray(self.bitmask[rows]),
            temperature=np.ascontiguousarray(self.temperature[sel]),
            uniforms=np.ascontiguousarray(self.uniforms[rows]),
            exp_noise=np.ascontiguousarray(self.exp_noise[rows]),
            description=self.description,
            top_k=None if self.top_k is None else np.ascontiguousarray(self.top_k[sel]),
            top_p=None if self.top_p is None else np.ascontiguousarray(self.top_p[sel]),
        )


# ----------------------------------------------------------------------------------------------
# generic batch builder
# ----------------------------------------------------------------------------------------------

def _softmax_rows_f64(x: np.ndarray) -> np.ndarray:
    # drafter-side synthesis of q only; the verifier's own softmax lives in each implementation
    m = np.max(x, axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def _mask_row(rng: np.random.Generator, V: int, density: float, run_len: int, run_frac: float) -> np.ndarray:
    """Allowed ids of one grammar row: contiguous runs at unaligned random starts plus singles."""
    target = max(1, int(round(density * V)))
    allowed = np.zeros(V, dtype=bool)
    n_runs = int(round(density * run_frac * V / run_len))
    if n_runs > 0 and V >= run_len:
        starts = rng.integers(0, V - run_len + 1, size=n_runs)
        allowed[(starts[:, None] + np.arange(run_len)[None, :]).ravel()] = True
    need = target - int(allowed.sum())
    if need > 0:
        free = np.flatnonzero(~allowed)
        allowed[rng.choice(free, size=min(need, free.size), replace=False)] = True
    return allowed


def make_batch(
    seed: int,
    *,
    name: str = "batch",
    B: int,
    V: int,
    k: Sequence[int] | int | tuple = 3,
    max_k: Optional[int] = None,
    logits_dtype: str = F32,
    logit_sigma: float = 2.0,
    temperature: str | float = 1.0,       # float, "uniform(lo,hi)", "half_greedy(lo,hi)" or array
    q_mode: str = "all",                  # "all" (draft model), "none" (model-free), "half"
    draft_sigma: float = 1.0,
    draft_temperature: str = "request",   # drafter softmax uses the request temperature (1.0 if greedy)
    mf_argmax_frac: float = 0.4,          # model-free drafts: share equal to the target argmax
    mask: str = "none",                   # "none", "all", "half", "ones" (all-ones rows)
    mask_density: float = 0.05,
    mask_run_len: int = 64,
    mask_run_frac: float = 0.8,
    forced_invalid_frac: float = 0.0,     # masked requests: share of drafts set to a disallowed id
    description: str = "",
    top_k=None,                           # None, an int for every request, or an int array [B]
    top_p=None,                           # None, a float for every request, or a float array [B]
) -> Workload:
    """Build one seeded batch. Parameters follow the workload recipes of the pages' configs."""
    # ---- ragged draft counts
    if isinstance(k, tuple) and len(k) == 2 and k and isinstance(k[0], int) and isinstance(k[1], int) and k[0] <= k[1]:
        kk = substream(seed, "k").integers(k[0], k[1] + 1, size=B)
    elif np.isscalar(k):
        kk = np.full(B, int(k), dtype=np.int64)
    else:
        kk = np.asarray(list(k), dtype=np.int64)
        assert kk.size == B
    cu = np.zeros(B + 1, dtype=np.int64)
    cu[1:] = np.cumsum(kk)
    N = int(cu[-1])
    T = N + B
    if max_k is None:
        max_k = int(kk.max()) if B else 0
    row_of_draft = np.repeat(cu[:-1] + np.arange(B), kk) + (np.arange(N) - np.repeat(cu[:-1], kk))
    bonus_rows = cu[1:] + np.arange(B)
    req_of_row = np.repeat(np.arange(B), kk + 1)

    # ---- per-request sampling settings
    if isinstance(temperature, str):
        kind, args = temperature.split("(")
        lo, hi = (float(a) for a in args.rstrip(")").split(","))
        temps = substream(seed, "temperature").uniform(lo, hi, size=B).astype(np.float32)
        if kind == "half_greedy":
            greedy = np.zeros(B, dtype=bool)
            greedy[substream(seed, "greedy_pick").permutation(B)[: B // 2]] = True
            temps[greedy] = 0.0
        else:
            assert kind == "uniform"
    elif np.isscalar(temperature):
        temps = np.full(B, float(temperature), dtype=np.float32)
    else:
        temps = np.asarray(temperature, dtype=np.float32)
    if q_mode == "all":
        has_q_req = np.ones(B, dtype=bool)
    elif q_mode == "none":
        has_q_req = np.zeros(B, dtype=bool)
    else:
        assert q_mode == "half"
        has_q_req = np.zeros(B, dtype=bool)
        has_q_req[substream(seed, "q_pick").permutation(B)[: B // 2]] = True
    if mask in ("none",):
        masked_req = np.zeros(B, dtype=bool)
    elif mask in ("all", "ones"):
        masked_req = np.ones(B, dtype=bool) if mask == "all" else np.zeros(B, dtype=bool)
    else:
        assert mask == "half"
        masked_req = np.zeros(B, dtype=bool)
        masked_req[substream(seed, "mask_pick").permutation(B)[: B // 2]] = True

    # ---- target logits
    if logits_dtype == BF16:
        logits = np.empty((T, V), dtype=np.uint16)
    else:
        logits = np.empty((T, V), dtype=np.float32)

    def _gen_logits(i, r0, r1):
        blk = substream(seed, "logits", i).standard_normal(size=(r1 - r0, V), dtype=np.float32)
        blk *= np.float32(logit_sigma)
        logits[r0:r1] = f32_to_bf16_bits(blk) if logits_dtype == BF16 else blk

    _for_blocks(T, _ROW_BLOCK, _gen_logits)

    def stored_logits(rows):
        return bf16_bits_to_f32(logits[rows]) if logits_dtype == BF16 else logits[rows]

    # ---- grammar masks
    allowed_rows = {}
    bitmask = None
    if mask != "none":
        W = (V + 31) // 32
        bitmask = np.full((T, W), -1, dtype=np.int32)   # all-ones rows (bits >= V set too)
        masked_rows = [t for t in range(T) if masked_req[req_of_row[t]]]

        def _gen_masks(i, r0, r1):
            for t in masked_rows[r0:r1]:
                a = _mask_row(substream(seed, "mask", t), V, mask_density, mask_run_len, mask_run_frac)
                allowed_rows[t] = a
                bitmask[t] = pack_mask_rows(a[None, :])[0]

        _for_blocks(len(masked_rows), _ROW_BLOCK, _gen_masks)

    # ---- drafts (and draft probabilities q)
    draft_ids = np.zeros(N, dtype=np.int32)
    q_any = bool(has_q_req.any())
    draft_probs = np.zeros((N, V), dtype=np.float32) if q_any else None
    req_of_draft = np.repeat(np.arange(B), kk)

    def _gen_drafts(bi, d0, d1):
        nb = d1 - d0
        rng_dn = substream(seed, "draft_logit_noise", bi)
        rng_ds = substream(seed, "draft_sample", bi)
        rng_da = substream(seed, "draft_argmax_pick", bi)
        rng_du = substream(seed, "draft_uniform_id", bi)
        rng_fi = substream(seed, "forced_invalid", bi)
        rows = row_of_draft[d0:d1]
        reqs = req_of_draft[d0:d1]
        z = stored_logits(rows).astype(np.float64)
        noise = rng_dn.standard_normal(size=(nb, V), dtype=np.float32) * np.float32(draft_sigma)
        v_sample = rng_ds.random(size=nb)
        pick_arg = rng_da.random(size=nb) < mf_argmax_frac
        v_uid = rng_du.random(size=nb)
        forced = rng_fi.random(size=nb) < forced_invalid_frac
        v_forced = rng_fi.random(size=nb)
        allowed = np.ones((nb, V), dtype=bool)
        has_mask = np.zeros(nb, dtype=bool)
        for i, t in enumerate(rows):
            a = allowed_rows.get(int(t))
            if a is not None:
                allowed[i] = a
                has_mask[i] = True
        x = np.zeros(nb, dtype=np.int64)
        qsel = has_q_req[reqs]
        if qsel.any():
            tq = np.where((temps[reqs] > 0) & (draft_temperature == "request"), temps[reqs], 1.0)[qsel]
            s_ = (z[qsel] + noise[qsel]) / tq[:, None]
            s_ = np.where(allowed[qsel], s_, -np.inf)
            s_ -= s_.max(axis=1, keepdims=True)
            q = np.exp(s_)
            q /= q.sum(axis=1, keepdims=True)
            draft_probs[d0:d1][qsel] = q.astype(np.float32)
            cdf = np.cumsum(q, axis=1)
            thr = v_sample[qsel] * cdf[:, -1]
            xq = np.minimum((cdf <= thr[:, None]).sum(axis=1), V - 1)
            # guard against the cdf tail landing on a zero-probability id: take the last positive one
            zero = q[np.arange(q.shape[0]), xq] <= 0.0
            if zero.any():
                for r in np.flatnonzero(zero):
                    xq[r] = int(np.flatnonzero(q[r] > 0.0)[-1])
            x[qsel] = xq
        msel = ~qsel
        if msel.any():
            zz = np.where(allowed[msel], z[msel], -np.inf)
            x_arg = np.argmax(zz, axis=1)
            cnt = allowed[msel].sum(axis=1)
            target = np.floor(v_uid[msel] * cnt).astype(np.int64) + 1
            cs = np.cumsum(allowed[msel], axis=1)
            x_uni = (cs < target[:, None]).sum(axis=1)
            x[msel] = np.where(pick_arg[msel], x_arg, x_uni)
        fsel = forced & has_mask
        if fsel.any():
            bad = ~allowed[fsel]
            cnt = bad.sum(axis=1)
            target = np.floor(v_forced[fsel] * cnt).astype(np.int64) + 1
            cs = np.cumsum(bad, axis=1)
            xf = (cs < target[:, None]).sum(axis=1)
            x[fsel] = np.where(cnt > 0, xf, x[fsel])
        draft_ids[d0:d1] = np.clip(x, 0, V - 1)

    _for_blocks(N, _ROW_BLOCK, _gen_drafts)

    # ---- random numbers consumed by the verifier
    uniforms = uniforms_from_bits(substream(seed, "uniforms").integers(0, 2 ** 32, size=T, dtype=np.uint32))
    exp_noise = np.empty((T, V), dtype=np.float32)

    def _gen_noise(i, r0, r1):
        bits = substream(seed, "exp_noise", i).integers(0, 2 ** 32, size=(r1 - r0, V), dtype=np.uint32)
        exp_noise[r0:r1] = exp1_from_bits(bits)

    _for_blocks(T, _ROW_BLOCK, _gen_noise)

    has_q = None
    if q_any and not has_q_req.all():
        has_q = has_q_req.astype(np.uint8)
    tk = None if top_k is None else np.broadcast_to(np.asarray(top_k, dtype=np.int32), (B,)).copy()
    tp = None if top_p is None else np.broadcast_to(np.asarray(top_p, dtype=np.float32), (B,)).copy()
    return Workload(
        name=name, B=B, V=V, max_k=int(max_k), logits_dtype=logits_dtype, logits=logits,
        draft_ids=draft_ids, draft_probs=draft_probs, has_q=has_q,
        cu_num_draft=cu.astype(np.int32), bitmask=bitmask, temperature=temps,
        uniforms=uniforms, exp_noise=exp_noise, description=description, top_k=tk, top_p=tp,
    )


# ----------------------------------------------------------------------------------------------
# the five workload recipes (sizes and distributions of the pages' verify step)
# ----------------------------------------------------------------------------------------------

CONFIG_NAMES = [
    "tiny_random_B4_k3_V1000_f32",
    "greedy_model_free_B64_k3to5_V32000_f32",
    "random_draft_model_B256_k4_V128256_f32",
    "structured_output_B128_k5_V151936_f32",
    "large_mixed_B1024_k1to8_V151936_bf16",
]

CONFIG_DESCRIPTIONS = [
    "tiny random-sampling verify: B=4, k=3, V=1000, fp32 logits ~N(0,2), q=softmax(logits+N(0,1)), "
    "x~q, T=1.0, no bitmask",
    "greedy model-free verify: B=64, k~U{3,4,5}, V=32000, fp32 logits ~N(0,3), no q, 40% of drafts = "
    "target argmax else uniform id, T=0",
    "random draft-model verify: B=256, k=4, V=128256, fp32 logits ~N(0,3), q=softmax((logits+N(0,0.5))/T), "
    "x~q, T~U[0.5,1.2]",
    "structured-output verify: B=128, k=5, V=151936, fp32 logits ~N(0,3), bitmask on every row with 5% "
    "allowed (runs of 64 + singles), 20% of drafts forced grammar-invalid, masked q as in the draft-model "
    "recipe, T=0.8",
    "large mixed batch: B=1024, k~U{1..8}, V=151936, bf16 logits ~N(0,3), q on half the requests (rest "
    "model-free), half greedy / half T~U[0.5,1.2], bitmask (5% allowed) on half the requests",
]


def config(i: int, seed: Optional[int] = None) -> Workload:
    """Workload recipe i (seed defaults to the recipe index)."""
    s = i if seed is None else seed
    name, desc = CONFIG_NAMES[i], CONFIG_DESCRIPTIONS[i]
    if i == 0:
        return make_batch(s, name=name, description=desc, B=4, V=1000, k=3, logit_sigma=2.0,
                          temperature=1.0, q_mode="all", draft_sigma=1.0)
    if i == 1:
        return make_batch(s, name=name, description=desc, B=64, V=32000, k=(3, 5), logit_sigma=3.0,
                          temperature=0.0, q_mode="none", mf_argmax_frac=0.4)
    if i == 2:
        return make_batch(s, name=name, description=desc, B=256, V=128256, k=4, logit_sigma=3.0,
                          temperature="uniform(0.5,1.2)", q_mode="all", draft_sigma=0.5)
    if i == 3:
        return make_batch(s, name=name, description=desc, B=128, V=151936, k=5, logit_sigma=3.0,
                          temperature=0.8, q_mode="all", draft_sigma=0.5, mask="all",
                          forced_invalid_frac=0.2)
    if i == 4:
        return make_batch(s, name=name, description=desc, B=1024, V=151936, k=(1, 8), logits_dtype=BF16,
                          logit_sigma=3.0, temperature="half_greedy(0.5,1.2)", q_mode="half",
                          draft_sigma=0.5, mf_argmax_frac=0.4, mask="half", forced_invalid_frac=0.2)
    raise IndexError(i)


# ----------------------------------------------------------------------------------------------
# n-gram proposer inputs: token histories
# ----------------------------------------------------------------------------------------------

@dataclasses.dataclass
class Histories:
    """Token histories of a batch back to back: tokens int32 [total], cu_hist int64 [B+1]."""
    name: str
    tokens: np.ndarray
    cu_hist: np.ndarray
    V: int

    @property
    def B(self) -> int:
        return int(self.cu_hist.size - 1)


def ngram_histories(seed: int, B: int = 1024, L: Tuple[int, int] = (1024, 8192), V: int = 151936,
                    copy_frac: float = 0.5, span: Tuple[int, int] = (8, 64), name: Optional[str] = None) -> Histories:
    """Histories in which text repeats, as in the workloads the n-gram drafter is meant for (output
    that quotes its prompt, code that repeats identifiers): each history grows in pieces, a piece
    being either fresh uniform tokens or a copy of an earlier span (with probability copy_frac),
    piece lengths uniform in `span`; lengths uniform in L. Inputs only."""
    rng = substream(seed, "ngram_histories")
    lens = rng.integers(L[0], L[1] + 1, size=B)
    out = []
    for b in range(B):
        n = int(lens[b])
        h = np.empty(n, dtype=np.int32)
        pos = 0
        while pos < n:
            m = min(int(rng.integers(span[0], span[1] + 1)), n - pos)
            if pos > m and rng.random() < copy_frac:
                src = int(rng.integers(0, pos - m + 1))
                h[pos:pos + m] = h[src:src + m]
            else:
                h[pos:pos + m] = rng.integers(0, V, size=m, dtype=np.int32)
            pos += m
        out.append(h)
    cu = np.zeros(B + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lens)
    tokens = np.concatenate(out) if B else np.zeros(0, dtype=np.int32)
    return Histories(name=name or f"ngram_histories_B{B}_L{L[0]}to{L[1]}_V{V}", tokens=tokens, cu_hist=cu, V=V)


def top_k_top_p_batch(seed: int = 5, B: int = 256, V: int = 128256) -> Workload:
    """The random draft-model batch (B=256, k=4, V=128256, fp32, T ~ U[0.5, 1.2]) with per-request
    top-k in {off, 20, 50, 200} and top-p in {off, 0.8, 0.9, 0.95}, drawn independently (the
    drafter's q is not filtered). Inputs only."""
    rng = substream(seed, "top_k_top_p")
    tk = rng.choice(np.array([0, 20, 50, 200], dtype=np.int32), size=B)
    tp = rng.choice(np.array([1.0, 0.8, 0.9, 0.95], dtype=np.float32), size=B)
    return make_batch(seed, name=f"random_draft_model_topk_topp_B{B}_k4_V{V}_f32", B=B, V=V, k=4,
                      logit_sigma=3.0, temperature="uniform(0.5,1.2)", q_mode="all", draft_sigma=0.5,
                      top_k=tk, top_p=tp,
                      description="random draft-model batch with per-request top-k / top-p")
