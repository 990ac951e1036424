"""Pins of the CPU oracle: facts the pages and the mathematics fix, independent of the
oracle's own code. Each check raises AssertionError on failure and takes the path of
the oracle library to check, so that the mutation tests can run the same pins against
deliberately broken copies of the oracle.
"""
from __future__ import annotations

import dataclasses
import json
import os

import numpy as np
from scipy import special, stats

import oracle
from speculative_decoding_verification_specdec_gb300 import metrics
from speculative_decoding_verification_specdec_gb300 import workloads as W

from _hand import batch, rows_of

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
CHI2_CRIT_DF7 = 24.32  # chi-square critical value, 7 degrees of freedom, alpha = 0.001


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------------------------
# worked counter example ("Structured output speculative decoding acceptance",
# section "Work a denominator example")
# ---------------------------------------------------------------------------------------------

def _greedy_counter_batch(n_invalid_first: int, n_full: int, n_reject0: int, k: int = 5, V: int = 16,
                          seed: int = 0):
    """Greedy requests with a unique argmax per row: n_invalid_first requests whose first draft the
    grammar forbids, n_full requests whose drafts are all the argmax, n_reject0 requests whose first
    draft is not the argmax."""
    rng = np.random.default_rng(seed)
    B = n_invalid_first + n_full + n_reject0
    ks = [k] * B
    T = B * (k + 1)
    logits = rng.normal(0, 1, size=(T, V)).astype(np.float32)
    ystar = rng.integers(0, V, size=T)
    logits[np.arange(T), ystar] = 10.0
    allowed = np.ones((T, V), dtype=bool)
    cu = np.arange(B + 1) * k
    drafts = np.zeros(B * k, dtype=np.int32)
    for b in range(B):
        for j in range(k):
            t = rows_of(cu, b, j)
            drafts[b * k + j] = ystar[t]
        t0 = rows_of(cu, b, 0)
        if b < n_invalid_first:
            bad = (ystar[t0] + 1) % V
            allowed[t0, bad] = False
            drafts[b * k] = bad
        elif b >= n_invalid_first + n_full:
            drafts[b * k] = (ystar[t0] + 1) % V
    return batch(V=V, ks=ks, logits=logits, draft_ids=drafts, temperature=0.0, allowed=allowed)


def check_worked_counter_example(lib_path=None):
    g = _golden("counters_worked_example.json")
    kw = {} if lib_path is None else {"lib_path": lib_path}
    ex = g["worked_example"]
    r = oracle.verify(_greedy_counter_batch(40, 120, 40), **kw)
    assert [int(c) for c in r.counters] == [ex["R"], ex["I"], ex["D"], ex["A"]], r.counters
    rates = metrics.acceptance_rates(r.counters)
    assert abs(rates["conditional_acceptance"] - ex["conditional_acceptance"]) < 1e-12
    assert abs(rates["grammar_survival"] - ex["grammar_survival"]) < 1e-12
    assert abs(rates["end_to_end_yield"] - ex["end_to_end_yield"]) < 1e-12

    un = g["unconstrained_contrast"]
    r = oracle.verify(_greedy_counter_batch(0, 120, 80, seed=1), **kw)
    assert [int(c) for c in r.counters] == [un["R"], un["I"], un["D"], un["A"]], r.counters
    assert abs(metrics.acceptance_rates(r.counters)["conditional_acceptance"] - un["conditional_acceptance"]) < 1e-12

    sc = g["second_contrast"]
    r2 = oracle.verify(_greedy_counter_batch(0, 150, 50, seed=2), **kw)
    assert [int(c) for c in r2.counters] == [sc["R"], sc["I"], sc["D"], sc["A"]], r2.counters
    assert abs(metrics.acceptance_rates(r2.counters)["conditional_acceptance"] - sc["conditional_acceptance"]) < 1e-12
    assert int(r2.counters[3]) - ex["A"] == sc["extra_accepted_vs_worked_example"]

    ml = g["mean_acceptance_length"]
    # 100 verification steps (requests), 60 of them accept all 3 drafts: 180 accepted drafts
    r3 = oracle.verify(_greedy_counter_batch(0, 60, 40, k=3, seed=3), **kw)
    assert int(r3.counters[3]) == ml["accepted"]
    assert abs(metrics.mean_acceptance_length(int(r3.counters[3]), ml["steps"]) - ml["value"]) < 1e-12
    assert (r3.out_num_accepted >= 0).all() and r3.out_num_accepted.sum() == ml["accepted"]


# ---------------------------------------------------------------------------------------------
# p == q accepts every draft (min(1, p/q) = 1)
# ---------------------------------------------------------------------------------------------

def check_p_equals_q_accepts_all(lib_path=None, B=300, V=64, k=4, seed=5):
    kw = {} if lib_path is None else {"lib_path": lib_path}
    rng = np.random.default_rng(seed)
    ks = [k] * B
    T = B * (k + 1)
    # exact case: constant logits on 2^m allowed ids -> p = 2^-m exactly, q = p exactly
    allowed = np.zeros((T, V), dtype=bool)
    for t in range(T):
        allowed[t, rng.choice(V, size=2 ** int(rng.integers(0, 6)), replace=False)] = True
    logits = np.repeat(rng.normal(0, 3, size=(T, 1)), V, axis=1).astype(np.float32)
    cu = np.arange(B + 1) * k
    drafts = np.zeros(B * k, dtype=np.int32)
    q = np.zeros((B * k, V), dtype=np.float32)
    for b in range(B):
        for j in range(k):
            t = rows_of(cu, b, j)
            ids = np.flatnonzero(allowed[t])
            q[b * k + j, ids] = 1.0 / ids.size
            drafts[b * k + j] = rng.choice(ids)
    temps = rng.uniform(0.3, 2.0, size=B).astype(np.float32)
    w = batch(V=V, ks=ks, logits=logits, draft_ids=drafts, temperature=temps, q=q, allowed=allowed,
              seed=seed)
    w.uniforms[:] = np.float32(1.0 - 2.0 ** -24)   # the largest draw the generator can make
    r = oracle.verify(w, **kw)
    assert (r.out_num_accepted == k).all(), r.out_num_accepted
    assert np.all(r.alpha == 1.0)

    # general case: q = p from a library softmax, stored in fp32 -> alpha within fp32 rounding of 1
    logits = rng.normal(0, 2, size=(T, V)).astype(np.float32)
    q = np.zeros((B * k, V), dtype=np.float32)
    for b in range(B):
        for j in range(k):
            t = rows_of(cu, b, j)
            p = special.softmax(logits[t].astype(np.float64) / float(temps[b]))
            q[b * k + j] = p.astype(np.float32)
            drafts[b * k + j] = rng.choice(V, p=p)
    w = batch(V=V, ks=ks, logits=logits, draft_ids=drafts, temperature=temps, q=q, seed=seed + 1)
    r = oracle.verify(w, **kw)
    assert np.all(r.alpha[~np.isnan(r.alpha)] >= 1.0 - 1e-6), np.nanmin(r.alpha)
    for b in range(B):
        rows = [rows_of(cu, b, j) for j in range(k)]
        if (w.uniforms[rows] < 1.0 - 1e-6).all():    # outside the 1e-6 band below alpha
            assert r.out_num_accepted[b] == k, (b, r.out_num_accepted[b])


# ---------------------------------------------------------------------------------------------
# greedy: brute force on tiny vocabularies (numpy argmax picks the first maximum)
# ---------------------------------------------------------------------------------------------

def _greedy_expect(w):
    B, V = w.B, w.V
    cu = w.cu_num_draft
    z_all = w.logits_f32().astype(np.float64)
    allowed_all = (np.ones((w.T, V), dtype=bool) if w.bitmask is None
                   else W.unpack_mask_rows(w.bitmask, V))
    tokens = np.full(w.T, -1, dtype=np.int32)
    acc = np.zeros(B, dtype=np.int32)
    ctr = np.zeros(4, dtype=np.int64)
    for b in range(B):
        k = int(cu[b + 1] - cu[b])
        g = k
        for j in range(k):
            x = int(w.draft_ids[cu[b] + j])
            if not (0 <= x < V and allowed_all[rows_of(cu, b, j), x]):
                g = j
                break
        a = k
        for j in range(k + 1):
            t = rows_of(cu, b, j)
            zz = np.where(allowed_all[t], z_all[t], -np.inf)
            if not np.isfinite(zz).any():
                tokens[t] = -1
                a = j
                break
            y = int(np.argmax(zz))
            if j == k:
                tokens[t] = y
                break
            x = int(w.draft_ids[cu[b] + j])
            if j < g and x == y:
                tokens[t] = x
                continue
            tokens[t] = y
            a = j
            break
        acc[b] = a
        ctr += [k, k - g, g, a]
    return tokens, acc, ctr


def check_greedy_brute_force(lib_path=None, cases=60, seed=11):
    kw = {} if lib_path is None else {"lib_path": lib_path}
    rng = np.random.default_rng(seed)
    for case in range(cases):
        V = int(rng.integers(1, 17))
        B = int(rng.integers(1, 12))
        ks = rng.integers(0, 5, size=B)
        T = int(ks.sum()) + B
        # small integer logits: ties are frequent, which exercises the lowest-index rule
        logits = rng.integers(-3, 4, size=(T, V)).astype(np.float32)
        allowed = rng.random((T, V)) < 0.75
        allowed[rng.random(T) < 0.05] = False            # a few empty rows
        cu = np.concatenate([[0], np.cumsum(ks)])
        drafts = []
        for b in range(B):
            for j in range(int(ks[b])):
                t = rows_of(cu, b, j)
                zz = np.where(allowed[t], logits[t], -np.inf)
                if rng.random() < 0.7 and np.isfinite(zz).any():
                    drafts.append(int(np.argmax(zz)))
                else:
                    drafts.append(int(rng.integers(0, V)))
        dtype = W.BF16 if case % 3 == 0 else W.F32
        w = batch(V=V, ks=ks, logits=logits, draft_ids=drafts, temperature=0.0,
                  allowed=allowed if case % 4 else None, seed=case, dtype=dtype, max_k=4)
        r = oracle.verify(w, **kw)
        tokens, acc, ctr = _greedy_expect(w)
        assert np.array_equal(r.out_tokens, tokens), (case, r.out_tokens, tokens)
        assert np.array_equal(r.out_num_accepted, acc), (case, r.out_num_accepted, acc)
        assert [int(c) for c in r.counters] == [int(c) for c in ctr], (case, r.counters, ctr)


# ---------------------------------------------------------------------------------------------
# grammar invariants: no accepted draft and no emitted token is ever disallowed
# ---------------------------------------------------------------------------------------------

def check_grammar_invariants(lib_path=None, seed=21):
    kw = {} if lib_path is None else {"lib_path": lib_path}
    for i, (qm, temp) in enumerate([("all", 0.9), ("none", 1.3), ("half", "half_greedy(0.5,1.2)")]):
        w = W.make_batch(seed + i, B=40, V=300, k=(0, 6), logit_sigma=3.0, temperature=temp, q_mode=qm,
                         draft_sigma=0.7, mask="all", mask_density=0.2, mask_run_len=8,
                         forced_invalid_frac=0.2)
        r = oracle.verify(w, **kw)
        allowed = W.unpack_mask_rows(w.bitmask, w.V)
        cu = w.cu_num_draft
        n_inval = 0
        for b in range(w.B):
            k = int(cu[b + 1] - cu[b])
            a = int(r.out_num_accepted[b])
            for j in range(k):
                x = int(w.draft_ids[cu[b] + j])
                if not allowed[rows_of(cu, b, j), x]:
                    n_inval += k - j
                    break
            for j in range(a):
                t = rows_of(cu, b, j)
                assert allowed[t, r.out_tokens[t]], (b, j)
                assert r.out_tokens[t] == w.draft_ids[cu[b] + j]
            t = rows_of(cu, b, a)
            y = int(r.out_tokens[t])
            if y >= 0:
                assert allowed[t, y], (b, a, y)
            else:
                assert r.status[b] & oracle.ST_EMPTY_MASK_ROW
            for j in range(a + 1, k + 1):
                assert r.out_tokens[rows_of(cu, b, j)] == -1
        R, I, D, A = (int(c) for c in r.counters)
        assert R == w.N and I == n_inval and D == R - I and A <= D


# ---------------------------------------------------------------------------------------------
# losslessness: the first emitted token is distributed as the target p (chi-square, V = 8)
# ---------------------------------------------------------------------------------------------

def _chi2(counts, p):
    n = counts.sum()
    nz = p > 0
    assert counts[~nz].sum() == 0, "a token with target probability 0 was emitted"
    e = n * p[nz]
    return float(((counts[nz] - e) ** 2 / e).sum()), int(nz.sum()) - 1


def _chi2_batch(n, z_rows, temps, mode, q_rows=None, x_fixed=None, allowed_rows=None, seed=0):
    """n independent requests that share the same k rows of logits (z_rows [k+1, V])."""
    k = z_rows.shape[0] - 1
    V = z_rows.shape[1]
    rng = np.random.default_rng([seed, 99])
    cu = (np.arange(n + 1) * k).astype(np.int32)
    T = n * (k + 1)
    logits = np.tile(z_rows.astype(np.float32), (n, 1))
    if mode == "q":
        drafts = np.stack([rng.choice(V, size=n, p=q_rows[j].astype(np.float64) / q_rows[j].astype(np.float64).sum())
                           for j in range(k)], axis=1).reshape(-1) if k else np.zeros(0, np.int64)
        q = np.tile(q_rows.astype(np.float32), (n, 1)) if k else None
    else:
        drafts = np.tile(np.asarray(x_fixed, dtype=np.int64), n) if k else np.zeros(0, np.int64)
        q = None
    bitmask = None
    if allowed_rows is not None:
        bitmask = np.tile(W.pack_mask_rows(allowed_rows), (n, 1))
    wl = W.Workload(
        name="chi2", B=n, V=V, max_k=k, logits_dtype=W.F32, logits=np.ascontiguousarray(logits),
        draft_ids=drafts.astype(np.int32), draft_probs=q, has_q=None, cu_num_draft=cu,
        bitmask=bitmask, temperature=np.full(n, temps, dtype=np.float32),
        uniforms=W.uniforms_from_bits(rng.integers(0, 2 ** 32, size=T, dtype=np.uint32)),
        exp_noise=W.exp1_from_bits(rng.integers(0, 2 ** 32, size=(T, V), dtype=np.uint32)))
    return wl


def _target_p(z, T, allowed=None):
    s = z.astype(np.float64) / T
    if allowed is not None:
        s = np.where(allowed, s, -np.inf)
    return special.softmax(s)


def check_chi_square(lib_path=None, n=1_000_000, seed=31):
    kw = {} if lib_path is None else {"lib_path": lib_path}
    V = 8
    rng = np.random.default_rng(seed)
    z0 = np.array([1.5, -0.5, 0.3, 2.2, -1.0, 0.0, 1.1, -2.0])
    z1 = np.array([-0.2, 0.9, 1.7, -1.3, 0.4, 2.0, -0.7, 0.1])
    q0 = np.array([0.05, 0.20, 0.10, 0.05, 0.25, 0.05, 0.10, 0.20])
    q1 = np.array([0.30, 0.02, 0.08, 0.20, 0.10, 0.05, 0.15, 0.10])
    results = {}

    # (1) draft model, k = 1, T = 1
    w = _chi2_batch(n, np.stack([z0, z1]), 1.0, "q", q_rows=q0[None, :], seed=seed)
    r = oracle.verify(w, **kw)
    first = r.out_tokens[0::2]
    results["draft_model_T1"] = _chi2(np.bincount(first, minlength=V), _target_p(z0, 1.0))

    # (2) draft model, k = 1, T = 0.7, grammar mask forbidding ids 1 and 5 (q still puts mass there)
    allow = np.ones(V, dtype=bool)
    allow[[1, 5]] = False
    w = _chi2_batch(n, np.stack([z0, z1]), 0.7, "q", q_rows=q0[None, :],
                    allowed_rows=np.stack([allow, allow]), seed=seed + 1)
    r = oracle.verify(w, **kw)
    results["draft_model_T0.7_masked"] = _chi2(np.bincount(r.out_tokens[0::2], minlength=V),
                                               _target_p(z0, 0.7, allow))

    # (3) model-free draft (one-hot q at x = 3), k = 1
    w = _chi2_batch(n, np.stack([z0, z1]), 1.0, "mf", x_fixed=[3], seed=seed + 2)
    r = oracle.verify(w, **kw)
    results["model_free"] = _chi2(np.bincount(r.out_tokens[0::2], minlength=V), _target_p(z0, 1.0))

    # (4) bonus only, k = 0: textbook categorical sampling from p
    w = _chi2_batch(n, z1[None, :], 1.3, "mf", x_fixed=[], seed=seed + 3)
    r = oracle.verify(w, **kw)
    results["bonus_only"] = _chi2(np.bincount(r.out_tokens, minlength=V), _target_p(z1, 1.3))

    # (5) second position given the first draft was accepted, k = 2, draft model
    w = _chi2_batch(n, np.stack([z0, z1, z0]), 1.0, "q", q_rows=np.stack([q0, q1]), seed=seed + 4)
    r = oracle.verify(w, **kw)
    acc1 = r.out_num_accepted >= 1
    second = r.out_tokens[1::3][acc1]
    results["second_position"] = _chi2(np.bincount(second, minlength=V), _target_p(z1, 1.0))

    bad = {name: v for name, v in results.items() if not v[0] < stats.chi2.ppf(0.999, v[1])}
    assert not bad, f"chi-square failures: {bad} (all: {results})"
    return results


# ---------------------------------------------------------------------------------------------
# softmax: the oracle's row statistics and p(x) match a library fp64 softmax
# ---------------------------------------------------------------------------------------------

def check_softmax_matches_library(lib_path=None, seed=41):
    kw = {} if lib_path is None else {"lib_path": lib_path}
    rng = np.random.default_rng(seed)
    B, V = 40, 1000
    ks = [1] * B
    T = 2 * B
    logits = (rng.normal(0, 3, size=(T, V))).astype(np.float32)
    temps = rng.uniform(0.2, 2.5, size=B).astype(np.float32)
    drafts = rng.integers(0, V, size=B)
    w = batch(V=V, ks=ks, logits=logits, draft_ids=drafts, temperature=temps, seed=seed)
    w.uniforms[:] = np.float32(1.0 - 2.0 ** -24)  # reject: both rows of each request are read
    r = oracle.verify(w, **kw)
    for b in range(B):
        t = 2 * b
        s = logits[t].astype(np.float64) / float(temps[b])
        lse = special.logsumexp(s)
        m = s.max()
        assert r.row_m[t] == m
        assert abs(r.row_S[t] - np.exp(lse - m)) <= 1e-12 * np.exp(lse - m)
        px = special.softmax(s)[drafts[b]]
        assert abs(r.alpha[b] - px) <= 1e-12 * px, (b, r.alpha[b], px)


# ---------------------------------------------------------------------------------------------
# strict comparison u < alpha, and the degenerate cases the method has
# ---------------------------------------------------------------------------------------------

def check_strict_accept_comparison(lib_path=None):
    kw = {} if lib_path is None else {"lib_path": lib_path}
    # V = 2 with equal logits: p(x) = 1/2 exactly; model-free alpha = p(x) = 1/2
    V = 2
    logits = np.zeros((4, V), dtype=np.float32)
    w = batch(V=V, ks=[1, 1], logits=logits, draft_ids=[0, 0], temperature=1.0)
    w.uniforms[[0, 2]] = [np.float32(0.5 - 2.0 ** -24), np.float32(0.5)]
    r = oracle.verify(w, **kw)
    assert r.alpha[0] == 0.5 and r.alpha[1] == 0.5
    assert list(r.out_num_accepted) == [1, 0]
    assert r.out_tokens[2] == 1          # the residual of a one-hot draft is p without x
    # a grammar-invalid draft is rejected even with the smallest draw u = 0
    allowed = np.ones((2, V), dtype=bool)
    allowed[0, 1] = False
    q = np.array([[0.5, 0.5]], dtype=np.float32)
    w = batch(V=V, ks=[1], logits=np.zeros((2, V)), draft_ids=[1], temperature=1.0, q=q, allowed=allowed)
    w.uniforms[:] = 0.0
    r = oracle.verify(w, **kw)
    assert r.out_num_accepted[0] == 0 and r.alpha[0] == 0.0 and r.out_tokens[0] == 0
    assert [int(c) for c in r.counters] == [1, 1, 0, 0]


def check_edge_cases(lib_path=None):
    kw = {} if lib_path is None else {"lib_path": lib_path}
    V = 8
    rng = np.random.default_rng(51)
    # B = 0: nothing happens
    w = batch(V=V, ks=[], logits=np.zeros((0, V)), draft_ids=[], temperature=[])
    w.max_k = 0
    r = oracle.verify(w, **kw)
    assert [int(c) for c in r.counters] == [0, 0, 0, 0]

    # k = 0 for every request: bonus rows only (greedy: argmax)
    z = rng.normal(0, 1, size=(3, V)).astype(np.float32)
    w = batch(V=V, ks=[0, 0, 0], logits=z, draft_ids=[], temperature=0.0, max_k=0)
    r = oracle.verify(w, **kw)
    assert list(r.out_tokens) == [int(np.argmax(z[i])) for i in range(3)]
    assert list(r.out_num_accepted) == [0, 0, 0] and [int(c) for c in r.counters] == [0, 0, 0, 0]

    # an empty mask row in the middle stops the request with -1 and a status bit
    z = np.tile(np.arange(V, dtype=np.float32), (4, 1))       # argmax = V - 1 everywhere
    allowed = np.ones((4, V), dtype=bool)
    allowed[1] = False
    w = batch(V=V, ks=[3], logits=z, draft_ids=[V - 1, V - 1, V - 1], temperature=0.0, allowed=allowed)
    r = oracle.verify(w, **kw)
    assert list(r.out_tokens) == [V - 1, -1, -1, -1] and r.out_num_accepted[0] == 1
    assert r.status[0] == oracle.ST_EMPTY_MASK_ROW
    # the draft at the empty row is grammar-invalid: I counts it and the rest
    assert [int(c) for c in r.counters] == [3, 2, 1, 1]

    # draft id out of range: flagged, counted invalid, never accepted
    w = batch(V=V, ks=[2], logits=z[:3], draft_ids=[V - 1, V], temperature=0.0)
    r = oracle.verify(w, **kw)
    assert r.status[0] == oracle.ST_BAD_DRAFT_ID and r.out_num_accepted[0] == 1
    assert list(r.out_tokens) == [V - 1, V - 1, -1] and [int(c) for c in r.counters] == [2, 1, 1, 1]

    # temperatures that are not 0 and not positive normal floats: flagged, verified greedily
    for bad in (-1.0, float("nan"), float("inf"), 1e-40):
        zz = rng.normal(0, 1, size=(2, V)).astype(np.float32)
        y = int(np.argmax(zz[0]))
        w = batch(V=V, ks=[1], logits=zz, draft_ids=[y], temperature=bad)
        w.uniforms[:] = np.float32(1.0 - 2.0 ** -24)
        r = oracle.verify(w, **kw)
        assert r.status[0] == oracle.ST_BAD_TEMPERATURE, bad
        assert r.out_num_accepted[0] == 1 and r.out_tokens[1] == int(np.argmax(zz[1]))

    # k_b > max_k: request skipped, -1 everywhere, counters untouched
    w = batch(V=V, ks=[1, 3], logits=rng.normal(size=(6, V)), draft_ids=[0, 1, 2, 3], temperature=0.0,
              max_k=2)
    r = oracle.verify(w, **kw)
    assert r.status[1] == oracle.ST_K_TOO_LARGE and list(r.out_tokens[2:]) == [-1, -1, -1, -1]
    assert int(r.counters[0]) == 1

    # decreasing offsets: request skipped
    w = batch(V=V, ks=[2, 1], logits=rng.normal(size=(5, V)), draft_ids=[0, 1, 2], temperature=0.0)
    w.cu_num_draft[:] = [0, 3, 3]            # request 0 claims 3 drafts, request 1 none
    w.cu_num_draft[1] = 4                    # request 0 ends past cu[B]
    r = oracle.verify(w, **kw)
    assert r.status[0] == oracle.ST_BAD_OFFSETS and r.status[1] == oracle.ST_BAD_OFFSETS

    # -inf logits are never emitted (they have probability 0), greedy or random
    zz = np.full((2, V), -np.inf, dtype=np.float32)
    zz[:, 5] = 0.0
    for temp in (0.0, 1.0):
        w = batch(V=V, ks=[1], logits=zz, draft_ids=[2], temperature=temp)
        r = oracle.verify(w, **kw)
        assert r.out_num_accepted[0] == 0 and r.out_tokens[0] == 5

    # bits at or above V in a mask word are ignored
    V = 37
    zz = rng.normal(size=(4, V)).astype(np.float32)
    allowed = rng.random((4, V)) < 0.6
    allowed[:, 0] = True
    w1 = batch(V=V, ks=[3], logits=zz, draft_ids=[0, 1, 2], temperature=0.9, allowed=allowed, seed=3)
    bm = w1.bitmask.copy()
    bm[:, -1] |= np.int32(-1 << (V % 32))     # set every padding bit of the last word
    w2 = batch(V=V, ks=[3], logits=zz, draft_ids=[0, 1, 2], temperature=0.9, bitmask=bm, seed=3)
    r1, r2 = oracle.verify(w1, **kw), oracle.verify(w2, **kw)
    assert np.array_equal(r1.out_tokens, r2.out_tokens)


def check_residual_excludes_draft(lib_path=None, seed=61):
    """A rejected one-hot draft is never re-emitted at its own position (the residual is p
    with x removed); a rejected draft-model position emits a token with p_i > q_i."""
    kw = {} if lib_path is None else {"lib_path": lib_path}
    for qm in ("none", "all"):
        w = W.make_batch(seed, B=300, V=50, k=(1, 4), logit_sigma=1.0, temperature=1.0, q_mode=qm,
                         draft_sigma=1.0, mf_argmax_frac=0.9)
        r = oracle.verify(w, **kw)
        cu = w.cu_num_draft
        z = w.logits_f32().astype(np.float64)
        n_checked = 0
        for b in range(w.B):
            k = int(cu[b + 1] - cu[b])
            a = int(r.out_num_accepted[b])
            if a == k:
                continue
            t = rows_of(cu, b, a)
            y = int(r.out_tokens[t])
            x = int(w.draft_ids[cu[b] + a])
            if qm == "none":
                assert y != x, (b, a)
            else:
                p = special.softmax(z[t] / float(w.temperature[b]))
                assert p[y] > w.draft_probs[cu[b] + a, y], (b, a)
            n_checked += 1
        assert n_checked > 50


# ---------------------------------------------------------------------------------------------
# per-position telemetry ("vLLM tour part 2", section "Telemetry and tuning"; "5.2 Draft models
# and model-free methods", section 7.2: a position counts drafts accepted all the way through it)
# ---------------------------------------------------------------------------------------------

def _telemetry_expect(entry, k):
    t = np.zeros((4, 33), dtype=np.uint64)
    t[0, :k] = entry["drafts_by_position"]
    t[1, :k] = entry["eligible_by_position"]
    t[2, :k] = entry["accepted_through_position"]
    for a, n in entry["accepted_length_histogram"].items():
        t[3, int(a)] = n
    return t


def check_telemetry(lib_path=None, seed=71):
    kw = {} if lib_path is None else {"lib_path": lib_path}
    g = _golden("telemetry_worked_example.json")
    r = oracle.verify(_greedy_counter_batch(40, 120, 40), **kw)
    assert np.array_equal(r.telemetry, _telemetry_expect(g["worked_example"], 5)), r.telemetry[:, :6]
    r3 = oracle.verify(_greedy_counter_batch(0, 60, 40, k=3, seed=3), **kw)
    assert np.array_equal(r3.telemetry, _telemetry_expect(g["mean_acceptance_length_example"], 3)), r3.telemetry[:, :4]
    # identities with the counters on mixed batches (every mode, masks, forced-invalid drafts,
    # a request with k > max_k that is skipped)
    for s in range(3):
        w = W.make_batch(seed + s, B=60, V=300, k=(0, 7), logit_sigma=2.0, temperature="half_greedy(0.5,1.2)",
                         q_mode="half", draft_sigma=0.3, mf_argmax_frac=0.5, mask="half", mask_density=0.2,
                         mask_run_len=8, forced_invalid_frac=0.2)
        if s == 2:
            w = dataclasses.replace(w, max_k=int(w.k.max()) - 1)       # the longest requests are skipped
        r = oracle.verify(w, **kw)
        tm = r.telemetry.astype(np.int64)
        R, I, D, A = (int(c) for c in r.counters)
        assert tm[0].sum() == R and tm[1].sum() == D and tm[2].sum() == A, (tm.sum(axis=1), r.counters)
        done = (r.status & 24) == 0
        assert tm[3].sum() == int(done.sum())
        assert int((np.arange(33) * tm[3]).sum()) == A
        assert (tm[2] <= tm[1]).all() and (tm[1] <= tm[0]).all()
        assert (np.diff(tm[:3], axis=1) <= 0).all()                    # non-increasing by position
        kk = w.k[done]
        assert tm[0].tolist() == [int((kk > j).sum()) for j in range(33)]
        if s == 2:
            assert not done.all()


# ---------------------------------------------------------------------------------------------
# n-gram proposer ("5.2 Draft models and model-free methods", sections 4.1 and 6)
# ---------------------------------------------------------------------------------------------

def _ngram_check_one(h, min_n, max_n, k, drafts, num, match):
    """The proposal against numpy sliding windows: the window is the longest length in
    [min_n, min(max_n, L - 1)] whose last-n tail occurs earlier, at its earliest start."""
    h = np.asarray(h, dtype=np.int64)
    L = h.size
    cap = min(max_n, L - 1)
    best = None
    for n in range(cap, min_n - 1, -1):
        if n < 1 or L - n < 1:
            continue
        win = np.lib.stride_tricks.sliding_window_view(h[: L - 1], n)     # windows starting at 0 .. L-n-1
        eq = np.flatnonzero((win == h[L - n:]).all(axis=1))
        if eq.size:
            best = (n, int(eq[0]))
            break
    if best is None:
        assert match == 0 and num == 0 and (np.asarray(drafts) == -1).all(), (h, match, num, drafts)
        return False
    n, start = best
    want = h[start + n: start + n + k]
    assert match == n and num == want.size, (h.tolist(), n, start, match, num)
    assert np.array_equal(np.asarray(drafts[:num]), want) and (np.asarray(drafts[num:]) == -1).all()
    return True


def check_ngram_proposer(lib_path=None, seed=81):
    kw = {} if lib_path is None else {"lib_path": lib_path}
    g = _golden("ngram_worked_example.json")
    for c in g["cases"]:
        d, num, match = oracle.ngram_propose([c["history"]], min_n=c["min_n"], max_n=c["max_n"], k=c["k"], **kw)
        want_match = 0 if c["match"] is None else c["match"]
        assert int(match[0]) == want_match and d[0, : int(num[0])].tolist() == c["drafts"], (c["name"], d, num, match)
    # random histories over a small vocabulary (plenty of repeats), every parameter combination
    rng = np.random.default_rng(seed)
    hits = 0
    for _ in range(400):
        L = int(rng.integers(0, 40))
        h = rng.integers(0, int(rng.integers(2, 6)), size=L).tolist()
        min_n = int(rng.integers(1, 5))
        max_n = int(rng.integers(min_n - 1, 7))
        k = int(rng.integers(0, 6))
        d, num, match = oracle.ngram_propose([h], min_n=min_n, max_n=max_n, k=k, **kw)
        hits += _ngram_check_one(h, min_n, max_n, k, d[0], int(num[0]), int(match[0]))
    assert hits > 100
    # a batch gives the same answers as one request at a time
    hs = [rng.integers(0, 4, size=int(rng.integers(0, 30))).tolist() for _ in range(50)]
    d, num, match = oracle.ngram_propose(hs, min_n=2, max_n=5, k=4, **kw)
    for b, h in enumerate(hs):
        d1, n1, m1 = oracle.ngram_propose([h], min_n=2, max_n=5, k=4, **kw)
        assert np.array_equal(d[b], d1[0]) and num[b] == n1[0] and match[b] == m1[0]


# ---------------------------------------------------------------------------------------------
# bitmask scatter ("vLLM tour part 2", section "Grammar gates: structured output")
# ---------------------------------------------------------------------------------------------

def _rows(cu, b):
    return np.arange(int(cu[b]) + b, int(cu[b + 1]) + b + 1)


def check_bitmask_scatter(seed=91):
    """Round trip: compacting a batch-order mask with numpy fancy indexing (constrained requests in
    a random scheduler order) and scattering it back gives the mask on the constrained rows and
    all-ones elsewhere; identity and empty cases; the readings for malformed lists."""
    from oracle import bitmask_ref

    rng = np.random.default_rng(seed)
    for trial in range(30):
        B = int(rng.integers(1, 40))
        V = int(rng.integers(1, 200))
        W = (V + 31) // 32
        ks = rng.integers(0, 6, size=B)
        cu = np.zeros(B + 1, dtype=np.int32)
        cu[1:] = np.cumsum(ks)
        T = int(cu[B]) + B
        full = rng.integers(-2 ** 31, 2 ** 31, size=(T, W), dtype=np.int64).astype(np.int32)
        order = rng.permutation(B)[: int(rng.integers(0, B + 1))]
        rows = np.concatenate([_rows(cu, b) for b in order]) if order.size else np.zeros(0, dtype=np.int64)
        compact = full[rows]
        out = bitmask_ref.bitmask_scatter(compact, order, cu, B, V)
        want = np.full((T, W), -1, dtype=np.int32)
        for b in order:
            want[_rows(cu, b)] = full[_rows(cu, b)]
        assert np.array_equal(out, want), trial
        # every request constrained, in batch order: the identity
        assert np.array_equal(bitmask_ref.bitmask_scatter(full, np.arange(B), cu, B, V), full)
        # nothing constrained: all ones
        assert (bitmask_ref.bitmask_scatter(full[:0], [], cu, B, V) == -1).all()
    # malformed lists: an out-of-range id owns no rows; a repeat keeps its first rows; rows past the
    # end of the compact array allow nothing
    cu = np.array([0, 1, 3], dtype=np.int32)                      # request 0: 2 rows, request 1: 3 rows
    comp = np.arange(10, dtype=np.int32).reshape(-1, 1) + 100     # 10 rows of one word (V <= 32)
    out = bitmask_ref.bitmask_scatter(comp, [7, 1, -3, 1, 0], cu, 2, 20)
    assert out[:, 0].tolist() == [106, 107, 100, 101, 102]        # request 0 after 1's two listings
    out = bitmask_ref.bitmask_scatter(comp[:4], [1, 0], cu, 2, 20)
    assert out[:, 0].tolist() == [103, 0, 100, 101, 102]          # request 0's second row is past the end
    cu_bad = np.array([0, 3, 2, 4], dtype=np.int32)               # request 1 has decreasing offsets:
    out = bitmask_ref.bitmask_scatter(comp, [1, 0, 2], cu_bad, 3, 20)   # it owns no rows
    assert out[:, 0].tolist() == [100, 101, 102, 103, 104, 105, 106]


# ---------------------------------------------------------------------------------------------
# top-k / top-p on the target distribution ("vLLM tour part 2", section "Verification: rejection
# sampling on the GPU": temperature and top-k/top-p are applied before acceptance)
# ---------------------------------------------------------------------------------------------

def _filtered_p(z, T, k, tp, allowed=None):
    """The filtered target distribution by an all-pairs restatement (numpy broadcasting, no sort):
    top-k keeps ids with at least k-1 ... fewer than k allowed ids strictly above; top-p keeps ids
    whose (top-k renormalised) mass of strictly larger logits is below tp."""
    s = z.astype(np.float64) / T
    if allowed is not None:
        s = np.where(allowed, s, -np.inf)
    live = np.isfinite(s)
    p = np.where(live, np.exp(s - s[live].max()), 0.0)
    p /= p.sum()
    above = (s[None, :] > s[:, None]) & live[None, :]          # above[i, j]: j strictly larger than i
    keep = live.copy()
    if k > 0:
        keep &= above.sum(axis=1) < k                           # fewer than k allowed ids above
    pk = np.where(keep, p, 0.0)
    pk /= pk.sum()
    if tp < 1.0:
        keep &= (above * pk[None, :]).sum(axis=1) < tp
    out = np.where(keep, p, 0.0)
    return out / out.sum()


def check_top_k_top_p(lib_path=None, n=400_000, seed=101):
    kw = {} if lib_path is None else {"lib_path": lib_path}
    rng = np.random.default_rng(seed)
    # (1) acceptance probabilities of single-draft requests against the restatement, V <= 24,
    #     every combination of top-k and top-p, with ties among the logits
    for trial in range(300):
        V = int(rng.integers(2, 25))
        z = rng.integers(-3, 4, size=(2, V)).astype(np.float32) * 0.5        # many ties
        T = float(rng.choice([0.6, 1.0, 1.7]))
        k = int(rng.choice([0, 1, 2, 3, V, V + 5]))
        tp = float(rng.choice([1.0, 0.95, 0.7, 0.4, 1e-4]))
        q = rng.random(V) + 0.05
        q /= q.sum()
        x = int(rng.integers(0, V))
        allowed = rng.random((2, V)) < 0.8
        allowed[:, x] = True
        w = batch(V=V, ks=[1], logits=z, draft_ids=[x], temperature=T, q=q[None, :].astype(np.float32),
                  allowed=allowed, seed=trial)
        w = dataclasses.replace(w, top_k=np.array([k], np.int32), top_p=np.array([tp], np.float32))
        r = oracle.verify(w, **kw)
        pf = _filtered_p(z[0], float(np.float32(T)), k, np.float32(tp), allowed[0])
        qx = float(np.float32(q[x]))
        want = 0.0 if pf[x] == 0 else min(1.0, pf[x] / qx)
        assert abs(r.alpha[0] - want) <= 1e-12 * max(1.0, want), (trial, r.alpha[0], want, k, tp)
    # (2) no filter when k covers every allowed id and top_p = 1: identical outputs
    w0 = W.make_batch(seed, B=40, V=200, k=(0, 4), logit_sigma=2.0, temperature="half_greedy(0.5,1.2)",
                      q_mode="half", draft_sigma=0.4, mask="half", mask_density=0.3, mask_run_len=4)
    r0 = oracle.verify(w0, **kw)
    for tk, tpv in ((200, 1.0), (0, 1.0), (10_000, 1.5)):
        r1 = oracle.verify(dataclasses.replace(w0, top_k=np.full(40, tk, np.int32), top_p=np.full(40, tpv, np.float32)), **kw)
        assert np.array_equal(r1.out_tokens, r0.out_tokens) and np.array_equal(r1.counters, r0.counters)
    # (3) a top_p that is not a number in (0, 1]: flagged, no top-p filter
    for bad in (0.0, -0.5, float("nan")):
        r1 = oracle.verify(dataclasses.replace(w0, top_p=np.full(40, bad, np.float32)), **kw)
        assert ((r1.status & 64) != 0).all()
        assert np.array_equal(r1.out_tokens, r0.out_tokens)
    # (4) losslessness on the filtered distribution: first emitted token ~ p' (chi-square, V = 8)
    V = 8
    z0 = np.array([1.5, -0.5, 0.3, 2.2, -1.0, 0.0, 1.1, -2.0])
    z1 = np.array([-0.2, 0.9, 1.7, -1.3, 0.4, 2.0, -0.7, 0.1])
    q0 = np.array([0.05, 0.20, 0.10, 0.05, 0.25, 0.05, 0.10, 0.20])
    results = {}
    for name, k, tp, mode, zz, T in (("topk3_q", 3, 1.0, "q", np.stack([z0, z1]), 1.0),
                                      ("topp0.7_q", 0, 0.7, "q", np.stack([z0, z1]), 1.0),
                                      ("topk4_topp0.8_model_free", 4, 0.8, "mf", np.stack([z0, z1]), 0.8),
                                      ("topk5_bonus_only", 5, 1.0, "mf", z1[None, :], 1.3)):
        w = _chi2_batch(n, zz, T, mode, q_rows=q0[None, :], x_fixed=[3] if zz.shape[0] > 1 else [], seed=seed + len(results))
        w = dataclasses.replace(w, top_k=np.full(n, k, np.int32), top_p=np.full(n, tp, np.float32))
        r = oracle.verify(w, **kw)
        first = r.out_tokens[0::zz.shape[0]]
        pf = _filtered_p(zz[0], float(np.float32(T)), k, np.float32(tp))
        support = pf > 0
        assert not np.bincount(first, minlength=V)[~support].any()      # nothing outside the kept set
        results[name] = _chi2(np.bincount(first, minlength=V)[support], pf[support])
    bad = {nm: v for nm, v in results.items() if not v[0] < stats.chi2.ppf(0.999, v[1])}
    assert not bad, f"chi-square failures: {bad} (all: {results})"
    return results


ALL_PINS = [
    check_worked_counter_example,
    check_telemetry,
    check_ngram_proposer,
    check_top_k_top_p,
    check_strict_accept_comparison,
    check_edge_cases,
    check_residual_excludes_draft,
    check_p_equals_q_accepts_all,
    check_greedy_brute_force,
    check_grammar_invariants,
    check_softmax_matches_library,
    check_chi_square,
]
