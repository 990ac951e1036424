"""The CUDA n-gram proposer (specdec_ngram_propose) against the CPU oracle: the pages' printed
examples, random small-vocabulary histories over every parameter combination, and the benchmark's
batch of 1024 long histories; bit-exact (drafts, lengths, window lengths)."""
import json
import os

import numpy as np
import pytest

import oracle
from speculative_decoding_verification_specdec_gb300 import _native, build
from speculative_decoding_verification_specdec_gb300 import workloads as W

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def cuda():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    if build.needs_rebuild():
        build.build_library()
    _native.load()
    torch.cuda.set_device(0)
    return "cuda:0"


def _pack(histories):
    lens = [len(h) for h in histories]
    cu = np.zeros(len(histories) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lens)
    tokens = np.concatenate([np.asarray(h, dtype=np.int32) for h in histories]) if cu[-1] else np.zeros(1, np.int32)
    return tokens, cu


def _gpu(tokens, cu, min_n, max_n, k, cuda):
    import torch

    B = cu.size - 1
    t = torch.from_numpy(np.ascontiguousarray(tokens, dtype=np.int32)).to(cuda)
    c = torch.from_numpy(np.ascontiguousarray(cu, dtype=np.int64)).to(cuda)
    d = torch.full((B, max(k, 1)), -7, dtype=torch.int32, device=cuda)
    n = torch.full((B,), -7, dtype=torch.int32, device=cuda)
    m = torch.full((B,), -7, dtype=torch.int32, device=cuda)
    _native.ngram_propose(t, c, B, min_n, max_n, k, d, n, m)
    torch.cuda.synchronize()
    return d.cpu().numpy()[:, :k], n.cpu().numpy(), m.cpu().numpy()


def _same(got, ref):
    for g, r, name in zip(got, ref, ("drafts", "num", "match")):
        assert np.array_equal(g, r), (name, np.flatnonzero((g != r).reshape(g.shape[0], -1).any(axis=1))[:10])


def test_printed_examples(cuda):
    g = json.load(open(os.path.join(GOLDEN, "ngram_worked_example.json")))
    for c in g["cases"]:
        tokens, cu = _pack([c["history"]])
        d, n, m = _gpu(tokens, cu, c["min_n"], c["max_n"], c["k"], cuda)
        assert int(m[0]) == (c["match"] or 0) and d[0, : int(n[0])].tolist() == c["drafts"], c["name"]


@pytest.mark.parametrize("min_n,max_n,k", [(1, 1, 1), (2, 4, 3), (2, 5, 8), (3, 3, 5), (1, 8, 32), (4, 2, 3),
                                           (2, 64, 4)])
def test_random_small_vocab(cuda, min_n, max_n, k):
    rng = np.random.default_rng(min_n * 100 + max_n * 10 + k)
    hs = [rng.integers(0, int(rng.integers(2, 6)), size=int(rng.integers(0, 300))).tolist() for _ in range(700)]
    hs += [[], [5], [5, 5], [1, 2, 1, 2, 1, 2, 1, 2]]
    tokens, cu = _pack(hs)
    _same(_gpu(tokens, cu, min_n, max_n, k, cuda), oracle.ngram_propose((tokens, cu), min_n=min_n, max_n=max_n, k=k))


def test_long_histories_with_copied_spans(cuda):
    hs = W.ngram_histories(3, B=1024, L=(1024, 8192))
    for (min_n, max_n, k) in ((2, 5, 8), (1, 3, 4), (5, 5, 16)):
        got = _gpu(hs.tokens, hs.cu_hist, min_n, max_n, k, cuda)
        ref = oracle.ngram_propose((hs.tokens, hs.cu_hist), min_n=min_n, max_n=max_n, k=k)
        _same(got, ref)
        assert (ref[2] > 0).mean() > 0.2                      # the batch does have matches


def test_bad_offsets_are_misses(cuda):
    tokens = np.array([1, 2, 1, 2, 1, 2], dtype=np.int32)
    cu = np.array([0, 6, 3, 6], dtype=np.int64)               # request 1 has a decreasing offset
    d, n, m = _gpu(tokens, cu, 1, 4, 3, cuda)
    assert m[1] == 0 and n[1] == 0 and (d[1] == -1).all()
    assert m[0] > 0 and m[2] > 0
