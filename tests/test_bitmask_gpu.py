"""The CUDA bitmask scatter (specdec_bitmask_scatter) against the host definition: random batches
and scheduler orders, malformed lists, and the large mixed batch's own masks; bit-exact."""
import numpy as np
import pytest

from oracle import bitmask_ref
from speculative_decoding_verification_specdec_gb300 import _native, build
from speculative_decoding_verification_specdec_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cuda():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    if build.needs_rebuild():
        build.build_library()
    _native.load()
    torch.cuda.set_device(0)
    return "cuda:0"


def _gpu(compact, constrained, cu, B, V, cuda, poison=77):
    import torch

    W_ = (V + 31) // 32
    T = max(int(cu[B]), 0) + B
    c = torch.from_numpy(np.ascontiguousarray(compact, dtype=np.int32).reshape(-1, W_)).to(cuda)
    ids = torch.from_numpy(np.ascontiguousarray(constrained, dtype=np.int32).reshape(-1)).to(cuda)
    cut = torch.from_numpy(np.ascontiguousarray(cu, dtype=np.int32)).to(cuda)
    out = torch.full((T, W_), poison, dtype=torch.int32, device=cuda)
    _native.bitmask_scatter(c if c.numel() else None, c.shape[0], ids if ids.numel() else None, ids.numel(), cut, B, V, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _rows(cu, b):
    return np.arange(int(cu[b]) + b, int(cu[b + 1]) + b + 1)


@pytest.mark.parametrize("V", [1, 31, 33, 128, 1000, 4096, 32000])
def test_random_batches(cuda, V):
    rng = np.random.default_rng(V)
    for _ in range(6):
        B = int(rng.integers(1, 300))
        ks = rng.integers(0, 9, size=B)
        cu = np.zeros(B + 1, dtype=np.int32)
        cu[1:] = np.cumsum(ks)
        T = int(cu[B]) + B
        Wd = (V + 31) // 32
        full = rng.integers(-2 ** 31, 2 ** 31, size=(T, Wd), dtype=np.int64).astype(np.int32)
        order = rng.permutation(B)[: int(rng.integers(0, B + 1))]
        rows = np.concatenate([_rows(cu, b) for b in order]) if order.size else np.zeros(0, dtype=np.int64)
        compact = full[rows]
        got = _gpu(compact, order, cu, B, V, cuda)
        assert np.array_equal(got, bitmask_ref.bitmask_scatter(compact, order, cu, B, V))


def test_malformed_lists(cuda):
    cu = np.array([0, 1, 3], dtype=np.int32)
    comp = (np.arange(10, dtype=np.int32).reshape(-1, 1) + 100)
    for ids, c in (([7, 1, -3, 1, 0], comp), ([1, 0], comp[:4]), ([], comp[:0]), ([0, 1, 0, 1], comp)):
        got = _gpu(c, ids, cu, 2, 20, cuda)
        assert np.array_equal(got, bitmask_ref.bitmask_scatter(c, ids, cu, 2, 20)), ids
    cu_bad = np.array([0, 3, 2, 4], dtype=np.int32)                    # request 1: decreasing offsets
    got = _gpu(comp, [1, 0, 2], cu_bad, 3, 20, cuda)
    assert got[:, 0].tolist() == [100, 101, 102, 103, 104, 105, 106]


def test_large_mixed_batch_masks(cuda):
    """The large mixed batch (B=1024, V=151936): its masked requests' rows, compacted in a random
    scheduler order, scatter back to exactly the batch's bitmask (unmasked rows are all ones)."""
    w = W.config(4)
    masked = [b for b in range(w.B) if not (w.bitmask[w.row(b, 0)] == -1).all()]
    order = np.random.default_rng(4).permutation(np.asarray(masked, dtype=np.int32))
    rows = np.concatenate([_rows(w.cu_num_draft, b) for b in order])
    got = _gpu(w.bitmask[rows], order, w.cu_num_draft, w.B, w.V, cuda)
    assert np.array_equal(got, w.bitmask)
