"""The benchmark's byte accounting (the numerators of its roofline and nominal figures) against
counts worked out by hand for a tiny batch (no GPU)."""
import importlib.util
import os

import numpy as np

from speculative_decoding_verification_specdec_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)

B, V = 2, 64                      # W = 2 mask words per row
CU = np.array([0, 2, 3], np.int32)   # k = 2 (request 0), 1 (request 1): N = 3 drafts, T = 5 rows


def _tiny(bitmask=None):
    return W.Workload(
        name="tiny", B=B, V=V, max_k=2, logits_dtype=W.F32, logits=np.zeros((5, V), np.float32),
        draft_ids=np.zeros(3, np.int32), draft_probs=np.full((3, V), 1.0 / V, np.float32),
        has_q=np.array([1, 0], np.uint8), cu_num_draft=CU, bitmask=bitmask,
        temperature=np.array([1.0, 0.0], np.float32),          # request 0 sampled with q, request 1 greedy
        uniforms=np.zeros(5, np.float32), exp_noise=np.ones((5, V), np.float32))


ACC = np.array([1, 1])            # request 0 rejected at row 1 (< k = 2); request 1 accepted all (bonus row 1)
OK = np.zeros(2, np.uint32)


def test_whole_rows():
    ab = bench.algorithmic_bytes(_tiny(), ACC, OK)
    # logits: rows 0..1 of each request, 64 ids x 4 bytes: 4 x 256
    assert ab["logits"] == 1024
    # noise: the stop row of the sampled request only
    assert ab["noise"] == 256
    # q: q(x) of the 2 tested drafts (8) and the whole q row of the rejected draft (256)
    assert ab["q"] == 264
    assert ab["mask"] == 0
    # small: cu 8 + temperature 4 + ids 4k + out_tokens 4(k+1) + accepted 4 per request
    # (36 and 28), plus the uniforms of request 0's 2 tested drafts (8)
    assert ab["small"] == 36 + 8 + 28
    assert ab["total"] == 1024 + 256 + 264 + 72 + 32          # + the four u64 counters
    assert ab["row_total"] == ab["total"]                     # no mask: whole rows are the same


def test_masked_rows_count_sectors():
    mask = np.full((5, 2), -1, np.int32)                     # request 1's rows (3, 4): all ones
    mask[0:3, 0] = (1 << 0) | (1 << 9)                       # request 0's rows (0..2): ids 0, 9 ...
    mask[0:3, 1] = np.int32(-2 ** 31)                        # ... and 63
    ab = bench.algorithmic_bytes(_tiny(mask), ACC, OK)
    # fp32: 8 ids per 32-byte sector; ids 0, 9, 63 lie in sectors 0, 1 and 7: 96 bytes per row
    assert ab["logits"] == 2 * 96 + 2 * 256
    assert ab["mask"] == 2 * 8 + 2 * 8                       # 2 rows x 2 words x 4 bytes, per request
    assert ab["noise"] == 96
    assert ab["q"] == 8 + 96
    assert ab["total"] == (192 + 512) + 32 + 96 + 104 + 72 + 32
    # whole rows: as in the unmasked case plus the mask words
    assert ab["row_total"] == 1648 + 32


def test_sector_bytes_by_element_size():
    allowed = np.zeros(V, bool)
    allowed[[0, 9, 63]] = True
    assert bench._sector_bytes(allowed, 8) == 3 * 32          # fp32: sectors 0, 1, 7
    assert bench._sector_bytes(allowed, 16) == 2 * 32         # bf16: sectors 0 and 3
    ragged = np.zeros(70, bool)
    ragged[69] = True                                          # the padded last sector still counts
    assert bench._sector_bytes(ragged, 8) == 32


def test_skipped_requests_and_nominal_bytes():
    ab = bench.algorithmic_bytes(_tiny(), ACC, np.array([8, 0], np.uint32))   # request 0 refused
    assert ab["total"] == 512 + 28 + 32
    # nominal: the full logits (T V 4), noise (T V 4), draft probs (N V 4) and mask (T W 4) tensors
    assert bench.nominal_bytes(_tiny()) == 5 * 64 * 4 + 5 * 64 * 4 + 3 * 64 * 4
    assert bench.nominal_bytes(_tiny(np.full((5, 2), -1, np.int32))) == 5 * 64 * 4 * 2 + 3 * 64 * 4 + 5 * 2 * 4
