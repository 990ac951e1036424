"""The request-sharded verify on the GPU.

One batch is split into contiguous request ranges (`shard.shard_bounds`, balanced by logit rows);
each range is verified by its own call through the C ABI, as each rank of a multi-GPU run does on
its own device; the shards' counters and telemetry are summed and their per-request outputs
concatenated in rank order (`shard.merge_outputs`). The merged result must equal the unsharded
GPU run bit for bit, and the oracle within the parity rules.

The shards run one after another on one GPU. They share nothing and never wait on one another
(requests are independent in the verify step), so each call executes exactly the code a rank
runs; only the exchange after the verify (summing counters, gathering outputs) is left to the
host here, and the gloo test covers it across processes.
"""
import numpy as np
import pytest

import oracle
from oracle import parity
from speculative_decoding_verification_specdec_gb300 import _native, build, device, shard
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


def _sharded(w, world, cuda):
    parts = []
    for b0, b1 in shard.shard_bounds(w.cu_num_draft, world):
        sub = w.subset(range(b0, b1))
        parts.append(device.run(sub, device=cuda, diag=False, telemetry=True))
    return shard.merge_outputs(parts)


def _mixed_batch(B=300):
    return W.make_batch(21, name=f"shard_mixed_B{B}", B=B, V=20000, k=(0, 8), logits_dtype=W.BF16, logit_sigma=3.0,
                        temperature="half_greedy(0.5,1.2)", q_mode="half", draft_sigma=0.5, mf_argmax_frac=0.4,
                        mask="half", mask_density=0.1, mask_run_len=16, forced_invalid_frac=0.2)


@pytest.mark.parametrize("world", [2, 3, 8])
def test_sharded_batch_equals_unsharded(cuda, world):
    w = _mixed_batch()
    whole = device.run(w, device=cuda, diag=False, telemetry=True)
    merged = _sharded(w, world, cuda)
    for key in ("out_tokens", "out_num_accepted", "status", "counters", "telemetry"):
        assert np.array_equal(np.asarray(merged[key], dtype=np.int64), np.asarray(whole[key], dtype=np.int64)), key
    rep = parity.compare(w, merged, oracle.verify(w))
    assert rep.ok, rep.summary()


def test_sharded_large_mixed_batch(cuda):
    """The large mixed batch (B=1024, k 1-8, bf16, V=151936) split over 4 shards: each shard is a
    quarter of the requests, below one wave of CTAs, so it runs unscheduled where the whole batch
    runs scheduled and split; the outputs must not depend on that."""
    w = W.config(4)
    whole = device.run(w, device=cuda, diag=False, telemetry=True)
    merged = _sharded(w, 4, cuda)
    for key in ("out_tokens", "out_num_accepted", "status", "counters", "telemetry"):
        assert np.array_equal(np.asarray(merged[key], dtype=np.int64), np.asarray(whole[key], dtype=np.int64)), key
