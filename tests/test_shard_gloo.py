"""Multi-process (world_size 2, gloo, CPU) check of the request-sharded path: each rank verifies
its contiguous request range, the counters are summed and the outputs gathered; the result equals
the unsharded verify. The per-rank verify here is the CPU oracle (no GPU in these tests)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from speculative_decoding_verification_specdec_gb300 import shard
from speculative_decoding_verification_specdec_gb300 import workloads as W


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out_q):
    import torch
    import torch.distributed as dist

    import oracle

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = W.make_batch(9, B=37, V=500, k=(0, 6), logit_sigma=3.0, temperature="half_greedy(0.5,1.2)",
                     q_mode="half", draft_sigma=0.5, mask="half", mask_density=0.2, mask_run_len=8,
                     forced_invalid_frac=0.2)
    b0, b1 = shard.shard_bounds(w.cu_num_draft, world)[rank]
    sub = w.subset(range(b0, b1))
    r = oracle.verify(sub)
    ctr = torch.from_numpy(r.counters.astype(np.int64))
    dist.all_reduce(ctr)                           # the only exchange: after the verify
    toks = [None] * world
    dist.all_gather_object(toks, (r.out_tokens.tolist(), r.out_num_accepted.tolist(), r.status.tolist()))
    # timing reduction used by the benchmark: max over ranks
    t = torch.tensor([float(rank + 1)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    if rank == 0:
        full = oracle.verify(w)
        merged_tokens = sum((x[0] for x in toks), [])
        merged_acc = sum((x[1] for x in toks), [])
        merged_status = sum((x[2] for x in toks), [])
        out_q.put({
            "tokens_equal": merged_tokens == full.out_tokens.tolist(),
            "acc_equal": merged_acc == full.out_num_accepted.tolist(),
            "status_equal": merged_status == full.status.tolist(),
            "counters_equal": ctr.tolist() == [int(c) for c in full.counters],
            "max_time": float(t.item()),
        })
    dist.barrier()
    dist.destroy_process_group()


def test_shard_bounds_cover_and_balance():
    cu = np.concatenate([[0], np.cumsum(np.random.default_rng(0).integers(0, 9, size=1000))])
    for world in (1, 2, 3, 8):
        bounds = shard.shard_bounds(cu, world)
        assert bounds[0][0] == 0 and bounds[-1][1] == 1000
        assert all(a[1] == b[0] for a, b in zip(bounds, bounds[1:]))
        rows = [int(cu[b1] - cu[b0] + (b1 - b0)) for b0, b1 in bounds]
        assert max(rows) - min(rows) <= 2 * 9


def test_two_rank_gloo_sharded_verify_matches_unsharded():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = q.get(timeout=180)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res["tokens_equal"] and res["acc_equal"] and res["status_equal"] and res["counters_equal"], res
    assert res["max_time"] == 2.0


def test_merge_outputs_concatenates_in_rank_order_and_sums():
    """The oracle's outputs for three contiguous request ranges, merged, equal its outputs for the
    whole batch: per-row tokens and per-request arrays concatenate, counters and telemetry add up."""
    import oracle

    w = W.make_batch(11, B=23, V=300, k=(0, 5), logit_sigma=2.5, temperature="half_greedy(0.5,1.2)",
                     q_mode="half", draft_sigma=0.5, mask="half", mask_density=0.3, mask_run_len=4)
    parts = []
    for b0, b1 in shard.shard_bounds(w.cu_num_draft, 3):
        r = oracle.verify(w.subset(range(b0, b1)))
        parts.append({"out_tokens": r.out_tokens, "out_num_accepted": r.out_num_accepted, "status": r.status,
                      "counters": r.counters, "telemetry": r.telemetry})
    merged = shard.merge_outputs(parts)
    full = oracle.verify(w)
    assert np.array_equal(merged["out_tokens"], full.out_tokens)
    assert np.array_equal(merged["out_num_accepted"], full.out_num_accepted)
    assert np.array_equal(merged["status"], full.status)
    assert np.array_equal(merged["counters"].astype(np.int64), np.asarray(full.counters, dtype=np.int64))
    assert np.array_equal(merged["telemetry"].astype(np.int64), np.asarray(full.telemetry, dtype=np.int64))
