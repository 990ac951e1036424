"""GPU library vs CPU oracle, element by element, through the C ABI (needs a GB300)."""
import dataclasses

import numpy as np
import pytest
from scipy import special, stats

import oracle
from oracle import parity
from speculative_decoding_verification_specdec_gb300 import _native, build, device
from speculative_decoding_verification_specdec_gb300 import workloads as W

from _hand import batch, rows_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session")
def cuda():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    if build.needs_rebuild():
        build.build_library()
    _native.load()
    torch.cuda.set_device(0)
    return "cuda:0"


_MODE = {"workspace": True}


def check_parity(w, cuda, label=""):
    # every output is followed by guard elements; a write past any output's end fails the check
    got = device.run(w, device=cuda, diag=True, workspace=_MODE["workspace"], guard=64)
    ref = oracle.verify(w)
    rep = parity.compare(w, got, ref)
    assert got["guards_intact"], f"{label or w.name}: a write landed past the end of an output"
    assert not (got["status"] & _native.ST_DEVICE_TIMEOUT).any()
    assert rep.ok, (f"{label or w.name}: {rep.summary()} tokens={rep.token_mismatches[:8]} "
                    f"acc={rep.accepted_mismatches[:8]} status={rep.status_mismatches[:8]} "
                    f"alpha={rep.alpha_bad[:5]} rows={rep.row_bad[:5]}")
    return rep, got, ref


KERNELS = ["stream", "stream_index_order", "cluster"]


@pytest.fixture(params=KERNELS)
def kernel(request, launch_options):
    """stream: the streaming kernel with a workspace (requests scheduled heaviest first);
    stream_index_order: the same kernel without one (requests in index order); cluster: the
    slice-resident cluster kernel (scheduled)."""
    launch_options(kernel="cluster" if request.param == "cluster" else "stream")
    launch_options(schedule=request.param != "stream_index_order")
    _MODE["workspace"] = request.param != "stream_index_order"
    yield request.param
    _MODE["workspace"] = True


@pytest.mark.parametrize("cfg", [0, 1, 2, 3])
def test_config_parity(cuda, cfg, kernel):
    w = W.config(cfg)
    rep, got, ref = check_parity(w, cuda)
    print(f"config {cfg} {w.name}: {rep.summary()} counters={list(ref['counters'])}")
    assert rep.excluded_requests <= max(1, w.B // 50)


def test_config4_full_size_parity(cuda, kernel):
    w = W.config(4)
    rep, got, ref = check_parity(w, cuda)
    print(f"config 4 {w.name}: {rep.summary()} counters={list(ref['counters'])}")
    assert rep.excluded_requests <= max(1, w.B // 50)


SWEEP = [
    # V, dtype, B, k range, q_mode, temperature, mask
    (1, W.F32, 9, (0, 3), "none", "half_greedy(0.5,1.2)", "none"),
    (7, W.BF16, 11, (0, 4), "half", 0.9, "all"),
    (37, W.F32, 17, (0, 6), "all", "uniform(0.3,1.5)", "half"),
    (128, W.F32, 13, (1, 5), "half", "half_greedy(0.5,1.2)", "all"),
    (129, W.BF16, 13, (1, 5), "none", 1.0, "half"),
    (1000, W.BF16, 21, (0, 8), "all", "half_greedy(0.5,1.2)", "none"),
    (1001, W.F32, 21, (0, 8), "half", 0.7, "all"),
    (5000, W.F32, 33, (2, 6), "all", "uniform(0.5,1.2)", "half"),
    (12345, W.BF16, 33, (0, 7), "half", "half_greedy(0.5,1.2)", "half"),
    (40000, W.F32, 29, (1, 8), "none", "uniform(0.5,2.0)", "all"),
    (70008, W.BF16, 40, (1, 8), "half", "half_greedy(0.5,1.2)", "half"),
    (131072, W.F32, 24, (3, 6), "all", 0.8, "all"),
    (4100, W.F32, 17, (1, 5), "all", 0.9, "none"),                    # last draw unit: 4 ids
    (8200, W.BF16, 17, (1, 5), "half", "uniform(0.5,1.2)", "none"),   # last draw unit: 8 ids
]


@pytest.mark.parametrize("case", range(len(SWEEP)))
def test_sweep_parity(cuda, case, kernel):
    V, dt, B, kr, qm, temp, mask = SWEEP[case]
    w = W.make_batch(100 + case, name=f"sweep{case}_V{V}", B=B, V=V, k=kr, logits_dtype=dt, logit_sigma=3.0,
                     temperature=temp, q_mode=qm, draft_sigma=0.5, mask=mask, mask_density=0.1,
                     mask_run_len=16 if V > 64 else 2, forced_invalid_frac=0.2, max_k=8)
    check_parity(w, cuda)


@pytest.mark.parametrize("ctas", ["1", "3", "16"])
def test_forced_cluster_shapes(cuda, ctas, launch_options):
    launch_options(kernel="cluster")
    launch_options(ctas_per_request=int(ctas))
    w = W.make_batch(200, name=f"ctas{ctas}", B=20, V=9000, k=(0, 6), logits_dtype=W.F32, logit_sigma=3.0,
                     temperature="half_greedy(0.5,1.2)", q_mode="half", draft_sigma=0.5, mask="half",
                     mask_density=0.1, mask_run_len=16, forced_invalid_frac=0.2)
    check_parity(w, cuda)


def test_edge_cases_match_oracle(cuda, kernel):
    rng = np.random.default_rng(5)
    V = 8
    cases = []
    z = rng.normal(0, 1, size=(3, V)).astype(np.float32)
    cases.append(batch(V=V, ks=[0, 0, 0], logits=z, draft_ids=[], temperature=0.0, max_k=0, name="k0_greedy"))
    cases.append(batch(V=V, ks=[0, 0, 0], logits=z, draft_ids=[], temperature=1.1, max_k=0, name="k0_random"))
    zz = np.tile(np.arange(V, dtype=np.float32), (4, 1))
    allowed = np.ones((4, V), dtype=bool)
    allowed[1] = False
    for temp in (0.0, 0.8):
        cases.append(batch(V=V, ks=[3], logits=zz, draft_ids=[V - 1] * 3, temperature=temp, allowed=allowed,
                           name=f"empty_row_T{temp}"))
        cases.append(batch(V=V, ks=[2], logits=zz[:3], draft_ids=[V - 1, V], temperature=temp, name=f"bad_id_T{temp}"))
        cases.append(batch(V=V, ks=[2], logits=zz[:3], draft_ids=[-5, 1], temperature=temp, name=f"neg_id_T{temp}"))
    for bad in (-1.0, float("nan"), float("inf"), 1e-40):
        cases.append(batch(V=V, ks=[1, 2], logits=rng.normal(size=(5, V)), draft_ids=[1, 2, 3],
                           temperature=[bad, 0.9], name=f"bad_T_{bad}"))
    cases.append(batch(V=V, ks=[1, 3], logits=rng.normal(size=(6, V)), draft_ids=[0, 1, 2, 3], temperature=0.0,
                       max_k=2, name="k_too_large"))
    w = batch(V=V, ks=[2, 1], logits=rng.normal(size=(5, V)), draft_ids=[0, 1, 2], temperature=0.7, name="bad_offsets")
    w.cu_num_draft[:] = [0, 4, 3]
    cases.append(w)
    zi = np.full((2, V), -np.inf, dtype=np.float32)
    zi[:, 5] = 0.0
    for temp in (0.0, 1.0):
        cases.append(batch(V=V, ks=[1], logits=zi, draft_ids=[2], temperature=temp, name=f"neg_inf_T{temp}"))
    # strict u < alpha at alpha = 1/2 exactly (V = 2, equal logits, one-hot draft)
    w = batch(V=2, ks=[1, 1], logits=np.zeros((4, 2)), draft_ids=[0, 0], temperature=1.0, name="strict")
    w.uniforms[[0, 2]] = [np.float32(0.5 - 2.0 ** -24), np.float32(0.5)]
    cases.append(w)
    # grammar-invalid draft with u = 0
    al = np.ones((2, 2), dtype=bool)
    al[0, 1] = False
    w = batch(V=2, ks=[1], logits=np.zeros((2, 2)), draft_ids=[1], temperature=1.0,
              q=np.array([[0.5, 0.5]], dtype=np.float32), allowed=al, name="invalid_u0")
    w.uniforms[:] = 0.0
    cases.append(w)
    # p == q exactly (uniform on 4 allowed ids): every draft accepted at the largest draw
    al = np.zeros((5, 16), dtype=bool)
    al[:, [1, 4, 9, 15]] = True
    q = np.zeros((4, 16), dtype=np.float32)
    q[:, [1, 4, 9, 15]] = 0.25
    w = batch(V=16, ks=[4], logits=np.full((5, 16), 3.0), draft_ids=[4, 9, 1, 15], temperature=0.6, q=q,
              allowed=al, name="p_equals_q")
    w.uniforms[:] = np.float32(1.0 - 2.0 ** -24)
    cases.append(w)
    for w in cases:
        _, got, ref = check_parity(w, cuda, label=w.name)
        if w.name == "p_equals_q":
            assert got["out_num_accepted"][0] == 4
        if w.name == "strict":
            assert list(got["out_num_accepted"]) == [1, 0]


def test_mixed_density_rows(cuda, kernel):
    """Rows of one request with different mask densities (all-ones, 5 %, one id, none) on an aligned
    layout, so that requests run the sparse or dense path and meet rows of the other kind."""
    rng = np.random.default_rng(77)
    V, B = 131072, 12
    ks = [5] * B
    T = 6 * B
    allowed = np.zeros((T, V), dtype=bool)
    kinds = rng.integers(0, 4, size=T)
    for t in range(T):
        if kinds[t] == 0:
            allowed[t] = True
        elif kinds[t] == 1:
            allowed[t, rng.choice(V, size=V // 20, replace=False)] = True
        elif kinds[t] == 2:
            allowed[t, rng.integers(0, V)] = True
    logits = rng.normal(0, 3, size=(T, V)).astype(np.float32)
    drafts = []
    for b in range(B):
        for j in range(5):
            t = 6 * b + j
            ids = np.flatnonzero(allowed[t])
            z = np.where(allowed[t], logits[t], -np.inf)
            drafts.append(int(np.argmax(z)) if ids.size and rng.random() < 0.7 else int(rng.integers(0, V)))
    for dt in (W.F32, W.BF16):
        for temp in (0.0, 0.9):
            w = batch(V=V, ks=ks, logits=logits, draft_ids=drafts, temperature=temp, allowed=allowed, seed=3, dtype=dt,
                      name=f"mixed_{dt}_{temp}")
            check_parity(w, cuda)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_sparse_draft_in_first_group(cuda, kernel, dtype):
    """Sparse rows (few allowed ids) whose draft sits in the row's first 16-byte group, with a
    short list of allowed groups: the draft's logit must survive the unused list slots."""
    V, ks = 512, [2, 2, 2, 2, 1, 1]
    B, N = len(ks), sum(ks)
    T = N + B
    rng = np.random.default_rng(5)
    logits = rng.normal(0.0, 2.0, size=(T, V)).astype(np.float32)
    allowed = np.zeros((T, V), dtype=bool)
    allowed[:, :8] = True
    allowed[:, [100, 201, 333, 511]] = True
    drafts = [1, 5, 3, 0, 7, 2, 6, 4, 1, 3][:N]
    q = rng.random((N, V)).astype(np.float32) + 0.01
    q /= q.sum(axis=1, keepdims=True)
    u = np.full(T, 0.01, dtype=np.float32)
    w = batch(V=V, ks=ks, logits=logits, draft_ids=drafts, temperature=[1.0, 0.8, 0.0, 1.3, 1.0, 0.0],
              q=q, has_q=[1, 0, 1, 0, 1, 0], allowed=allowed, uniforms=u, dtype=dtype, name=f"first_group_{dtype}")
    rep, got, ref = check_parity(w, cuda)
    assert (ref.out_num_accepted > 0).any()          # some drafts are accepted: p(x) was read


def test_rows_after_stop_are_never_read(cuda, kernel):
    """No output depends on a row after a request's stop row: those rows are poisoned with NaN.
    (The streaming kernel may fetch the first two ring chunks of the row after the stop before the
    decision, and discards them; the library's diagnostics report exactly rows 0..a_b as read.)"""
    w = W.make_batch(300, B=40, V=3000, k=(2, 6), logits_dtype=W.F32, logit_sigma=3.0,
                     temperature="half_greedy(0.5,1.2)", q_mode="half", draft_sigma=0.5, mask="half",
                     mask_density=0.2, mask_run_len=16, forced_invalid_frac=0.2)
    ref = oracle.verify(w)
    # logits and noise rows after each stop row are poisoned; mask rows stay (the word holding each
    # draft's bit is read at every position for the grammar-valid prefix behind I and D)
    poisoned = dataclasses.replace(w, logits=w.logits.copy(), exp_noise=w.exp_noise.copy())
    cu = w.cu_num_draft
    n_poisoned = 0
    for b in range(w.B):
        k = int(cu[b + 1] - cu[b])
        for j in range(int(ref["out_num_accepted"][b]) + 1, k + 1):
            t = rows_of(cu, b, j)
            poisoned.logits[t] = np.nan
            poisoned.exp_noise[t] = np.nan
            n_poisoned += 1
    assert n_poisoned > 20
    got = device.run(poisoned, device=cuda, diag=True, workspace=_MODE["workspace"])
    rep = parity.compare(w, got, ref)
    assert rep.ok, rep.summary()
    # the library reports which rows it read: exactly rows 0..a_b of each request
    read = np.isfinite(got["diag_row_stats"][: w.T, 0]) | (got["diag_row_stats"][: w.T, 0] == -np.inf)
    for b in range(w.B):
        k = int(cu[b + 1] - cu[b])
        a = int(ref["out_num_accepted"][b])
        for j in range(k + 1):
            assert read[rows_of(cu, b, j)] == (j <= a), (b, j, a)


def test_counters_accumulate_and_runs_are_deterministic(cuda, kernel):
    import torch

    w = W.make_batch(400, B=64, V=4096, k=(1, 6), logit_sigma=3.0, temperature="half_greedy(0.5,1.2)",
                     q_mode="half", draft_sigma=0.5, mask="half", mask_density=0.1, mask_run_len=16,
                     forced_invalid_frac=0.2)
    dev = device.device_tensors(w, cuda)
    out = device.alloc_outputs(w, cuda, diag=True, workspace=_MODE["workspace"])
    device.verify(w, dev, out)
    torch.cuda.synchronize()
    first = out.numpy()
    device.verify(w, dev, out)
    torch.cuda.synchronize()
    second = out.numpy()
    assert np.array_equal(second["counters"], 2 * first["counters"])
    assert np.array_equal(second["telemetry"], 2 * first["telemetry"])
    tm = first["telemetry"].astype(np.int64)
    assert tm[0].sum() == first["counters"][0] and tm[1].sum() == first["counters"][2]
    assert tm[2].sum() == first["counters"][3]
    for key in ("out_tokens", "out_num_accepted", "status"):
        assert np.array_equal(first[key], second[key])
    assert np.array_equal(first["diag_accept_prob"], second["diag_accept_prob"], equal_nan=True)


def test_runs_on_a_side_stream(cuda):
    import torch

    w = W.make_batch(500, B=16, V=20000, k=(1, 4), logit_sigma=3.0, temperature=0.9, q_mode="all",
                     draft_sigma=0.5)
    dev = device.device_tensors(w, cuda)
    torch.cuda.synchronize()
    out = device.alloc_outputs(w, cuda, diag=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        device.verify(w, dev, out, stream=s)
    _native.specdec_wait(s, timeout_ms=60000)
    got = out.numpy()
    ref = oracle.verify(w)
    assert parity.compare(w, got, ref).ok


def test_chi_square_on_gpu(cuda, kernel):
    """The kernel's first emitted token is distributed as the target p (V = 8, 10^6 requests)."""
    import _pins

    n, V = 1_000_000, 8
    z0 = np.array([1.5, -0.5, 0.3, 2.2, -1.0, 0.0, 1.1, -2.0])
    z1 = np.array([-0.2, 0.9, 1.7, -1.3, 0.4, 2.0, -0.7, 0.1])
    q0 = np.array([0.05, 0.20, 0.10, 0.05, 0.25, 0.05, 0.10, 0.20])
    allow = np.ones(V, dtype=bool)
    allow[[1, 5]] = False
    variants = {
        "draft_model": (_pins._chi2_batch(n, np.stack([z0, z1]), 1.0, "q", q_rows=q0[None, :], seed=71), z0, 1.0, None, 2),
        "draft_model_masked": (_pins._chi2_batch(n, np.stack([z0, z1]), 0.7, "q", q_rows=q0[None, :],
                                                 allowed_rows=np.stack([allow, allow]), seed=72), z0, 0.7, allow, 2),
        "model_free": (_pins._chi2_batch(n, np.stack([z0, z1]), 1.0, "mf", x_fixed=[3], seed=73), z0, 1.0, None, 2),
        "bonus_only": (_pins._chi2_batch(n, z1[None, :], 1.3, "mf", x_fixed=[], seed=74), z1, 1.3, None, 1),
    }
    for name, (w, z, T, al, stride) in variants.items():
        got = device.run(w, device=cuda, diag=False, workspace=_MODE["workspace"])
        first = got["out_tokens"][0::stride]
        p = _pins._target_p(z, T, al)
        chi2, df = _pins._chi2(np.bincount(first, minlength=V), p)
        assert chi2 < stats.chi2.ppf(0.999, df), (name, chi2)
        ref = oracle.verify(w)
        rep = parity.compare(w, got, ref)
        assert rep.ok, (name, rep.summary())


def _schedule(w, cuda):
    """Run one scheduled verify and return (order, keys) read back from the workspace."""
    import torch

    dev = device.device_tensors(w, cuda)
    out = device.alloc_outputs(w, cuda, workspace=True)
    device.verify(w, dev, out)
    torch.cuda.synchronize()
    ws = out.workspace.cpu().numpy()
    order = ws[: 4 * w.B].view(np.int32).copy()
    koff = (4 * w.B + 15) // 16 * 16
    keys = ws[koff: koff + w.B].copy()
    return order, keys, out.numpy()


@pytest.mark.parametrize("B", [1, 37, 1024, 2500])
def test_schedule_is_a_stable_descending_permutation(cuda, B, launch_options):
    """The request order the schedule kernel writes: every request exactly once, cost keys
    non-increasing along it, equal keys in index order (one and several 1024-request tiles)."""
    launch_options(kernel="stream")
    launch_options(schedule=True)        # small batches fit one wave: force it
    w = W.make_batch(23, name=f"sched_B{B}", B=B, V=1024, k=(0, 6), logit_sigma=3.0,
                     temperature="half_greedy(0.5,1.2)", q_mode="half", draft_sigma=0.5,
                     mask="half", mask_density=0.05, mask_run_len=16, forced_invalid_frac=0.2)
    order, keys, _ = _schedule(w, cuda)
    assert sorted(order.tolist()) == list(range(B))
    ko = keys[order].astype(np.int64)
    assert (np.diff(ko) <= 0).all()
    same = np.diff(ko) == 0
    assert (np.diff(order)[same] > 0).all()
    if B > 1:
        assert len(set(keys.tolist())) > 1          # the batch mixes request kinds


def test_scheduled_parity_across_tiles(cuda, launch_options):
    """More requests than one schedule tile, mixed kinds: identical to the oracle."""
    launch_options(kernel="stream")
    launch_options(schedule=None)   # 2100 CTAs: scheduled by default
    w = W.make_batch(29, name="sched_parity_B2100", B=2100, V=640, k=(0, 5), logit_sigma=3.0,
                     temperature="half_greedy(0.5,1.2)", q_mode="half", draft_sigma=0.5,
                     mask="half", mask_density=0.1, mask_run_len=8, forced_invalid_frac=0.2)
    check_parity(w, cuda)


def test_wait_times_out_on_a_busy_stream(cuda):
    """specdec_wait gives up after its host-side limit while the stream is still busy (a device
    spin of about 0.2 s, which ends by itself), then waits it out without a limit."""
    import ctypes
    import time

    import torch

    lib = _native.load()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(400_000_000)             # clock cycles
    t0 = time.perf_counter()
    rc = lib.specdec_wait(ctypes.c_void_p(s.cuda_stream), 10)
    dt = time.perf_counter() - t0
    assert rc == _native.SPECDEC_ERR_TIMEOUT
    assert dt < 0.15, dt
    assert lib.specdec_wait(ctypes.c_void_p(s.cuda_stream), -1) == _native.SPECDEC_OK


@pytest.mark.parametrize("ctas", [1, 4])
def test_device_wait_expiry_is_reported_and_the_context_stays_usable(cuda, ctas, launch_options):
    """With every wait of the streaming kernel limited to 0 us, waits expire: each request reports
    SPECDEC_ST_DEVICE_TIMEOUT, the call completes (the CTAs stop issuing copies and drain the ones
    in flight before they leave), nothing is written past an output, and the same batch then
    verifies exactly with the default limit."""
    w = W.make_batch(501, name=f"expiry_G{ctas}", B=12, V=70000, k=(2, 5), logits_dtype=W.BF16,
                     logit_sigma=3.0, temperature="half_greedy(0.5,1.2)", q_mode="half", draft_sigma=0.5)
    launch_options(kernel="stream", ctas_per_request=ctas, wait_limit_us=0)
    got = device.run(w, device=cuda, diag=False, workspace=True, guard=64)
    assert got["guards_intact"]
    timed = (got["status"] & _native.ST_DEVICE_TIMEOUT) != 0
    assert timed.all(), got["status"]
    launch_options(wait_limit_us=None)
    check_parity(w, cuda)


@pytest.mark.parametrize("split", [1, 4, 40])
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_split_heavy_requests_parity(cuda, split, dtype, launch_options):
    """Clusters of 2 CTAs: the first `split` requests of the schedule are split over both CTAs of a
    cluster, the others run two per cluster, one per CTA (an odd remainder leaves the last
    cluster's second CTA without a request). Every request matches the oracle."""
    launch_options(kernel="stream", ctas_per_request=1, schedule=True, split_requests=split)
    w = W.make_batch(600 + split, name=f"split{split}_{dtype}", B=40, V=9000, k=(0, 6), logits_dtype=dtype,
                     logit_sigma=3.0, temperature="half_greedy(0.5,1.2)", q_mode="half", draft_sigma=0.5,
                     mask="half", mask_density=0.1, mask_run_len=16, forced_invalid_frac=0.2)
    check_parity(w, cuda)


def _tie_batch(V, dtype, ties, allowed=None, seed=0, name="ties"):
    """Greedy requests over rows whose maximum (an integer logit, exact in bf16) sits at every
    position in `ties`: a bonus-only request, a draft on a later copy of the maximum (rejected:
    the lowest index is the argmax), a draft on the lowest copy (accepted; its bonus row ties
    too), and two drafts (the second on a later copy)."""
    rng = np.random.default_rng([seed, V])
    ks = [0, 1, 1, 2]
    T = sum(ks) + len(ks)
    z = rng.integers(-60, 60, size=(T, V)).astype(np.float32)
    z[:, ties] = 100.0
    lo, later = ties[0], ties[-1]
    drafts = [later, lo, lo, later]
    return batch(V=V, ks=ks, logits=z, draft_ids=drafts, temperature=0.0, allowed=allowed, dtype=dtype,
                 name=name), lo


@pytest.mark.parametrize("ctas", [1, 2, 4])
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_greedy_ties_across_slices_and_chunks(cuda, ctas, dtype, launch_options):
    """The row maximum occurs in several CTAs' slices of a cluster and in several ring chunks of a
    slice: every CTA and every chunk folds to its own lowest index, and the fold across them keeps
    the lowest, so every emitted token is the first copy of the maximum."""
    launch_options(kernel="stream", ctas_per_request=ctas)
    V = 40000
    ties = [11000, 5, 9000, 10500, 19999, 30001, 39990]
    w, lo = _tie_batch(V, dtype, sorted(ties), name=f"ties_G{ctas}_{dtype}")
    rep, got, ref = check_parity(w, cuda)
    cu = w.cu_num_draft
    assert got["out_tokens"][rows_of(cu, 0, 0)] == lo                 # bonus only
    assert got["out_tokens"][rows_of(cu, 1, 0)] == lo                 # later copy rejected, lowest emitted
    assert got["out_num_accepted"][2] == 1 and got["out_tokens"][rows_of(cu, 2, 1)] == lo
    assert got["out_num_accepted"][3] == 1 and got["out_tokens"][rows_of(cu, 3, 1)] == lo


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_greedy_ties_across_sparse_list_segments(cuda, dtype, launch_options):
    """A sparse bitmask over a vocabulary wider than one list segment (5120 mask words): the maximum
    is allowed in both segments and in several 16-byte groups of each; the lowest allowed copy wins."""
    launch_options(kernel="stream", ctas_per_request=1)
    V = 200064                                        # 6252 mask words: two list segments
    ties = [777, 3001, 120003, 170000, 199999]
    w0, _ = _tie_batch(V, dtype, ties, name="shape")
    rng = np.random.default_rng(9)
    allowed = rng.random((w0.T, V)) < 0.05
    allowed[:, ties] = True
    allowed[:, 777] = False                           # the first copy is forbidden: 3001 must win
    w, _ = _tie_batch(V, dtype, ties, allowed=allowed, name=f"ties_sparse_{dtype}")
    assert _native.launch_config(V, 1 if dtype == W.BF16 else 0, B=w.B)["ctas_per_request"] == 1
    rep, got, ref = check_parity(w, cuda)
    cu = w.cu_num_draft
    assert got["out_tokens"][rows_of(cu, 0, 0)] == 3001
    assert got["out_tokens"][rows_of(cu, 1, 0)] == 3001
