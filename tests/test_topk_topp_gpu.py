"""Top-k / top-p on the GPU against the oracle: mixed batches (fp32 and bf16, dense and sparse
rows, greedy and sampled, draft-model and model-free), ties at the top-k boundary, filters that
keep everything, and the bad-top_p flag."""
import dataclasses

import numpy as np
import pytest

import oracle
from oracle import parity
from speculative_decoding_verification_specdec_gb300 import _native, build, device
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


@pytest.fixture(autouse=True)
def stream_kernel(launch_options):
    launch_options(kernel="stream")


def _check(w, cuda, workspace=True):
    """Parity with the per-draft diagnostics (every filtered row runs the threshold search), then
    without them (accepted rows may be settled by the acceptance bound of the statistics pass,
    which must never change an outcome: the two runs agree bit for bit)."""
    got = device.run(w, device=cuda, diag=True, workspace=workspace)
    ref = oracle.verify(w)
    rep = parity.compare(w, got, ref)
    assert not (got["status"] & _native.ST_DEVICE_TIMEOUT).any()
    assert rep.ok, (f"{w.name}: {rep.summary()} tokens={rep.token_mismatches[:8]} acc={rep.accepted_mismatches[:8]} "
                    f"status={rep.status_mismatches[:8]} alpha={rep.alpha_bad[:5]}")
    fast = device.run(w, device=cuda, diag=False, workspace=workspace, telemetry=True)
    for key in ("out_tokens", "out_num_accepted", "status", "counters", "telemetry"):
        assert np.array_equal(fast[key], got[key]), (w.name, key)
    return rep, got, ref


def _filters(B, seed, ks=(0, 1, 3, 20, 200), ps=(1.0, 0.5, 0.8, 0.95, 0.999)):
    rng = np.random.default_rng(seed)
    return rng.choice(np.array(ks, np.int32), size=B), rng.choice(np.array(ps, np.float32), size=B)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("mask", ["none", "half"])
def test_mixed_batches(cuda, dtype, mask):
    B = 96
    tk, tp = _filters(B, 7 if dtype == W.F32 else 8)
    w = W.make_batch(61, name=f"topkp_{dtype}_{mask}", B=B, V=5000, k=(0, 5), logits_dtype=dtype, logit_sigma=2.5,
                     temperature="half_greedy(0.5,1.2)", q_mode="half", draft_sigma=0.4, mf_argmax_frac=0.5,
                     mask=mask, mask_density=0.1, mask_run_len=16, forced_invalid_frac=0.1, top_k=tk, top_p=tp)
    rep, got, ref = _check(w, cuda)
    assert rep.compared_tokens > 300


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_ties_at_the_boundary(cuda, dtype):
    """Logits on a coarse grid (many ties): every tie group at a top-k or top-p boundary is kept."""
    B, V = 120, 64
    rng = np.random.default_rng(3)
    tk, tp = _filters(B, 4, ks=(0, 1, 2, 5, 9), ps=(1.0, 0.3, 0.6, 0.9))
    w = W.make_batch(62, name=f"topkp_ties_{dtype}", B=B, V=V, k=(1, 4), logits_dtype=dtype, logit_sigma=1.0,
                     temperature="uniform(0.7,1.3)", q_mode="half", draft_sigma=0.5, top_k=tk, top_p=tp)
    grid = np.round(W.bf16_bits_to_f32(w.logits) if dtype == W.BF16 else w.logits)
    logits = W.f32_to_bf16_bits(grid.astype(np.float32)) if dtype == W.BF16 else grid.astype(np.float32)
    w = dataclasses.replace(w, logits=np.ascontiguousarray(logits))
    _check(w, cuda)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_top_k_ties_beyond_the_kept_id_slots(cuda, dtype):
    """Top-k 5 on rows whose maximum logit occurs about 3000 times: every copy is kept (ties at the
    threshold), more ids than the kept-id draw can list, so the stop row's draw streams the row as
    usual; top-k 3 on rows with a few copies takes the kept-id draw. Both against the oracle."""
    B, V = 24, 40000
    w = W.make_batch(65, name=f"topk_wide_ties_{dtype}", B=B, V=V, k=(1, 4), logits_dtype=dtype, logit_sigma=1.0,
                     temperature="uniform(0.7,1.3)", q_mode="half", draft_sigma=0.5,
                     top_k=np.where(np.arange(B) % 2 == 0, 5, 3).astype(np.int32))
    z = W.bf16_bits_to_f32(w.logits) if dtype == W.BF16 else w.logits
    scale = np.where((np.arange(w.T) % 2) == 0, 0.35, 3.0).astype(np.float32)[:, None]   # wide ties / few ties
    grid = np.round(z * scale).astype(np.float32)
    logits = W.f32_to_bf16_bits(grid) if dtype == W.BF16 else grid
    w = dataclasses.replace(w, logits=np.ascontiguousarray(logits))
    top = grid.max(axis=1, keepdims=True)
    assert ((grid == top).sum(axis=1) > 2048).any()
    _check(w, cuda)


def test_random_draft_model_batch_with_filters(cuda):
    """The benchmark's filtered batch: B=256, k=4, V=128256, fp32, per-request top-k / top-p."""
    _check(W.top_k_top_p_batch(), cuda)


def test_filters_that_keep_everything_change_nothing(cuda):
    w0 = W.make_batch(63, name="topkp_noop", B=48, V=3000, k=(0, 4), logit_sigma=2.0,
                      temperature="half_greedy(0.5,1.2)", q_mode="half", draft_sigma=0.4, mask="half",
                      mask_density=0.2, mask_run_len=8)
    base = device.run(w0, device=cuda, diag=False)
    for tk, tpv in ((0, 1.0), (3000, 1.0), (100000, 2.0)):
        w = dataclasses.replace(w0, top_k=np.full(48, tk, np.int32), top_p=np.full(48, tpv, np.float32))
        got = device.run(w, device=cuda, diag=False)
        assert np.array_equal(got["out_tokens"], base["out_tokens"]), (tk, tpv)
        assert np.array_equal(got["counters"], base["counters"])


def test_bad_top_p_is_flagged(cuda):
    w0 = W.make_batch(64, name="topkp_bad", B=16, V=1000, k=2, logit_sigma=2.0, temperature=1.0, q_mode="all",
                      draft_sigma=0.4)
    w = dataclasses.replace(w0, top_p=np.array([0.0, -1.0, np.nan, 0.5] * 4, np.float32))
    rep, got, ref = _check(w, cuda)
    flagged = (got["status"] & _native.ST_BAD_TOP_P) != 0
    assert flagged.tolist() == [True, True, True, False] * 4


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("route", ["streamed_digits", "bin_on_chip", "all_kept_on_chip", "top_p_peaked"])
def test_threshold_search_routes(cuda, dtype, route):
    """Rows of 65536 logits that drive each route of the threshold search: a near-flat row whose
    chosen mass bin holds far more elements than fit on chip (every digit pass streams the row), a
    top-k of 3000 (above the top-slice limit; the chosen bin fits on chip, the elements above it do
    not), a small top-k followed by top-p (the top slice of logits holds every kept element, so the
    top-p search streams nothing), and top-p alone on peaked rows (a small chosen bin, its digits on
    chip)."""
    B, V = 24, 65536
    rng = np.random.default_rng({"streamed_digits": 11, "bin_on_chip": 12, "all_kept_on_chip": 13,
                                 "top_p_peaked": 14}[route])
    temperature = "uniform(0.5,1.2)"
    if route == "streamed_digits":
        # (k = 100: the top slice of a near-flat row is empty, so the top-k search falls back to the row)
        sigma, tk, tp = 0.02, rng.choice(np.array([0, 100, 5000, 20000], np.int32), B), \
            rng.choice(np.array([1.0, 0.3, 0.5, 0.7], np.float32), B)
    elif route == "bin_on_chip":
        sigma, tk, tp = 3.0, np.full(B, 3000, np.int32), rng.choice(np.array([1.0, 0.9, 0.97], np.float32), B)
    elif route == "all_kept_on_chip":
        sigma, tk, tp = 3.0, rng.choice(np.array([10, 50, 300], np.int32), B), \
            rng.choice(np.array([1.0, 0.5, 0.8, 0.95], np.float32), B)
    else:
        sigma, tk, tp = 3.0, np.zeros(B, np.int32), rng.choice(np.array([0.5, 0.8, 0.9], np.float32), B)
        temperature = "uniform(0.4,0.6)"
    w = W.make_batch(65, name=f"topkp_route_{route}_{dtype}", B=B, V=V, k=(1, 4), logits_dtype=dtype,
                     logit_sigma=sigma, temperature=temperature, q_mode="half", draft_sigma=0.4,
                     top_k=tk, top_p=tp)
    rep, got, ref = _check(w, cuda)
    assert rep.compared_tokens > 40


def test_largest_filtered_vocabulary(cuda):
    """V = 2^20, the widest row a filtered launch takes, with near-flat logits: about 2^20 elements
    share one mass bin, where the 32-bit sums of 12-bit mass halves reach their bound (the top-k
    request's digit passes sum the masses of that bin). The top-p request runs too, but every
    element there carries about 1e-6 of the mass, so its boundary lies inside the excluded band."""
    B, V = 2, 1 << 20
    w = W.make_batch(66, name="topkp_V2p20", B=B, V=V, k=2, logit_sigma=0.001, temperature=1.0, q_mode="all",
                     draft_sigma=0.0005, top_k=np.array([0, 300000], np.int32),
                     top_p=np.array([0.5, 1.0], np.float32))
    rep, got, ref = _check(w, cuda)
    assert rep.compared_tokens >= 1
