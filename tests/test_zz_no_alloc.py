"""specdec_verify_noalloc, whose request-schedule scratch is a fixed array inside the library,
against specdec_verify with a caller workspace. The file name sorts last, so in a full run this
file is collected after every other test; it also passes on its own."""
import numpy as np
import pytest

import oracle
from oracle import parity
from speculative_decoding_verification_specdec_gb300 import _native, build, device
from speculative_decoding_verification_specdec_gb300 import workloads as W


@pytest.fixture(scope="module")
def lib():
    if build.needs_rebuild():
        build.build_library()
    return _native.load()


def test_requests_beyond_the_scratch_are_refused(lib):
    """B above SPECDEC_NOALLOC_MAX_REQUESTS fails before any CUDA call (fake, aligned pointers:
    nothing is dereferenced, no device is needed)."""
    f = 4096
    B = _native.NOALLOC_MAX_REQUESTS + 1
    rc = lib.specdec_verify_noalloc(f, 0, f, None, None, f, B, 1000, 3, None, f, None, None, f, f, f, f, f,
                                    None, None, None, None, None)
    assert rc == _native.SPECDEC_ERR_UNSUPPORTED
    rc0 = lib.specdec_verify_noalloc(f, 0, f, None, None, f, 0, 1000, 3, None, f, None, None, f, f, f, f, f,
                                     None, None, None, None, None)
    assert rc0 == _native.SPECDEC_OK                  # an empty batch needs no scratch


def _outputs(w, cuda, workspace):
    return device.alloc_outputs(w, cuda, diag=True, workspace=workspace)


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls(lib, launch_options):
    """Two calls in a row through each entry point on one batch large enough to be scheduled
    (1200 requests, mixed kinds): identical tokens, accepted counts, status and diagnostics on
    every call, counters doubled, and equal to the oracle."""
    import torch

    launch_options(schedule=None)
    launch_options(kernel="stream")
    torch.cuda.set_device(0)
    cuda = "cuda:0"
    w = W.make_batch(41, name="noalloc_B1200", B=1200, V=2048, k=(0, 6), logit_sigma=3.0,
                     temperature="half_greedy(0.5,1.2)", q_mode="half", draft_sigma=0.5,
                     mask="half", mask_density=0.05, mask_run_len=16, forced_invalid_frac=0.2)
    assert _native.launch_config(w.V, 0, B=w.B)["kernels_with_workspace"] == 2       # scheduled
    dev = device.device_tensors(w, cuda)

    ws_out = _outputs(w, cuda, workspace=True)
    na_out = _outputs(w, cuda, workspace=False)
    ws_calls, na_calls = [], []
    for _ in range(2):
        device.verify(w, dev, ws_out)
        torch.cuda.synchronize()
        ws_calls.append(ws_out.numpy())
    for _ in range(2):
        _native.specdec_verify_noalloc(
            dev["logits"], dev["draft_ids"], dev["draft_probs"], dev["has_q"], dev["cu_num_draft"],
            w.B, w.V, w.max_k, dev["bitmask"], dev["temperature"], dev["uniforms"], dev["exp_noise"],
            na_out.out_tokens, na_out.out_num_accepted, na_out.counters, na_out.status,
            na_out.diag_accept_prob, na_out.diag_row_stats, telemetry=na_out.telemetry)
        torch.cuda.synchronize()
        na_calls.append(na_out.numpy())

    for i in range(2):
        for k in ("out_tokens", "out_num_accepted", "status"):
            assert np.array_equal(na_calls[i][k], ws_calls[i][k]), (i, k)
        for k in ("diag_accept_prob", "diag_row_stats"):
            assert np.array_equal(na_calls[i][k], ws_calls[i][k], equal_nan=True), (i, k)
        assert np.array_equal(na_calls[i]["counters"], ws_calls[i]["counters"]), i
        assert np.array_equal(na_calls[i]["telemetry"], ws_calls[i]["telemetry"]), i
    assert np.array_equal(na_calls[1]["counters"], 2 * na_calls[0]["counters"])
    assert np.array_equal(na_calls[1]["telemetry"], 2 * na_calls[0]["telemetry"])

    ref = oracle.verify(w)
    rep = parity.compare(w, na_calls[0], ref)
    assert rep.ok, rep.summary()


@pytest.mark.gpu
def test_noalloc_with_top_k_top_p_matches_workspace_entry_point(lib, launch_options):
    """A filtered batch of 400 requests (scheduled: one CTA per filtered request) through both
    entry points: identical outputs, and equal to the oracle."""
    import torch

    launch_options(schedule=None)
    launch_options(kernel="stream")
    torch.cuda.set_device(0)
    cuda = "cuda:0"
    rng = np.random.default_rng(42)
    B = 400
    w = W.make_batch(42, name="noalloc_filters_B400", B=B, V=4096, k=(0, 5), logit_sigma=3.0,
                     temperature="half_greedy(0.5,1.2)", q_mode="half", draft_sigma=0.5, mask="half",
                     mask_density=0.1, mask_run_len=16,
                     top_k=rng.choice(np.array([0, 1, 20, 200], np.int32), B),
                     top_p=rng.choice(np.array([1.0, 0.5, 0.9], np.float32), B))
    assert _native.launch_config(w.V, 0, B=w.B)["kernels_with_workspace"] == 2
    dev = device.device_tensors(w, cuda)
    ws_out = _outputs(w, cuda, workspace=True)
    na_out = _outputs(w, cuda, workspace=False)
    device.verify(w, dev, ws_out)
    _native.specdec_verify_noalloc(
        dev["logits"], dev["draft_ids"], dev["draft_probs"], dev["has_q"], dev["cu_num_draft"],
        w.B, w.V, w.max_k, dev["bitmask"], dev["temperature"], dev["uniforms"], dev["exp_noise"],
        na_out.out_tokens, na_out.out_num_accepted, na_out.counters, na_out.status,
        na_out.diag_accept_prob, na_out.diag_row_stats, telemetry=na_out.telemetry,
        top_k=dev["top_k"], top_p=dev["top_p"])
    torch.cuda.synchronize()
    ws, na = ws_out.numpy(), na_out.numpy()
    for k in ("out_tokens", "out_num_accepted", "status", "counters", "telemetry"):
        assert np.array_equal(na[k], ws[k]), k
    for k in ("diag_accept_prob", "diag_row_stats"):
        assert np.array_equal(na[k], ws[k], equal_nan=True), k
    rep = parity.compare(w, na, oracle.verify(w))
    assert rep.ok, rep.summary()


@pytest.mark.gpu
def test_noalloc_at_the_largest_batch(lib, launch_options):
    """B = SPECDEC_NOALLOC_MAX_REQUESTS: the request order and the cost keys fill the array
    exactly. The schedule is forced on; the outputs equal those of specdec_verify given a
    workspace of specdec_workspace_size(B, V) bytes, and the oracle's."""
    import torch

    launch_options(schedule=True)
    launch_options(kernel="stream")
    torch.cuda.set_device(0)
    cuda = "cuda:0"
    B = _native.NOALLOC_MAX_REQUESTS
    w = W.make_batch(43, name="noalloc_Bmax", B=B, V=64, k=(0, 2), logit_sigma=3.0,
                     temperature="half_greedy(0.5,1.2)", q_mode="half", draft_sigma=0.5,
                     mask="half", mask_density=0.25, mask_run_len=4, forced_invalid_frac=0.2)
    dev = device.device_tensors(w, cuda)
    ws_out = _outputs(w, cuda, workspace=True)
    assert ws_out.workspace.numel() == _native.workspace_size(B, w.V)
    na_out = _outputs(w, cuda, workspace=False)
    device.verify(w, dev, ws_out)
    _native.specdec_verify_noalloc(
        dev["logits"], dev["draft_ids"], dev["draft_probs"], dev["has_q"], dev["cu_num_draft"],
        w.B, w.V, w.max_k, dev["bitmask"], dev["temperature"], dev["uniforms"], dev["exp_noise"],
        na_out.out_tokens, na_out.out_num_accepted, na_out.counters, na_out.status,
        na_out.diag_accept_prob, na_out.diag_row_stats, telemetry=na_out.telemetry)
    torch.cuda.synchronize()
    ws, na = ws_out.numpy(), na_out.numpy()
    for k in ("out_tokens", "out_num_accepted", "status", "counters", "telemetry"):
        assert np.array_equal(na[k], ws[k]), k
    for k in ("diag_accept_prob", "diag_row_stats"):
        assert np.array_equal(na[k], ws[k], equal_nan=True), k
    rep = parity.compare(w, na, oracle.verify(w))
    assert rep.ok, rep.summary()
