"""ctypes binding of libspecdec.so (include/specdec.h). Argument marshalling only:
every step of the verify runs in the CUDA library. There is no fallback; a missing
library raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libspecdec.so")

SPECDEC_OK = 0
SPECDEC_ERR_INVALID_ARG = 1
SPECDEC_ERR_UNSUPPORTED = 2
SPECDEC_ERR_CUDA = 3
SPECDEC_ERR_TIMEOUT = 4
SPECDEC_F32 = 0
SPECDEC_BF16 = 1
SPECDEC_KMAX = 32
TELEMETRY_SHAPE = (4, SPECDEC_KMAX + 1)   # rows: drafts, eligible, accepted-through by position; histogram

ST_BAD_DRAFT_ID = 1
ST_EMPTY_MASK_ROW = 2
ST_BAD_TEMPERATURE = 4
ST_K_TOO_LARGE = 8
ST_BAD_OFFSETS = 16
ST_DEVICE_TIMEOUT = 32
ST_BAD_TOP_P = 64

EXPORTED = ("specdec_verify", "specdec_verify_noalloc", "specdec_wait", "specdec_status_string",
            "specdec_launch_config", "specdec_workspace_size", "specdec_ngram_propose",
            "specdec_bitmask_scatter", "specdec_set_launch_options")
NGRAM_MAX_N = 64                        # SPECDEC_NGRAM_MAX_N
NOALLOC_MAX_REQUESTS = 16384            # SPECDEC_NOALLOC_MAX_REQUESTS

_lib = None


class SpecdecError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library. Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    lib.specdec_verify.restype = ctypes.c_int
    lib.specdec_verify.argtypes = [vp, ctypes.c_int, vp, vp, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                   vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.specdec_verify_noalloc.restype = ctypes.c_int
    lib.specdec_verify_noalloc.argtypes = [vp, ctypes.c_int, vp, vp, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                           vp, vp, vp, vp, vp, vp, vp, vp]
    lib.specdec_ngram_propose.restype = ctypes.c_int
    lib.specdec_ngram_propose.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp]
    lib.specdec_bitmask_scatter.restype = ctypes.c_int
    lib.specdec_bitmask_scatter.argtypes = [vp, ctypes.c_int64, vp, i32, vp, i32, i32, vp, vp]
    lib.specdec_workspace_size.restype = ctypes.c_size_t
    lib.specdec_workspace_size.argtypes = [i32, i32]
    lib.specdec_wait.restype = ctypes.c_int
    lib.specdec_wait.argtypes = [vp, i32]
    lib.specdec_status_string.restype = ctypes.c_char_p
    lib.specdec_status_string.argtypes = [ctypes.c_int]
    lib.specdec_launch_config.restype = ctypes.c_int
    lib.specdec_launch_config.argtypes = [i32, i32, ctypes.c_int, vp, vp, vp, vp, vp, vp]
    lib.specdec_set_launch_options.restype = ctypes.c_int
    lib.specdec_set_launch_options.argtypes = [i32, i32, i32, i32, i32]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().specdec_status_string(int(status)).decode()


def launch_config(V: int, dtype: int, B: int = 1024) -> dict:
    c, t, s, w, k, n = (ctypes.c_int32() for _ in range(6))
    rc = load().specdec_launch_config(int(B), int(V), int(dtype), ctypes.byref(c), ctypes.byref(t),
                                      ctypes.byref(s), ctypes.byref(w), ctypes.byref(k), ctypes.byref(n))
    if rc != SPECDEC_OK:
        raise SpecdecError(rc, "specdec_launch_config")
    return {"ctas_per_request": c.value, "threads_per_cta": t.value, "smem_bytes": s.value,
            "slice_ids": w.value, "kernels_with_workspace": k.value, "split_requests": n.value}


_KERNELS = {None: -1, "stream": 0, "cluster": 1}


def set_launch_options(kernel: Optional[str] = None, ctas_per_request: Optional[int] = None,
                       schedule: Optional[bool] = None, wait_limit_us: Optional[int] = None,
                       split_requests: Optional[int] = None) -> None:
    """specdec_set_launch_options: None leaves a choice to the library."""
    rc = load().specdec_set_launch_options(_KERNELS[kernel], -1 if ctas_per_request is None else int(ctas_per_request),
                                           -1 if schedule is None else int(bool(schedule)),
                                           -1 if wait_limit_us is None else int(wait_limit_us),
                                           -1 if split_requests is None else int(split_requests))
    if rc != SPECDEC_OK:
        raise SpecdecError(rc, "specdec_set_launch_options")


def workspace_size(B: int, V: int) -> int:
    return int(load().specdec_workspace_size(int(B), int(V)))


def _p(t) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr() if hasattr(t, "data_ptr") else int(t)


def _marshal(target_logits, logits_dtype, stream, tensors):
    import torch

    if logits_dtype is None:
        if target_logits.dtype == torch.bfloat16:
            logits_dtype = SPECDEC_BF16
        elif target_logits.dtype == torch.float32:
            logits_dtype = SPECDEC_F32
        else:
            raise SpecdecError(SPECDEC_ERR_UNSUPPORTED, f"logits dtype {target_logits.dtype}")
    for name, t in tensors:
        if t is not None and hasattr(t, "is_cuda"):
            if not t.is_cuda:
                raise ValueError(f"{name} must be a CUDA tensor")
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    return int(logits_dtype), stream


def specdec_verify(target_logits, draft_ids, draft_probs, has_q, cu_num_draft, B: int, V: int, max_k: int,
                   bitmask, temperature, uniforms, exp_noise, out_tokens, out_num_accepted, counters,
                   status=None, diag_accept_prob=None, diag_row_stats=None, workspace=None, stream=None,
                   logits_dtype=None, telemetry=None, top_k=None, top_p=None) -> None:
    """Queue one verify on `stream` (default: torch's current stream). Tensors are CUDA tensors
    (or raw device addresses as ints, with logits_dtype given); raises SpecdecError on a
    non-zero status."""
    dt, stream = _marshal(target_logits, logits_dtype, stream, (
        ("target_logits", target_logits), ("draft_ids", draft_ids), ("draft_probs", draft_probs),
        ("has_q", has_q), ("cu_num_draft", cu_num_draft), ("bitmask", bitmask),
        ("temperature", temperature), ("uniforms", uniforms), ("exp_noise", exp_noise),
        ("out_tokens", out_tokens), ("out_num_accepted", out_num_accepted), ("counters", counters),
        ("status", status), ("diag_accept_prob", diag_accept_prob), ("diag_row_stats", diag_row_stats),
        ("telemetry", telemetry), ("workspace", workspace), ("top_k", top_k), ("top_p", top_p)))
    rc = load().specdec_verify(
        _p(target_logits), dt, _p(draft_ids), _p(draft_probs), _p(has_q), _p(cu_num_draft),
        int(B), int(V), int(max_k), _p(bitmask), _p(temperature), _p(top_k), _p(top_p), _p(uniforms), _p(exp_noise),
        _p(out_tokens), _p(out_num_accepted), _p(counters), _p(status), _p(diag_accept_prob),
        _p(diag_row_stats), _p(telemetry), _p(workspace), 0 if workspace is None else _nbytes(workspace), stream)
    if rc != SPECDEC_OK:
        raise SpecdecError(rc, "specdec_verify")


def specdec_verify_noalloc(target_logits, draft_ids, draft_probs, has_q, cu_num_draft, B: int, V: int,
                           max_k: int, bitmask, temperature, uniforms, exp_noise, out_tokens, out_num_accepted,
                           counters, status=None, diag_accept_prob=None, diag_row_stats=None, stream=None,
                           logits_dtype=None, telemetry=None, top_k=None, top_p=None) -> None:
    """specdec_verify with the library's own schedule scratch (no workspace argument)."""
    dt, stream = _marshal(target_logits, logits_dtype, stream, (
        ("target_logits", target_logits), ("draft_ids", draft_ids), ("draft_probs", draft_probs),
        ("has_q", has_q), ("cu_num_draft", cu_num_draft), ("bitmask", bitmask),
        ("temperature", temperature), ("uniforms", uniforms), ("exp_noise", exp_noise),
        ("out_tokens", out_tokens), ("out_num_accepted", out_num_accepted), ("counters", counters),
        ("status", status), ("diag_accept_prob", diag_accept_prob), ("diag_row_stats", diag_row_stats),
        ("telemetry", telemetry), ("top_k", top_k), ("top_p", top_p)))
    rc = load().specdec_verify_noalloc(
        _p(target_logits), dt, _p(draft_ids), _p(draft_probs), _p(has_q), _p(cu_num_draft),
        int(B), int(V), int(max_k), _p(bitmask), _p(temperature), _p(top_k), _p(top_p), _p(uniforms), _p(exp_noise),
        _p(out_tokens), _p(out_num_accepted), _p(counters), _p(status), _p(diag_accept_prob),
        _p(diag_row_stats), _p(telemetry), stream)
    if rc != SPECDEC_OK:
        raise SpecdecError(rc, "specdec_verify_noalloc")


def _nbytes(t) -> int:
    return t.numel() * t.element_size() if hasattr(t, "numel") else 0


def specdec_wait(stream=None, timeout_ms: int = -1) -> None:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    rc = load().specdec_wait(stream, int(timeout_ms))
    if rc != SPECDEC_OK:
        raise SpecdecError(rc, "specdec_wait")


def ngram_propose(tokens, cu_hist, B: int, min_n: int, max_n: int, k: int, out_drafts, out_num, out_match,
                  stream=None) -> None:
    """Queue the n-gram proposer (specdec_ngram_propose) on `stream` (default: torch's current
    stream); raises SpecdecError on a non-zero status."""
    import torch

    for name, t in (("tokens", tokens), ("cu_hist", cu_hist), ("out_drafts", out_drafts), ("out_num", out_num),
                    ("out_match", out_match)):
        if t is not None and hasattr(t, "is_cuda") and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    rc = load().specdec_ngram_propose(_p(tokens), _p(cu_hist), int(B), int(min_n), int(max_n), int(k),
                                      _p(out_drafts), _p(out_num), _p(out_match), stream)
    if rc != SPECDEC_OK:
        raise SpecdecError(rc, "specdec_ngram_propose")


def bitmask_scatter(compact, compact_rows: int, constrained, n: int, cu_num_draft, B: int, V: int, bitmask,
                    stream=None) -> None:
    """Queue specdec_bitmask_scatter on `stream` (default: torch's current stream)."""
    import torch

    for name, t in (("compact", compact), ("constrained", constrained), ("cu_num_draft", cu_num_draft),
                    ("bitmask", bitmask)):
        if t is not None and hasattr(t, "is_cuda") and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    rc = load().specdec_bitmask_scatter(_p(compact), int(compact_rows), _p(constrained), int(n), _p(cu_num_draft),
                                        int(B), int(V), _p(bitmask), stream)
    if rc != SPECDEC_OK:
        raise SpecdecError(rc, "specdec_bitmask_scatter")
