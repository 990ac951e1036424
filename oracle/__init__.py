"""CPU oracle for batched speculative-decoding verification (TEST INFRASTRUCTURE ONLY).

Plain C, fp64, single-threaded (``specdec_ref.c``); this module only compiles it
with gcc and marshals numpy arrays through ctypes. Only the test suite,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import it;
the product package never does.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sysconfig
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "specdec_ref.c")
_LIB = os.path.join(_HERE, "libspecdec_ref.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall", "-Wextra"]

ST_BAD_DRAFT_ID = 1
ST_EMPTY_MASK_ROW = 2
ST_BAD_TEMPERATURE = 4
ST_K_TOO_LARGE = 8
ST_BAD_OFFSETS = 16


def build(src: str = _SRC, out: str = _LIB, extra_flags=(), quiet: bool = True) -> str:
    """Compile the oracle (gcc, plain C11) into a shared library; returns its path."""
    tmp = f"{out}.tmp{os.getpid()}"
    cmd = ["gcc", *_CFLAGS, *extra_flags, "-o", tmp, src, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"oracle build failed: {' '.join(cmd)}\n{res.stderr}")
    os.replace(tmp, out)
    if not quiet and res.stderr:
        print(res.stderr)
    return out


class _Diag(ctypes.Structure):
    _fields_ = [
        ("alpha", ctypes.c_void_p),
        ("row_m", ctypes.c_void_p),
        ("row_S", ctypes.c_void_p),
        ("emit_top1", ctypes.c_void_p),
        ("emit_top2", ctypes.c_void_p),
        ("emit_scores", ctypes.c_void_p),
        ("score_request", ctypes.c_int32),
        ("top_p_margin", ctypes.c_void_p),
        ("telemetry", ctypes.c_void_p),
    ]

TELEMETRY_SHAPE = (4, 33)   # rows: drafts, eligible, accepted by position; histogram of accepted


_loaded = {}


def load(path: str = _LIB):
    """Load (building first if missing or stale) the oracle library at `path`."""
    if path in _loaded:
        return _loaded[path]
    if path == _LIB and (not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC)):
        build()
    lib = ctypes.CDLL(path)
    fn = lib.specdec_verify_ref
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int32,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.POINTER(_Diag)]
    ng = lib.specdec_ngram_ref
    ng.restype = ctypes.c_int
    ng.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                   ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    _loaded[path] = lib
    return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


class OracleResult(dict):
    """out_tokens [T], out_num_accepted [B], counters [4] (R, I, D, A), status [B],
    alpha [N], row_m [T], row_S [T], emit_top1 [B], emit_top2 [B], emit_scores [V],
    telemetry [4, 33], top_p_margin [T] (see specdec_ref.h)."""

    def __getattr__(self, k):
        try:
            return self[k]
        except KeyError as e:
            raise AttributeError(k) from e


def verify(w, *, score_request: int = -1, counters: Optional[np.ndarray] = None,
           lib_path: str = _LIB) -> OracleResult:
    """Run the oracle on a host workload (``workloads.Workload``)."""
    lib = load(lib_path)
    B, V, N, T = w.B, w.V, w.N, w.T
    out_tokens = np.full(T, -7, dtype=np.int32)
    out_num = np.full(B, -7, dtype=np.int32)
    ctr = np.zeros(4, dtype=np.uint64) if counters is None else counters
    status = np.zeros(B, dtype=np.uint32)
    alpha = np.empty(N, dtype=np.float64)
    row_m = np.empty(T, dtype=np.float64)
    row_S = np.empty(T, dtype=np.float64)
    top1 = np.empty(B, dtype=np.float64)
    top2 = np.empty(B, dtype=np.float64)
    scores = np.empty(V, dtype=np.float64)
    telemetry = np.zeros(TELEMETRY_SHAPE, dtype=np.uint64)
    margin = np.empty(T, dtype=np.float64)
    diag = _Diag(alpha.ctypes.data, row_m.ctypes.data, row_S.ctypes.data, top1.ctypes.data,
                 top2.ctypes.data, scores.ctypes.data, int(score_request), margin.ctypes.data,
                 telemetry.ctypes.data)
    logits = np.ascontiguousarray(w.logits)
    dtype = 1 if w.logits_dtype == "bf16" else 0
    args = [np.ascontiguousarray(a) if a is not None else None for a in
            (w.draft_ids, w.draft_probs, w.has_q, w.cu_num_draft, w.bitmask, w.temperature,
             w.uniforms, w.exp_noise, getattr(w, "top_k", None), getattr(w, "top_p", None))]
    rc = lib.specdec_verify_ref(
        _ptr(logits), dtype, _ptr(args[0]), _ptr(args[1]), _ptr(args[2]), _ptr(args[3]),
        B, V, int(w.max_k), _ptr(args[4]), _ptr(args[5]), _ptr(args[6]), _ptr(args[7]),
        _ptr(args[8]), _ptr(args[9]),
        _ptr(out_tokens), _ptr(out_num), _ptr(ctr), _ptr(status), ctypes.byref(diag))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return OracleResult(out_tokens=out_tokens, out_num_accepted=out_num, counters=ctr, status=status,
                        alpha=alpha, row_m=row_m, row_S=row_S, emit_top1=top1, emit_top2=top2,
                        emit_scores=scores, telemetry=telemetry, top_p_margin=margin)


def ngram_propose(histories, *, min_n: int = 2, max_n: int = 4, k: int = 3, lib_path: str = _LIB):
    """N-gram proposer on the host (specdec_ngram_ref). `histories` is a list of token sequences,
    or a pair (tokens int32 [total], cu_hist int64 [B+1]). Returns (drafts [B, k] with -1 padding,
    num [B], match [B]) as numpy arrays."""
    lib = load(lib_path)
    if isinstance(histories, tuple):
        tokens, cu = (np.ascontiguousarray(histories[0], dtype=np.int32),
                      np.ascontiguousarray(histories[1], dtype=np.int64))
    else:
        lens = [len(h) for h in histories]
        cu = np.zeros(len(histories) + 1, dtype=np.int64)
        cu[1:] = np.cumsum(lens)
        tokens = (np.concatenate([np.asarray(h, dtype=np.int32) for h in histories])
                  if histories and cu[-1] > 0 else np.zeros(1, dtype=np.int32))
    B = cu.size - 1
    drafts = np.full((B, max(k, 1)), -7, dtype=np.int32)
    num = np.full(B, -7, dtype=np.int32)
    match = np.full(B, -7, dtype=np.int32)
    rc = lib.specdec_ngram_ref(_ptr(tokens), _ptr(cu), B, int(min_n), int(max_n), int(k), _ptr(drafts),
                               _ptr(num), _ptr(match))
    if rc != 0:
        raise ValueError(f"oracle rejected the n-gram arguments (rc={rc})")
    return drafts[:, :k], num, match
