"""The C-ABI library loads, exports every symbol include/specdec.h declares, and rejects bad
arguments on the host before touching the GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

from speculative_decoding_verification_specdec_gb300 import _native, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specdec.h")


@pytest.fixture(scope="module")
def lib():
    if build.needs_rebuild():
        build.build_library()
    return _native.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(specdec_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    assert declared_functions() == sorted(_native.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in [(0, "SPECDEC_OK"), (1, "SPECDEC_ERR_INVALID_ARG"), (2, "SPECDEC_ERR_UNSUPPORTED"),
                       (3, "SPECDEC_ERR_CUDA"), (4, "SPECDEC_ERR_TIMEOUT")]:
        assert _native.status_string(code) == name


@pytest.mark.parametrize("V,dtype", [(1, 0), (8, 0), (37, 1), (1000, 0), (32000, 0), (128256, 0), (151936, 0),
                                     (151936, 1), (262144, 1), (786432, 0)])
@pytest.mark.parametrize("kernel", ["stream", "cluster"])
@pytest.mark.parametrize("B", [1, 64, 128, 1024])
def test_launch_config_covers_the_row(lib, V, dtype, kernel, B, launch_options):
    launch_options(kernel=kernel)
    c = _native.launch_config(V, dtype, B=B)
    G, sl = c["ctas_per_request"], c["slice_ids"]
    assert 1 <= G <= 16 and sl % 128 == 0
    assert G * sl >= V and (G - 1) * sl < V          # every CTA owns a non-empty slice
    es = 4 if dtype == 0 else 2
    if kernel == "cluster":
        assert c["smem_bytes"] >= sl * es and c["smem_bytes"] <= 200 * 1024
        assert c["threads_per_cta"] == 256
    else:
        assert c["smem_bytes"] == 3 * 32 * 1024 and c["threads_per_cta"] == 288
        assert G <= 4
        if B >= 256:
            assert G == 1                            # enough requests to fill the GPU


def test_launch_config_reports_the_schedule(lib, launch_options):
    """Two kernels per call with a workspace once the grid exceeds one wave of resident CTAs
    (two per SM; 152 SMs when no device is visible), one otherwise; the override forces either."""
    launch_options(kernel="stream")
    launch_options(schedule=None)
    assert _native.launch_config(151936, 1, B=1024)["kernels_with_workspace"] == 2
    assert _native.launch_config(151936, 0, B=128)["kernels_with_workspace"] == 1
    assert _native.launch_config(32000, 0, B=64)["kernels_with_workspace"] == 1
    launch_options(schedule=True)
    assert _native.launch_config(32000, 0, B=64)["kernels_with_workspace"] == 2
    launch_options(schedule=False)
    assert _native.launch_config(151936, 1, B=1024)["kernels_with_workspace"] == 1
    assert _native.launch_config(151936, 1, B=1024)["split_requests"] == 0


def test_launch_config_reports_the_split(lib, launch_options):
    """A scheduled batch larger than one wave of resident CTAs (304 when no device is visible) splits
    its heaviest sixth of a wave over clusters of 2; smaller batches, and forced counts, as set."""
    launch_options(kernel="stream")
    assert _native.launch_config(151936, 1, B=1024)["split_requests"] == 50
    assert _native.launch_config(151936, 1, B=200)["split_requests"] == 0
    assert _native.launch_config(151936, 0, B=128)["split_requests"] == 0
    launch_options(split_requests=7)
    c = _native.launch_config(32000, 0, B=40)
    assert c["ctas_per_request"] > 1 and c["split_requests"] == 0      # small batches use clusters per request
    launch_options(ctas_per_request=1, split_requests=7)
    assert _native.launch_config(32000, 0, B=40)["split_requests"] == 7
    assert _native.launch_config(32000, 0, B=5)["split_requests"] == 5  # capped at B
    launch_options(ctas_per_request=1, split_requests=0)
    assert _native.launch_config(151936, 1, B=1024)["split_requests"] == 0


def test_launch_options_validation(lib):
    """specdec_set_launch_options refuses values outside its ranges and changes nothing then."""
    E = _native
    for bad in ((2, -1, -1, -1, -1), (-2, -1, -1, -1, -1), (-1, 0, -1, -1, -1), (-1, 17, -1, -1, -1),
                (-1, -2, -1, -1, -1), (-1, -1, 2, -1, -1), (-1, -1, -2, -1, -1), (-1, -1, -1, -2, -1),
                (-1, -1, -1, 2000001, -1), (-1, -1, -1, -1, -2)):
        assert lib.specdec_set_launch_options(*bad) == E.SPECDEC_ERR_INVALID_ARG, bad
    assert lib.specdec_set_launch_options(-1, 16, 1, 0, 5) == E.SPECDEC_OK
    assert _native.launch_config(1000, 0, B=4096)["kernels_with_workspace"] == 2
    assert lib.specdec_set_launch_options(-1, -1, 7, -1, -1) == E.SPECDEC_ERR_INVALID_ARG
    assert _native.launch_config(1000, 0, B=4096)["kernels_with_workspace"] == 2     # unchanged
    assert lib.specdec_set_launch_options(-1, -1, -1, -1, -1) == E.SPECDEC_OK


def test_launch_config_rejects(lib, launch_options):
    launch_options(kernel="cluster")
    with pytest.raises(_native.SpecdecError) as e:
        _native.launch_config(0, 0)
    assert e.value.status == _native.SPECDEC_ERR_INVALID_ARG
    with pytest.raises(_native.SpecdecError) as e:
        _native.launch_config(1000, 5)
    assert e.value.status == _native.SPECDEC_ERR_UNSUPPORTED
    with pytest.raises(_native.SpecdecError) as e:
        _native.launch_config(4 * 1024 * 1024, 0)     # a 16 MiB row cannot be staged on chip
    assert e.value.status == _native.SPECDEC_ERR_UNSUPPORTED
    launch_options(kernel="stream")   # the streaming kernel has no row-size limit
    assert _native.launch_config(4 * 1024 * 1024, 0, B=1024)["ctas_per_request"] == 1


def _call(lib, **over):
    # fake, aligned, non-NULL device addresses: every case below fails (or returns) before any
    # CUDA call, so nothing is dereferenced
    a = dict(logits=4096, dtype=0, ids=4096, q=None, has_q=None, cu=4096, B=4, V=1000, max_k=3, mask=None,
             temp=4096, u=4096, noise=4096, out=4096, acc=4096, ctr=4096, status=None, da=None, dr=None,
             tm=None, ws=None, ws_bytes=0, tk=None, tp=None)
    a.update(over)
    return lib.specdec_verify(a["logits"], a["dtype"], a["ids"], a["q"], a["has_q"], a["cu"], a["B"], a["V"],
                              a["max_k"], a["mask"], a["temp"], a["tk"], a["tp"], a["u"], a["noise"], a["out"], a["acc"],
                              a["ctr"], a["status"], a["da"], a["dr"], a["tm"], a["ws"], a["ws_bytes"], None)


def test_host_validation(lib, launch_options):
    launch_options(kernel="cluster")
    E = _native
    assert _call(lib, B=0) == E.SPECDEC_OK                        # empty batch: nothing launched
    assert _call(lib, B=-1) == E.SPECDEC_ERR_INVALID_ARG
    assert _call(lib, V=0) == E.SPECDEC_ERR_INVALID_ARG
    assert _call(lib, max_k=33) == E.SPECDEC_ERR_INVALID_ARG
    assert _call(lib, max_k=-1) == E.SPECDEC_ERR_INVALID_ARG
    assert _call(lib, dtype=2) == E.SPECDEC_ERR_UNSUPPORTED
    assert _call(lib, ids=None, B=0) == E.SPECDEC_OK                # no drafts: the id array may be NULL
    for k in ("logits", "cu", "temp", "u", "noise", "out", "acc", "ctr"):
        assert _call(lib, **{k: None}) == E.SPECDEC_ERR_INVALID_ARG, k
    assert _call(lib, logits=4098) == E.SPECDEC_ERR_INVALID_ARG   # fp32 logits not 4-byte aligned
    assert _call(lib, dtype=1, logits=4098, B=0) == E.SPECDEC_OK  # bf16 needs 2-byte alignment only
    assert _call(lib, ctr=4100) == E.SPECDEC_ERR_INVALID_ARG      # counters need 8-byte alignment
    assert _call(lib, mask=4097) == E.SPECDEC_ERR_INVALID_ARG
    assert _call(lib, tm=4100) == E.SPECDEC_ERR_INVALID_ARG        # telemetry needs 8-byte alignment
    assert _call(lib, tk=4098) == E.SPECDEC_ERR_INVALID_ARG
    assert _call(lib, tk=4096) == E.SPECDEC_ERR_UNSUPPORTED        # cluster kernel: no top-k / top-p
    assert _call(lib, V=4 * 1024 * 1024) == E.SPECDEC_ERR_UNSUPPORTED


def test_filter_vocabulary_limit(lib, launch_options):
    # top-k / top-p sum 12-bit mass parts in 32-bit bins: exact up to 2^20 elements per row
    launch_options(kernel=None)
    E = _native
    assert _call(lib, tp=4096, V=(1 << 20) + 1) == E.SPECDEC_ERR_UNSUPPORTED
    assert _call(lib, tk=4096, V=(1 << 20) + 1) == E.SPECDEC_ERR_UNSUPPORTED
    assert _call(lib, tk=4096, V=1 << 20, B=0) == E.SPECDEC_OK       # at the limit (empty batch: no launch)
    assert _call(lib, V=(1 << 20) + 1, B=0) == E.SPECDEC_OK          # no filter: no limit


def test_workspace_size_and_validation(lib, launch_options):
    E = _native
    assert _native.workspace_size(0, 1000) == 0 and _native.workspace_size(4, 0) == 0
    small, big = _native.workspace_size(4, 1000), _native.workspace_size(1024, 151936)
    assert small > 0 and big > small and small % 16 == 0 and big % 16 == 0
    assert big <= 5 * 1024 + 32                       # an int32 order and a key byte per request
    launch_options(kernel="stream")
    # a workspace that is too small or misaligned is refused before anything runs
    assert _call(lib, ws=4096, ws_bytes=small - 16) == E.SPECDEC_ERR_INVALID_ARG
    assert _call(lib, ws=4104, ws_bytes=small) == E.SPECDEC_ERR_INVALID_ARG


def test_product_path_has_no_oracle_import():
    """The package never imports, links or runs the oracle (test infrastructure only)."""
    pkg = os.path.join(ROOT, "speculative_decoding_verification_specdec_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "specdec_ref" not in text, f


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        saved = _native._lib
        _native._lib = None
        try:
            _native.load(str(tmp_path / "nope.so"))
        finally:
            _native._lib = saved


def test_ngram_host_validation(lib):
    """specdec_ngram_propose rejects bad sizes before any CUDA call (fake aligned pointers)."""
    E = _native
    f = 4096
    call = lambda **o: lib.specdec_ngram_propose(o.get("tok", f), o.get("cu", f), o.get("B", 4), o.get("min_n", 2),
                                                 o.get("max_n", 4), o.get("k", 3), o.get("d", f), o.get("n", f),
                                                 o.get("m", f), None)
    assert call(B=0) == E.SPECDEC_OK
    assert call(B=-1) == E.SPECDEC_ERR_INVALID_ARG
    assert call(min_n=0) == E.SPECDEC_ERR_INVALID_ARG
    assert call(k=-1) == E.SPECDEC_ERR_INVALID_ARG
    assert call(k=33) == E.SPECDEC_ERR_INVALID_ARG
    assert call(max_n=65) == E.SPECDEC_ERR_UNSUPPORTED
    assert call(tok=None) == E.SPECDEC_ERR_INVALID_ARG
    assert call(cu=4100) == E.SPECDEC_ERR_INVALID_ARG          # int64 offsets need 8-byte alignment


def test_bitmask_scatter_host_validation(lib):
    """specdec_bitmask_scatter rejects bad sizes before any CUDA call (fake aligned pointers)."""
    E = _native
    f = 4096
    call = lambda **o: lib.specdec_bitmask_scatter(o.get("c", f), o.get("rows", 10), o.get("ids", f), o.get("n", 3),
                                                   o.get("cu", f), o.get("B", 4), o.get("V", 1000), o.get("out", f), None)
    assert call(B=0) == E.SPECDEC_OK
    assert call(B=-1) == E.SPECDEC_ERR_INVALID_ARG
    assert call(V=0) == E.SPECDEC_ERR_INVALID_ARG
    assert call(n=-1) == E.SPECDEC_ERR_INVALID_ARG
    assert call(rows=-1) == E.SPECDEC_ERR_INVALID_ARG
    assert call(out=None) == E.SPECDEC_ERR_INVALID_ARG
    assert call(ids=None) == E.SPECDEC_ERR_INVALID_ARG
    assert call(c=4098) == E.SPECDEC_ERR_INVALID_ARG
