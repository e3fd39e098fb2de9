"""C-ABI checks that need no GPU: the library builds for sm_103a, loads, exports every function that
include/vsamp.h declares, and its host-only calls answer."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vsamp.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(vsamp_[a-z_]+)\s*\(", src)))


def _header_enum(name):
    src = open(HEADER).read()
    m = re.search(r"\b" + name + r"\s*=\s*(\d+)", src)
    return int(m.group(1))


@pytest.fixture(scope="module")
def lib():
    from top_sampling_gb300 import build as b

    path = b.build()
    return ctypes.CDLL(path)


def test_header_declares_the_five_stage_calls():
    fns = _declared_functions()
    for f in ("vsamp_softmax_lse", "vsamp_topk_select", "vsamp_topp_minp_mask", "vsamp_sample", "vsamp_logprob",
              "vsamp_status_string", "vsamp_device_info", "vsamp_version"):
        assert f in fns


def test_library_exports_every_declared_function(lib):
    for f in _declared_functions():
        assert hasattr(lib, f), f"libvsamp.so does not export {f}"


def test_status_strings_and_version(lib):
    lib.vsamp_status_string.restype = ctypes.c_char_p
    lib.vsamp_status_string.argtypes = [ctypes.c_int]
    for code in range(6):
        s = lib.vsamp_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.vsamp_status_string(99).decode() == "unknown status"
    lib.vsamp_version.restype = ctypes.c_int32
    assert lib.vsamp_version() >> 16 == 1


def test_status_codes_agree_across_header_binding_and_oracle():
    import top_sampling_gb300 as ts
    from oracle import sampler as osm

    assert _header_enum("VSAMP_OK") == ts.VSAMP_OK == osm.STATUS_OK
    assert _header_enum("VSAMP_ERR_INVALID_ARG") == ts.VSAMP_ERR_INVALID_ARG == osm.STATUS_INVALID_ARG
    assert _header_enum("VSAMP_ERR_NONFINITE") == ts.VSAMP_ERR_NONFINITE == osm.STATUS_NONFINITE
    assert _header_enum("VSAMP_ERR_UNSUPPORTED") == ts.VSAMP_ERR_UNSUPPORTED
    assert _header_enum("VSAMP_ERR_TIMEOUT") == ts.VSAMP_ERR_TIMEOUT
    assert _header_enum("VSAMP_BF16") == ts.VSAMP_BF16


def test_binding_declares_argument_types(lib):
    import top_sampling_gb300 as ts

    l2 = ts.load()
    assert set(ts.EXPORTED) == set(_declared_functions())
    for f in ts.EXPORTED:
        assert getattr(l2, f).restype is not None


def test_host_argument_checks_reject_before_any_device_work(lib):
    # NULL logits / bad sizes are rejected on the host; no CUDA call is made, so no GPU is needed
    vp = ctypes.c_void_p
    lib.vsamp_sample.restype = ctypes.c_int
    lib.vsamp_sample.argtypes = [vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64] + [vp] * 12
    assert lib.vsamp_sample(None, 0, 4, 100, 100, *([None] * 12)) == 1
    dummy = ctypes.c_void_p(16)
    assert lib.vsamp_sample(dummy, 7, 4, 100, 100, *([None] * 12)) == 1        # bad dtype
    assert lib.vsamp_sample(dummy, 0, 4, 100, 50, *([None] * 12)) == 1         # ld < V
    assert lib.vsamp_sample(dummy, 0, 0, 100, 100, *([None] * 12)) == 1        # B = 0
    assert lib.vsamp_sample(dummy, 0, 4, 100, 100, *([None] * 7), None, *([None] * 4)) == 1   # token NULL


def test_workspace_size_and_host_checks_of_the_workspace_entry_point(lib):
    import top_sampling_gb300 as ts

    l2 = ts.load()
    # a 256-byte reserved header and 32 + 128 bytes per 4 KB piece of a row (piece record, draw codes)
    assert l2.vsamp_sample_workspace_size(ts.VSAMP_BF16, 256, 151936) == 256 + 256 * 75 * 160
    assert l2.vsamp_sample_workspace_size(ts.VSAMP_F32, 4, 32000) == 256 + 4 * 32 * 160
    assert l2.vsamp_sample_workspace_size(7, 4, 100) == 0
    assert l2.vsamp_sample_workspace_size(ts.VSAMP_F32, 0, 100) == 0
    dummy = ctypes.c_void_p(16)
    args = [dummy, ts.VSAMP_F32, 4, 100, 100] + [None] * 7 + [dummy] + [None] * 3
    assert l2.vsamp_sample_ws(*args, None, 4096, None) == ts.VSAMP_ERR_INVALID_ARG          # no workspace
    assert l2.vsamp_sample_ws(*args, ctypes.c_void_p(4096 + 8), 4096, None) == ts.VSAMP_ERR_INVALID_ARG   # unaligned
    assert l2.vsamp_sample_ws(*args, ctypes.c_void_p(4096), 16, None) == ts.VSAMP_ERR_INVALID_ARG  # too small


def test_host_checks_of_the_topn_entry_point(lib):
    # list length and the required outputs are checked on the host, before any CUDA call
    import top_sampling_gb300 as ts
    l2 = ts.load()
    hdr = open(os.path.join(ROOT, "include", "vsamp.h")).read()
    assert "#define VSAMP_TOPN_MAX 4096" in hdr
    d = ctypes.c_void_p(4096)
    good = dict(rm=d, rl=d, oi=d, ol=d)

    def call(N, rm, rl, oi, ol):
        return l2.vsamp_topn_logprobs(d, ts.VSAMP_F32, 4, 100, 100, None, N, rm, rl, oi, ol, None, None)

    assert call(0, **good) == ts.VSAMP_ERR_INVALID_ARG
    assert call(4097, **good) == ts.VSAMP_ERR_INVALID_ARG
    assert call(20, **{**good, "rm": None}) == ts.VSAMP_ERR_INVALID_ARG
    assert call(20, **{**good, "rl": None}) == ts.VSAMP_ERR_INVALID_ARG
    assert call(20, **{**good, "oi": None}) == ts.VSAMP_ERR_INVALID_ARG
    assert call(20, **{**good, "ol": None}) == ts.VSAMP_ERR_INVALID_ARG
    assert l2.vsamp_topn_logprobs(None, ts.VSAMP_F32, 4, 100, 100, None, 20, d, d, d, d, None, None) == \
        ts.VSAMP_ERR_INVALID_ARG


def test_host_checks_of_the_kept_logprob_entry_point(lib):
    import top_sampling_gb300 as ts
    l2 = ts.load()
    d = ctypes.c_void_p(4096)
    args = (d, ts.VSAMP_F32, 4, 100, 100, None, None, None, None)
    assert l2.vsamp_kept_logprob(*args, None, d, None, None) == ts.VSAMP_ERR_INVALID_ARG   # no tokens
    assert l2.vsamp_kept_logprob(*args, d, None, None, None) == ts.VSAMP_ERR_INVALID_ARG   # no output
    assert l2.vsamp_kept_logprob(None, ts.VSAMP_F32, 4, 100, 100, None, None, None, None, d, d, None, None) == \
        ts.VSAMP_ERR_INVALID_ARG


def test_binding_rejects_host_tensors_and_bad_dtypes():
    # argument marshalling refuses what the library cannot take, before any call into it
    torch = pytest.importorskip("torch")
    import top_sampling_gb300 as ts
    x = torch.zeros(2, 8)
    for fn in (ts.vsamp_sample, ts.vsamp_softmax_lse, ts.vsamp_topp_minp_mask):
        with pytest.raises(ValueError):
            fn(x)
    with pytest.raises(ValueError):
        ts.vsamp_topn_logprobs(x, 4)
    with pytest.raises(ValueError):
        ts.vsamp_kept_logprob(x, torch.zeros(2, dtype=torch.int32))
    with pytest.raises(TypeError):
        ts._dtype_code(torch.zeros(2, 8, dtype=torch.float16))
