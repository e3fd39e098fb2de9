"""Thin Python binding of libvsamp.so, the GB300 per-row vocabulary sampling stage.

The functions carry the C-ABI names (include/vsamp.h) and only marshal arguments: torch tensors are
passed as device pointers, missing outputs are allocated with torch on the input's device, and the
call is enqueued on the current torch stream. Every step of the stage runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback. If the library is missing the import still works, but
every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libvsamp.so")

VSAMP_OK = 0
VSAMP_ERR_INVALID_ARG = 1
VSAMP_ERR_UNSUPPORTED = 2
VSAMP_ERR_CUDA = 3
VSAMP_ERR_NONFINITE = 4
VSAMP_ERR_TIMEOUT = 5
VSAMP_ERR_SCRATCH_LIMIT = 6
VSAMP_STATIC_SCRATCH_BYTES = 1 << 22   # the fixed scratch array of vsamp_sample_static
VSAMP_F32 = 0
VSAMP_BF16 = 1

EXPORTED = ("vsamp_softmax_lse", "vsamp_topk_select", "vsamp_topp_minp_mask", "vsamp_sample",
            "vsamp_sample_ws", "vsamp_sample_workspace_size", "vsamp_sample_static", "vsamp_logprob", "vsamp_topn_logprobs", "vsamp_kept_logprob",
            "vsamp_shard_pieces", "vsamp_shard_workspace_size", "vsamp_shard_partial", "vsamp_shard_merge",
            "vsamp_sample_rejection",
            "vsamp_status_string",
            "vsamp_device_info", "vsamp_version")


class VsampError(RuntimeError):
    def __init__(self, status: int, fn: str):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


class vsamp_cut(ctypes.Structure):
    _fields_ = [("pivot_key", ctypes.c_uint32), ("idx_cut", ctypes.c_int32), ("kept", ctypes.c_int32),
                ("status", ctypes.c_int32)]


class vsamp_limits(ctypes.Structure):
    _fields_ = [("sm_count", ctypes.c_int32), ("smem_optin_bytes", ctypes.c_int32),
                ("max_cluster", ctypes.c_int32), ("max_row_f32", ctypes.c_int64),
                ("max_row_bf16", ctypes.c_int64)]


_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libvsamp.so (once) and declare the C signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is not built: run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(p)
    vp, i64, i32, st = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int
    lib.vsamp_softmax_lse.argtypes = [vp, st, i64, i64, i64, vp, vp, vp, vp, vp]
    lib.vsamp_topk_select.argtypes = [vp, st, i64, i64, i64, vp, vp, i32, vp, vp, vp]
    lib.vsamp_topp_minp_mask.argtypes = [vp, st, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.vsamp_sample.argtypes = [vp, st, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.vsamp_logprob.argtypes = [vp, st, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp]
    lib.vsamp_sample_ws.argtypes = [vp, st, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                    ctypes.c_size_t, vp]
    lib.vsamp_sample_static.argtypes = [vp, st, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.vsamp_topn_logprobs.argtypes = [vp, st, i64, i64, i64, vp, i32, vp, vp, vp, vp, vp, vp]
    lib.vsamp_shard_pieces.argtypes = [st, i64]
    lib.vsamp_shard_pieces.restype = i64
    lib.vsamp_shard_workspace_size.argtypes = [st, i64, i64]
    lib.vsamp_shard_workspace_size.restype = ctypes.c_size_t
    lib.vsamp_shard_partial.argtypes = [vp, st, i64, i64, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp,
                                        ctypes.c_size_t, vp]
    lib.vsamp_shard_merge.argtypes = [vp, vp, i32, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.vsamp_shard_partial.restype = st
    lib.vsamp_sample_rejection.argtypes = [vp, st, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.vsamp_sample_rejection.restype = st
    lib.vsamp_shard_merge.restype = st
    lib.vsamp_kept_logprob.argtypes = [vp, st, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.vsamp_sample_workspace_size.argtypes = [st, i64, i64]
    lib.vsamp_sample_workspace_size.restype = ctypes.c_size_t
    for f in ("vsamp_softmax_lse", "vsamp_topk_select", "vsamp_topp_minp_mask", "vsamp_sample", "vsamp_logprob",
              "vsamp_sample_ws", "vsamp_sample_static", "vsamp_topn_logprobs", "vsamp_kept_logprob"):
        getattr(lib, f).restype = st
    lib.vsamp_status_string.argtypes = [st]
    lib.vsamp_status_string.restype = ctypes.c_char_p
    lib.vsamp_device_info.argtypes = [ctypes.c_int, ctypes.POINTER(vsamp_limits)]
    lib.vsamp_device_info.restype = st
    lib.vsamp_version.argtypes = []
    lib.vsamp_version.restype = i32
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().vsamp_status_string(int(status)).decode()


def version() -> int:
    return int(load().vsamp_version())


def device_info(device: int = 0) -> vsamp_limits:
    out = vsamp_limits()
    _check(load().vsamp_device_info(int(device), ctypes.byref(out)), "vsamp_device_info")
    return out


# ------------------------------------------------------------------------------------------------
# marshalling helpers
# ------------------------------------------------------------------------------------------------
def _check(status: int, fn: str):
    if status != VSAMP_OK:
        raise VsampError(status, fn)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return VSAMP_F32
    if t.dtype == torch.bfloat16:
        return VSAMP_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _rows(x: torch.Tensor, V: Optional[int]):
    if x.dim() != 2 or not x.is_cuda:
        raise ValueError("logits must be a 2-D CUDA tensor [B, >= V]")
    if x.stride(1) != 1:
        raise ValueError("logits rows must be contiguous (stride(1) == 1)")
    B = x.shape[0]
    V = x.shape[1] if V is None else int(V)
    return B, V, x.stride(0) if B > 1 else max(x.stride(0), V)


def _ptr(t: Optional[torch.Tensor], dtype=None, dev=None, B=None, name="") -> int:
    if t is None:
        return 0
    if not t.is_cuda or (dev is not None and t.device != dev):
        raise ValueError(f"{name} must be on {dev}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if B is not None and t.numel() < B:
        raise ValueError(f"{name} needs at least {B} elements")
    return t.data_ptr()


def _param(v, B: int, dtype, dev, name):
    """Per-row parameter: None, a scalar (broadcast) or a [B] device tensor."""
    if v is None:
        return None
    if isinstance(v, torch.Tensor):
        return v.to(device=dev, dtype=dtype).contiguous()
    return torch.full((B,), v, dtype=dtype, device=dev)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


# ------------------------------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ------------------------------------------------------------------------------------------------
def vsamp_softmax_lse(logits, temperature=None, V=None, row_max=None, row_logsum=None, row_status=None,
                      stream=None):
    """Row maximum and log-sum-exp of (x - max)/T. Returns (row_max, row_logsum, row_status)."""
    B, V, ld = _rows(logits, V)
    dev = logits.device
    temperature = _param(temperature, B, torch.float32, dev, "temperature")
    row_max = torch.empty(B, dtype=torch.float32, device=dev) if row_max is None else row_max
    row_logsum = torch.empty(B, dtype=torch.float32, device=dev) if row_logsum is None else row_logsum
    row_status = torch.empty(B, dtype=torch.int32, device=dev) if row_status is None else row_status
    st = load().vsamp_softmax_lse(
        logits.data_ptr(), _dtype_code(logits), B, V, ld, _ptr(temperature, torch.float32, dev, B, "temperature"),
        _ptr(row_max, torch.float32, dev, B, "row_max"), _ptr(row_logsum, torch.float32, dev, B, "row_logsum"),
        _ptr(row_status, torch.int32, dev, B, "row_status"), _stream(stream))
    _check(st, "vsamp_softmax_lse")
    return row_max, row_logsum, row_status


def vsamp_topk_select(scores, k, k_max=None, lengths=None, max_len=None, out_idx=None, row_status=None,
                      stream=None):
    """Top-k indices per row in ascending index order, -1 padded. Returns (out_idx [B, k_max], row_status)."""
    B, max_len, ld = _rows(scores, max_len)
    dev = scores.device
    if isinstance(k, int) and k_max is None:
        k_max = k
    if k_max is None:
        raise ValueError("k_max is required when k is a tensor")
    k = _param(k, B, torch.int32, dev, "k")
    lengths = _param(lengths, B, torch.int32, dev, "lengths")
    out_idx = torch.empty((B, int(k_max)), dtype=torch.int32, device=dev) if out_idx is None else out_idx
    row_status = torch.empty(B, dtype=torch.int32, device=dev) if row_status is None else row_status
    st = load().vsamp_topk_select(
        scores.data_ptr(), _dtype_code(scores), B, max_len, ld, _ptr(lengths, torch.int32, dev, B, "lengths"),
        _ptr(k, torch.int32, dev, B, "k"), int(k_max), _ptr(out_idx, torch.int32, dev, B * int(k_max), "out_idx"),
        _ptr(row_status, torch.int32, dev, B, "row_status"), _stream(stream))
    _check(st, "vsamp_topk_select")
    return out_idx, row_status


def vsamp_topp_minp_mask(logits, temperature=None, top_k=None, top_p=None, min_p=None, V=None,
                         want_mask=True, cut=None, mask=None, stats=None, stream=None):
    """Cut descriptors [B, 4] int32 (pivot_key as int32 bits, idx_cut, kept, status), mask [B, V] uint8
    (or None) and stats [B, 4]."""
    B, V, ld = _rows(logits, V)
    dev = logits.device
    temperature = _param(temperature, B, torch.float32, dev, "temperature")
    top_k = _param(top_k, B, torch.int32, dev, "top_k")
    top_p = _param(top_p, B, torch.float32, dev, "top_p")
    min_p = _param(min_p, B, torch.float32, dev, "min_p")
    cut = torch.empty((B, 4), dtype=torch.int32, device=dev) if cut is None else cut
    if want_mask and mask is None:
        mask = torch.empty((B, V), dtype=torch.uint8, device=dev)
    stats = torch.empty((B, 4), dtype=torch.int32, device=dev) if stats is None else stats
    st = load().vsamp_topp_minp_mask(
        logits.data_ptr(), _dtype_code(logits), B, V, ld, _ptr(temperature, torch.float32, dev, B, "temperature"),
        _ptr(top_k, torch.int32, dev, B, "top_k"), _ptr(top_p, torch.float32, dev, B, "top_p"),
        _ptr(min_p, torch.float32, dev, B, "min_p"), _ptr(cut, torch.int32, dev, 4 * B, "cut"),
        _ptr(mask, torch.uint8, dev, B * V, "mask"), _ptr(stats, torch.int32, dev, 4 * B, "stats"),
        _stream(stream))
    _check(st, "vsamp_topp_minp_mask")
    return cut, mask, stats


def vsamp_sample(logits, temperature=None, top_k=None, top_p=None, min_p=None, seed=None, step=None,
                 row_id=None, V=None, token=None, logprob=None, row_status=None, stats=None,
                 want_logprob=True, want_stats=False, stream=None):
    """The fused stage. Returns (token [B] int32, logprob [B] fp32 or None, row_status [B], stats or None)."""
    B, V, ld = _rows(logits, V)
    dev = logits.device
    temperature = _param(temperature, B, torch.float32, dev, "temperature")
    top_k = _param(top_k, B, torch.int32, dev, "top_k")
    top_p = _param(top_p, B, torch.float32, dev, "top_p")
    min_p = _param(min_p, B, torch.float32, dev, "min_p")
    seed = _param(seed, B, torch.int64, dev, "seed")
    step = _param(step, B, torch.int64, dev, "step")
    row_id = _param(row_id, B, torch.int32, dev, "row_id")
    token = torch.empty(B, dtype=torch.int32, device=dev) if token is None else token
    if want_logprob and logprob is None:
        logprob = torch.empty(B, dtype=torch.float32, device=dev)
    row_status = torch.empty(B, dtype=torch.int32, device=dev) if row_status is None else row_status
    if want_stats and stats is None:
        stats = torch.empty((B, 4), dtype=torch.int32, device=dev)
    st = load().vsamp_sample(
        logits.data_ptr(), _dtype_code(logits), B, V, ld, _ptr(temperature, torch.float32, dev, B, "temperature"),
        _ptr(top_k, torch.int32, dev, B, "top_k"), _ptr(top_p, torch.float32, dev, B, "top_p"),
        _ptr(min_p, torch.float32, dev, B, "min_p"), _ptr(seed, torch.int64, dev, B, "seed"),
        _ptr(step, torch.int64, dev, B, "step"), _ptr(row_id, torch.int32, dev, B, "row_id"),
        _ptr(token, torch.int32, dev, B, "token"), _ptr(logprob, torch.float32, dev, B, "logprob"),
        _ptr(row_status, torch.int32, dev, B, "row_status"), _ptr(stats, torch.int32, dev, 4 * B, "stats"),
        _stream(stream))
    _check(st, "vsamp_sample")
    return token, logprob, row_status, stats


def vsamp_sample_rejection(logits, temperature=None, top_k=None, top_p=None, min_p=None, seed=None, step=None,
                           row_id=None, V=None, token=None, logprob=None, row_status=None, stats=None,
                           want_logprob=True, want_stats=False, stream=None):
    """The dual-pivot rejection sampler: the law of vsamp_sample from other random numbers. Returns (token,
    logprob or None, row_status, stats or None); stats rows are {passes, rounds, 0, path flags}."""
    B, V, ld = _rows(logits, V)
    dev = logits.device
    temperature = _param(temperature, B, torch.float32, dev, "temperature")
    top_k = _param(top_k, B, torch.int32, dev, "top_k")
    top_p = _param(top_p, B, torch.float32, dev, "top_p")
    min_p = _param(min_p, B, torch.float32, dev, "min_p")
    seed = _param(seed, B, torch.int64, dev, "seed")
    step = _param(step, B, torch.int64, dev, "step")
    row_id = _param(row_id, B, torch.int32, dev, "row_id")
    token = torch.empty(B, dtype=torch.int32, device=dev) if token is None else token
    if want_logprob and logprob is None:
        logprob = torch.empty(B, dtype=torch.float32, device=dev)
    row_status = torch.empty(B, dtype=torch.int32, device=dev) if row_status is None else row_status
    if want_stats and stats is None:
        stats = torch.empty((B, 4), dtype=torch.int32, device=dev)
    st = load().vsamp_sample_rejection(
        logits.data_ptr(), _dtype_code(logits), B, V, ld, _ptr(temperature, torch.float32, dev, B, "temperature"),
        _ptr(top_k, torch.int32, dev, B, "top_k"), _ptr(top_p, torch.float32, dev, B, "top_p"),
        _ptr(min_p, torch.float32, dev, B, "min_p"), _ptr(seed, torch.int64, dev, B, "seed"),
        _ptr(step, torch.int64, dev, B, "step"), _ptr(row_id, torch.int32, dev, B, "row_id"),
        _ptr(token, torch.int32, dev, B, "token"), _ptr(logprob, torch.float32, dev, B, "logprob"),
        _ptr(row_status, torch.int32, dev, B, "row_status"), _ptr(stats, torch.int32, dev, 4 * B, "stats"),
        _stream(stream))
    _check(st, "vsamp_sample_rejection")
    return token, logprob, row_status, stats


_WORKSPACES = {}


def sample_workspace(device, nbytes: int, stream=None) -> torch.Tensor:
    """A workspace of at least nbytes for vsamp_sample_ws, cached per (device, stream).

    A call writes everything it reads in the workspace, so it is reused as is; calls
    on one stream never overlap, so a workspace per stream is enough."""
    dev = torch.device(device)
    key = (dev.index if dev.index is not None else torch.cuda.current_device(), _stream(stream))
    ws = _WORKSPACES.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=dev)
        _WORKSPACES[key] = ws
    return ws


def vsamp_sample_ws(logits, temperature=None, top_k=None, top_p=None, min_p=None, seed=None, step=None,
                    row_id=None, V=None, token=None, logprob=None, row_status=None, stats=None,
                    want_logprob=True, want_stats=False, stream=None, workspace=None):
    """vsamp_sample through the split-vocabulary kernels and a workspace (cached per device and stream
    unless given). Returns (token, logprob or None, row_status, stats or None)."""
    B, V, ld = _rows(logits, V)
    dev = logits.device
    temperature = _param(temperature, B, torch.float32, dev, "temperature")
    top_k = _param(top_k, B, torch.int32, dev, "top_k")
    top_p = _param(top_p, B, torch.float32, dev, "top_p")
    min_p = _param(min_p, B, torch.float32, dev, "min_p")
    seed = _param(seed, B, torch.int64, dev, "seed")
    step = _param(step, B, torch.int64, dev, "step")
    row_id = _param(row_id, B, torch.int32, dev, "row_id")
    token = torch.empty(B, dtype=torch.int32, device=dev) if token is None else token
    if want_logprob and logprob is None:
        logprob = torch.empty(B, dtype=torch.float32, device=dev)
    row_status = torch.empty(B, dtype=torch.int32, device=dev) if row_status is None else row_status
    if want_stats and stats is None:
        stats = torch.empty((B, 4), dtype=torch.int32, device=dev)
    lib = load()
    need = int(lib.vsamp_sample_workspace_size(_dtype_code(logits), B, V))
    if workspace is None:
        workspace = sample_workspace(dev, need, stream)
    st = lib.vsamp_sample_ws(
        logits.data_ptr(), _dtype_code(logits), B, V, ld, _ptr(temperature, torch.float32, dev, B, "temperature"),
        _ptr(top_k, torch.int32, dev, B, "top_k"), _ptr(top_p, torch.float32, dev, B, "top_p"),
        _ptr(min_p, torch.float32, dev, B, "min_p"), _ptr(seed, torch.int64, dev, B, "seed"),
        _ptr(step, torch.int64, dev, B, "step"), _ptr(row_id, torch.int32, dev, B, "row_id"),
        _ptr(token, torch.int32, dev, B, "token"), _ptr(logprob, torch.float32, dev, B, "logprob"),
        _ptr(row_status, torch.int32, dev, B, "row_status"), _ptr(stats, torch.int32, dev, 4 * B, "stats"),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "vsamp_sample_ws")
    return token, logprob, row_status, stats


def vsamp_sample_static(logits, temperature=None, top_k=None, top_p=None, min_p=None, seed=None, step=None,
                        row_id=None, V=None, token=None, logprob=None, row_status=None, stats=None,
                        want_logprob=True, want_stats=False, stream=None):
    """vsamp_sample_ws on the library's fixed scratch array (no allocation by the library; calls that
    overlap on one device race). Returns (token, logprob or None, row_status, stats or None)."""
    B, V, ld = _rows(logits, V)
    dev = logits.device
    temperature = _param(temperature, B, torch.float32, dev, "temperature")
    top_k = _param(top_k, B, torch.int32, dev, "top_k")
    top_p = _param(top_p, B, torch.float32, dev, "top_p")
    min_p = _param(min_p, B, torch.float32, dev, "min_p")
    seed = _param(seed, B, torch.int64, dev, "seed")
    step = _param(step, B, torch.int64, dev, "step")
    row_id = _param(row_id, B, torch.int32, dev, "row_id")
    token = torch.empty(B, dtype=torch.int32, device=dev) if token is None else token
    if want_logprob and logprob is None:
        logprob = torch.empty(B, dtype=torch.float32, device=dev)
    row_status = torch.empty(B, dtype=torch.int32, device=dev) if row_status is None else row_status
    if want_stats and stats is None:
        stats = torch.empty((B, 4), dtype=torch.int32, device=dev)
    st = load().vsamp_sample_static(
        logits.data_ptr(), _dtype_code(logits), B, V, ld, _ptr(temperature, torch.float32, dev, B, "temperature"),
        _ptr(top_k, torch.int32, dev, B, "top_k"), _ptr(top_p, torch.float32, dev, B, "top_p"),
        _ptr(min_p, torch.float32, dev, B, "min_p"), _ptr(seed, torch.int64, dev, B, "seed"),
        _ptr(step, torch.int64, dev, B, "step"), _ptr(row_id, torch.int32, dev, B, "row_id"),
        _ptr(token, torch.int32, dev, B, "token"), _ptr(logprob, torch.float32, dev, B, "logprob"),
        _ptr(row_status, torch.int32, dev, B, "row_status"), _ptr(stats, torch.int32, dev, 4 * B, "stats"),
        _stream(stream))
    _check(st, "vsamp_sample_static")
    return token, logprob, row_status, stats


def vsamp_logprob(logits, token, temperature=None, row_max=None, row_logsum=None, V=None, out=None,
                  row_status=None, stream=None):
    """min((x_t - max)/T - log S, 0) per row. Returns (logprob, row_status)."""
    B, V, ld = _rows(logits, V)
    dev = logits.device
    temperature = _param(temperature, B, torch.float32, dev, "temperature")
    token = _param(token, B, torch.int32, dev, "token")
    out = torch.empty(B, dtype=torch.float32, device=dev) if out is None else out
    row_status = torch.empty(B, dtype=torch.int32, device=dev) if row_status is None else row_status
    st = load().vsamp_logprob(
        logits.data_ptr(), _dtype_code(logits), B, V, ld, _ptr(temperature, torch.float32, dev, B, "temperature"),
        _ptr(token, torch.int32, dev, B, "token"), _ptr(row_max, torch.float32, dev, B, "row_max"),
        _ptr(row_logsum, torch.float32, dev, B, "row_logsum"), _ptr(out, torch.float32, dev, B, "out"),
        _ptr(row_status, torch.int32, dev, B, "row_status"), _stream(stream))
    _check(st, "vsamp_logprob")
    return out, row_status


def vsamp_topn_logprobs(logits, n, temperature=None, V=None, row_max=None, row_logsum=None, out_idx=None,
                        out_lp=None, row_status=None, stream=None):
    """The n most probable tokens per row by (logit desc, index asc) with their log-probabilities.
    Returns (out_idx [B, n] int32, out_lp [B, n] fp32, row_max, row_logsum, row_status)."""
    B, V, ld = _rows(logits, V)
    dev = logits.device
    n = int(n)
    temperature = _param(temperature, B, torch.float32, dev, "temperature")
    row_max = torch.empty(B, dtype=torch.float32, device=dev) if row_max is None else row_max
    row_logsum = torch.empty(B, dtype=torch.float32, device=dev) if row_logsum is None else row_logsum
    out_idx = torch.empty((B, max(n, 1)), dtype=torch.int32, device=dev) if out_idx is None else out_idx
    out_lp = torch.empty((B, max(n, 1)), dtype=torch.float32, device=dev) if out_lp is None else out_lp
    row_status = torch.empty(B, dtype=torch.int32, device=dev) if row_status is None else row_status
    st = load().vsamp_topn_logprobs(
        logits.data_ptr(), _dtype_code(logits), B, V, ld, _ptr(temperature, torch.float32, dev, B, "temperature"),
        n, _ptr(row_max, torch.float32, dev, B, "row_max"), _ptr(row_logsum, torch.float32, dev, B, "row_logsum"),
        _ptr(out_idx, torch.int32, dev, B * max(n, 1), "out_idx"),
        _ptr(out_lp, torch.float32, dev, B * max(n, 1), "out_lp"),
        _ptr(row_status, torch.int32, dev, B, "row_status"), _stream(stream))
    _check(st, "vsamp_topn_logprobs")
    return out_idx, out_lp, row_max, row_logsum, row_status


def vsamp_kept_logprob(logits, token, temperature=None, top_k=None, top_p=None, min_p=None, V=None, out=None,
                       row_status=None, stream=None):
    """Log-probability of token[r] renormalised over the kept set of the row's cut (-inf outside it).
    Returns (out [B] fp32, row_status)."""
    B, V, ld = _rows(logits, V)
    dev = logits.device
    temperature = _param(temperature, B, torch.float32, dev, "temperature")
    top_k = _param(top_k, B, torch.int32, dev, "top_k")
    top_p = _param(top_p, B, torch.float32, dev, "top_p")
    min_p = _param(min_p, B, torch.float32, dev, "min_p")
    token = _param(token, B, torch.int32, dev, "token")
    out = torch.empty(B, dtype=torch.float32, device=dev) if out is None else out
    row_status = torch.empty(B, dtype=torch.int32, device=dev) if row_status is None else row_status
    st = load().vsamp_kept_logprob(
        logits.data_ptr(), _dtype_code(logits), B, V, ld, _ptr(temperature, torch.float32, dev, B, "temperature"),
        _ptr(top_k, torch.int32, dev, B, "top_k"), _ptr(top_p, torch.float32, dev, B, "top_p"),
        _ptr(min_p, torch.float32, dev, B, "min_p"), _ptr(token, torch.int32, dev, B, "token"),
        _ptr(out, torch.float32, dev, B, "out"), _ptr(row_status, torch.int32, dev, B, "row_status"),
        _stream(stream))
    _check(st, "vsamp_kept_logprob")
    return out, row_status


# ------------------------------------------------------------------------------------------------
# vocabulary-sharded sampling: rank-local summaries, rank-ordered exchange, the owned merge
# ------------------------------------------------------------------------------------------------
PIECE_REC_BYTES = 32
SHARD_WIN_BYTES = 16


def shard_bounds(V: int, R: int, dtype=torch.bfloat16, align_to_pieces: bool = True):
    """Split [0, V) into R contiguous shards in rank order: [(v0, V_r)]. With align_to_pieces every boundary is a
    multiple of the 4 KB piece (2048 bf16 or 1024 fp32 logits), which makes the merged outputs bit-identical to the
    unsharded streaming sampler; otherwise boundaries are multiples of the 16-byte vector (8 bf16 or 4 fp32)."""
    if R <= 0 or V <= 0:
        raise ValueError("V and R must be positive")
    unit = (2048 if dtype == torch.bfloat16 else 1024) if align_to_pieces else (8 if dtype == torch.bfloat16 else 4)
    units = -(-V // unit)
    out, start = [], 0
    for r in range(R):
        end = min(V, (units * (r + 1) // R) * unit)
        out.append((start, max(0, end - start)))
        start = end
    if any(n <= 0 for _, n in out):
        raise ValueError(f"V = {V} is too short for {R} shards of whole {unit}-logit units")
    return out


def shard_record_slots(bounds, dtype=torch.bfloat16) -> int:
    """NP: the record slots per row every shard writes (the most pieces of any shard)."""
    dt = VSAMP_F32 if dtype == torch.float32 else VSAMP_BF16
    return max(int(load().vsamp_shard_pieces(dt, n)) for _, n in bounds)


def vsamp_shard_partial(logits_shard, v0: int, NP: int, temperature=None, seed=None, step=None, row_id=None,
                        target=None, recs=None, win=None, workspace=None, stream=None):
    """Rank-local summaries of one vocabulary shard [B, V_r] starting at token v0: (recs [B, NP, 32] uint8,
    win [B, 16] uint8), as vsamp_piece_rec / vsamp_shard_win bytes."""
    B, Vr, ld = _rows(logits_shard, None)
    dev = logits_shard.device
    dt = _dtype_code(logits_shard)
    temperature = _param(temperature, B, torch.float32, dev, "temperature")
    seed = _param(seed, B, torch.int64, dev, "seed")
    step = _param(step, B, torch.int64, dev, "step")
    row_id = _param(row_id, B, torch.int32, dev, "row_id")
    target = _param(target, B, torch.int32, dev, "target")
    lib = load()
    recs = torch.empty((B, int(NP), PIECE_REC_BYTES), dtype=torch.uint8, device=dev) if recs is None else recs
    win = torch.empty((B, SHARD_WIN_BYTES), dtype=torch.uint8, device=dev) if win is None else win
    need = int(lib.vsamp_shard_workspace_size(dt, B, Vr))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    st = lib.vsamp_shard_partial(
        logits_shard.data_ptr(), dt, B, Vr, ld, int(v0), int(NP), _ptr(temperature, torch.float32, dev, B, "temperature"),
        _ptr(seed, torch.int64, dev, B, "seed"), _ptr(step, torch.int64, dev, B, "step"),
        _ptr(row_id, torch.int32, dev, B, "row_id"), _ptr(target, torch.int32, dev, B, "target"),
        _ptr(recs, torch.uint8, dev, B * int(NP) * PIECE_REC_BYTES, "recs"),
        _ptr(win, torch.uint8, dev, B * SHARD_WIN_BYTES, "win"), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "vsamp_shard_partial")
    return recs, win


def vsamp_shard_merge(recs, wins, V: int, temperature=None, seed=None, step=None, row_id=None,
                      want_target=False, stream=None):
    """The owned merge of rank-ordered records recs [R, B, NP, 32] and wins [R, B, 16] (uint8). Returns
    (row_max, row_logsum, token, logprob, target_logprob or None, row_status)."""
    if recs.dim() != 4 or wins.dim() != 3 or recs.shape[:2] != wins.shape[:2]:
        raise ValueError("recs must be [R, B, NP, 32] and wins [R, B, 16]")
    R, B, NP = int(recs.shape[0]), int(recs.shape[1]), int(recs.shape[2])
    dev = recs.device
    temperature = _param(temperature, B, torch.float32, dev, "temperature")
    seed = _param(seed, B, torch.int64, dev, "seed")
    step = _param(step, B, torch.int64, dev, "step")
    row_id = _param(row_id, B, torch.int32, dev, "row_id")
    f32 = lambda: torch.empty(B, dtype=torch.float32, device=dev)
    row_max, row_logsum, logprob = f32(), f32(), f32()
    target_lp = f32() if want_target else None
    token = torch.empty(B, dtype=torch.int32, device=dev)
    row_status = torch.empty(B, dtype=torch.int32, device=dev)
    st = load().vsamp_shard_merge(
        _ptr(recs.contiguous(), torch.uint8, dev, None, "recs"), _ptr(wins.contiguous(), torch.uint8, dev, None, "wins"),
        R, B, NP, int(V), _ptr(temperature, torch.float32, dev, B, "temperature"), _ptr(seed, torch.int64, dev, B, "seed"),
        _ptr(step, torch.int64, dev, B, "step"), _ptr(row_id, torch.int32, dev, B, "row_id"),
        row_max.data_ptr(), row_logsum.data_ptr(), token.data_ptr(), logprob.data_ptr(),
        0 if target_lp is None else target_lp.data_ptr(), row_status.data_ptr(), _stream(stream))
    _check(st, "vsamp_shard_merge")
    return row_max, row_logsum, token, logprob, target_lp, row_status


def gather_shard_records(recs, win, group=None):
    """The rank-ordered exchange: all-gather this rank's recs [B, NP, 32] and win [B, 16] into [R, B, NP, 32] and
    [R, B, 16] in rank order, with no reduction in transit (torch.distributed; any backend)."""
    import torch.distributed as dist

    R = dist.get_world_size(group)
    # concatenated along the first dimension (the form every backend accepts), then viewed rank-major
    out_r = torch.empty((R * recs.shape[0],) + tuple(recs.shape[1:]), dtype=recs.dtype, device=recs.device)
    out_w = torch.empty((R * win.shape[0],) + tuple(win.shape[1:]), dtype=win.dtype, device=win.device)
    dist.all_gather_into_tensor(out_r, recs.contiguous(), group=group)
    dist.all_gather_into_tensor(out_w, win.contiguous(), group=group)
    return out_r.view((R,) + tuple(recs.shape)), out_w.view((R,) + tuple(win.shape))


def vsamp_sample_sharded(logits, R: int, temperature=None, seed=None, step=None, row_id=None, target=None,
                         align_to_pieces: bool = True, stream=None):
    """R vocabulary shards of one device's [B, V] logits, each summarised by vsamp_shard_partial into its slice of
    the rank-ordered record arrays, then vsamp_shard_merge. Returns (row_max, row_logsum, token, logprob,
    target_logprob or None, row_status)."""
    B, V, _ = _rows(logits, None)
    bounds = shard_bounds(V, R, logits.dtype, align_to_pieces)
    NP = shard_record_slots(bounds, logits.dtype)
    dev = logits.device
    recs = torch.empty((R, B, NP, PIECE_REC_BYTES), dtype=torch.uint8, device=dev)
    wins = torch.empty((R, B, SHARD_WIN_BYTES), dtype=torch.uint8, device=dev)
    for r, (v0, n) in enumerate(bounds):
        vsamp_shard_partial(logits[:, v0:v0 + n], v0, NP, temperature=temperature, seed=seed, step=step,
                            row_id=row_id, target=target, recs=recs[r], win=wins[r], stream=stream)
    return vsamp_shard_merge(recs, wins, V, temperature=temperature, seed=seed, step=step, row_id=row_id,
                             want_target=target is not None, stream=stream)
