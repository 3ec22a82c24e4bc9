"""Python binding of the GB300 GQA decode library (``include/gqa_decode.h``).

Argument marshalling only: every function below turns PyTorch tensors into
the plain pointers and sizes of the C entry point of the same name and calls
it.  All computation happens in the sm_103a kernels of
``libgqa_decode_sm103.so``; there is no fallback.  If the library has not
been built, the first call raises ``RuntimeError`` (build it with
``gqa_decode_blackwell_gb300.build.build()``).
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from typing import Optional

from .build import HEADER, LIB

GQA_OK = 0
GQA_ERR_INVALID_ARG = 1
GQA_ERR_UNSUPPORTED = 2
GQA_ERR_WORKSPACE = 3
GQA_ERR_CUDA = 4
GQA_ERR_TIMEOUT = 5
GQA_ERR_BAD_SEQLEN = 6
GQA_ERR_BOUNDS = 7
GQA_DTYPE_BF16 = 0
GQA_DTYPE_FP32 = 1
GQA_DTYPE_FP16 = 2
GQA_REDUCE_AUTO = 0
GQA_REDUCE_COMBINE = 1
GQA_REDUCE_CLUSTER = 2
_REDUCTIONS = {"auto": GQA_REDUCE_AUTO, "combine": GQA_REDUCE_COMBINE, "cluster": GQA_REDUCE_CLUSTER}

_lock = threading.Lock()
_lib = None


class GQAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {gqa_status_string(status)} (status {status})")


class gqa_desc_t(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int),
        ("q_tokens", ctypes.c_int),
        ("q_heads", ctypes.c_int),
        ("kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("max_seqlen", ctypes.c_int),
        ("scale", ctypes.c_float),
        ("causal", ctypes.c_int),
        ("out_dtype", ctypes.c_int),
        ("in_dtype", ctypes.c_int),
        ("reduction", ctypes.c_int),
    ]


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB):
                raise RuntimeError(f"GQA decode CUDA library not built ({LIB}); run "
                                   "gqa_decode_blackwell_gb300.build.build() or __graft_entry__.build()")
            _lib = load_library(LIB)
        return _lib


def load_library(path: str) -> ctypes.CDLL:
    """A build of the C library at `path` (say the -DGQA_DEBUG one) with its
    functions' argument and result types declared."""
    L = ctypes.CDLL(path)
    P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    D = ctypes.POINTER(gqa_desc_t)
    L.gqa_decode_workspace_size.argtypes = [D, I]
    L.gqa_decode_workspace_size.restype = SZ
    L.gqa_decode_attn.argtypes = [D, P, P, P, P, P, P, I, P, SZ, P]
    L.gqa_decode_attn.restype = I
    L.gqa_decode_attn_static_workspace.argtypes = [D, P, P, P, P, P, P, I, P]
    L.gqa_decode_attn_static_workspace.restype = I
    L.gqa_decode_attn_split.argtypes = [D, P, P, P, P, P, P, I, P, SZ, P]
    L.gqa_decode_attn_split.restype = I
    L.gqa_decode_attn_merge.argtypes = [D, P, P, I, P, SZ, P]
    L.gqa_decode_attn_merge.restype = I
    L.gqa_decode_splitkv.argtypes = [D, P, P, P, P, I, P, P, P]
    L.gqa_decode_splitkv.restype = I
    L.gqa_decode_combine.argtypes = [P, P, I, I64, I, P, I, P, P]
    L.gqa_decode_combine.restype = I
    L.gqa_decode_get_error.argtypes = [I]
    L.gqa_decode_get_error.restype = I
    L.gqa_status_string.argtypes = [I]
    L.gqa_status_string.restype = ctypes.c_char_p
    L.gqa_decode_plan.argtypes = [D, P, I, I, ctypes.POINTER(I), ctypes.POINTER(I), ctypes.POINTER(I), P,
                                  I64, ctypes.POINTER(I64)]
    L.gqa_decode_plan.restype = I
    L.gqa_decode_selftest_timeout.argtypes = [ctypes.c_uint, P]
    L.gqa_decode_selftest_timeout.restype = I
    return L


def header_functions():
    """Names of the functions ``include/gqa_decode.h`` declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gqa_[a-z_0-9]+)\s*\(", text)))


def _check(status: int, where: str):
    if status != GQA_OK:
        raise GQAError(status, where)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(dtype, allowed):
    import torch

    code = {torch.bfloat16: GQA_DTYPE_BF16, torch.float32: GQA_DTYPE_FP32, torch.float16: GQA_DTYPE_FP16}.get(dtype)
    if code is None or code not in allowed:
        raise ValueError(f"unsupported dtype {dtype}")
    return code


def _reduction_code(reduction) -> int:
    if isinstance(reduction, str):
        if reduction not in _REDUCTIONS:
            raise ValueError(f"reduction must be one of {sorted(_REDUCTIONS)}")
        return _REDUCTIONS[reduction]
    return int(reduction)


def make_desc(q, k_cache, *, scale: float = 0.0, causal: bool = False, out_dtype=None,
              reduction="auto") -> gqa_desc_t:
    """Problem description from q [B, nq, Hq, d] and a cache [B, S_max, Hkv, d]
    (inputs bf16 or fp16; out_dtype fp32 or the inputs' type, the default;
    reduction "auto", "combine" or "cluster", see gqa_reduction_t)."""
    import torch

    B, nq, Hq, d = q.shape
    Bk, s_max, Hkv, dk = k_cache.shape
    if Bk != B or dk != d:
        raise ValueError(f"q {tuple(q.shape)} and cache {tuple(k_cache.shape)} disagree")
    if out_dtype is None:
        out_dtype = q.dtype
    code = _dtype_code(out_dtype, (GQA_DTYPE_BF16, GQA_DTYPE_FP32, GQA_DTYPE_FP16))
    in_code = _dtype_code(q.dtype, (GQA_DTYPE_BF16, GQA_DTYPE_FP16))
    return gqa_desc_t(B, nq, Hq, Hkv, d, s_max, float(scale), int(bool(causal)), code, in_code,
                      _reduction_code(reduction))


def _inputs_ok(q, k_cache, v_cache, seqlens):
    import torch

    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        if t.dtype not in (torch.bfloat16, torch.float16) or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 or fp16 tensor, all three of one type")
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    if seqlens.dtype != torch.int32 or not seqlens.is_contiguous():
        raise ValueError("seqlens must be a contiguous int32 tensor")


def gqa_decode_workspace_size(q, k_cache, num_splits: int = 0, *, causal: bool = False, out_dtype=None,
                              reduction="auto") -> int:
    desc = make_desc(q, k_cache, causal=causal, out_dtype=out_dtype, reduction=reduction)
    return int(lib().gqa_decode_workspace_size(ctypes.byref(desc), int(num_splits)))


def gqa_decode_attn(q, k_cache, v_cache, seqlens, out, lse=None, num_splits: int = 0, workspace=None, *,
                    scale: float = 0.0, causal: bool = False, reduction="auto", stream=None) -> None:
    """Full decode into ``out`` (and ``lse``); see gqa_decode_attn in the C header."""
    _inputs_ok(q, k_cache, v_cache, seqlens)
    desc = make_desc(q, k_cache, scale=scale, causal=causal, out_dtype=out.dtype, reduction=reduction)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().gqa_decode_attn(ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens),
                               _ptr(out), _ptr(lse), int(num_splits), _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc, "gqa_decode_attn")


def gqa_decode_attn_static_workspace(q, k_cache, v_cache, seqlens, out, lse=None, num_splits: int = 0, *,
                                     scale: float = 0.0, causal: bool = False, reduction="auto",
                                     stream=None) -> None:
    """gqa_decode_attn using the library's static device workspace instead of a
    caller-allocated one (for callers that cannot allocate; see the C header)."""
    _inputs_ok(q, k_cache, v_cache, seqlens)
    desc = make_desc(q, k_cache, scale=scale, causal=causal, out_dtype=out.dtype, reduction=reduction)
    rc = lib().gqa_decode_attn_static_workspace(ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                                _ptr(seqlens), _ptr(out), _ptr(lse), int(num_splits),
                                                _stream(stream))
    _check(rc, "gqa_decode_attn_static_workspace")


def gqa_decode_attn_split(q, k_cache, v_cache, seqlens, out, lse=None, num_splits: int = 0, workspace=None, *,
                          scale: float = 0.0, causal: bool = False, reduction="auto", stream=None) -> None:
    """The decode-kernel half of gqa_decode_attn (see the C header)."""
    _inputs_ok(q, k_cache, v_cache, seqlens)
    desc = make_desc(q, k_cache, scale=scale, causal=causal, out_dtype=out.dtype, reduction=reduction)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().gqa_decode_attn_split(ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens),
                                     _ptr(out), _ptr(lse), int(num_splits), _ptr(workspace), ws_bytes,
                                     _stream(stream))
    _check(rc, "gqa_decode_attn_split")


def gqa_decode_attn_merge(q, k_cache, out, lse=None, num_splits: int = 0, workspace=None, *, causal: bool = False,
                          reduction="auto", stream=None) -> None:
    """The combine half of gqa_decode_attn over the workspace of gqa_decode_attn_split."""
    desc = make_desc(q, k_cache, causal=causal, out_dtype=out.dtype, reduction=reduction)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().gqa_decode_attn_merge(ctypes.byref(desc), _ptr(out), _ptr(lse), int(num_splits), _ptr(workspace),
                                     ws_bytes, _stream(stream))
    _check(rc, "gqa_decode_attn_merge")


def gqa_decode_splitkv(q, k_cache, v_cache, seqlens, num_splits: int, o_part, lse_part, *, scale: float = 0.0,
                       causal: bool = False, stream=None) -> None:
    """Per-split partials (o_part fp32 [S, B, nq, Hq, d], lse_part fp32 [S, B, nq, Hq])."""
    _inputs_ok(q, k_cache, v_cache, seqlens)
    desc = make_desc(q, k_cache, scale=scale, causal=causal)
    rc = lib().gqa_decode_splitkv(ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens),
                                  int(num_splits), _ptr(o_part), _ptr(lse_part), _stream(stream))
    _check(rc, "gqa_decode_splitkv")


def gqa_decode_combine(o_part, lse_part, out, lse=None, stream=None) -> None:
    """Merge partials o_part fp32 [S, rows..., d] / lse_part [S, rows...] into out [rows..., d]."""
    import torch

    S, d = o_part.shape[0], o_part.shape[-1]
    rows = lse_part[0].numel()
    code = _dtype_code(out.dtype, (GQA_DTYPE_BF16, GQA_DTYPE_FP32, GQA_DTYPE_FP16))
    rc = lib().gqa_decode_combine(_ptr(o_part), _ptr(lse_part), int(S), int(rows), int(d), _ptr(out), code,
                                  _ptr(lse), _stream(stream))
    _check(rc, "gqa_decode_combine")


def gqa_decode_get_error(clear: bool = True) -> int:
    return int(lib().gqa_decode_get_error(1 if clear else 0))


def gqa_status_string(status: int) -> str:
    try:
        return lib().gqa_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def gqa_decode_plan(desc: gqa_desc_t, seqlens_host, num_splits: int = 0, sm_count: int = 0, max_items=None):
    """Work decomposition as (num_ctas, plan_mode, num_slots, items int32 [n, 8])."""
    import numpy as np

    sl = np.ascontiguousarray(np.asarray(seqlens_host, dtype=np.int32))
    nc, mode, slots = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    n = ctypes.c_int64()
    L = lib()
    rc = L.gqa_decode_plan(ctypes.byref(desc), sl.ctypes.data, int(num_splits), int(sm_count), ctypes.byref(nc),
                           ctypes.byref(mode), ctypes.byref(slots), None, 0, ctypes.byref(n))
    _check(rc, "gqa_decode_plan")
    cap = n.value if max_items is None else min(n.value, max_items)
    items = np.zeros((max(cap, 1), 8), dtype=np.int32)
    rc = L.gqa_decode_plan(ctypes.byref(desc), sl.ctypes.data, int(num_splits), int(sm_count), ctypes.byref(nc),
                           ctypes.byref(mode), ctypes.byref(slots), items.ctypes.data, cap, ctypes.byref(n))
    _check(rc, "gqa_decode_plan")
    return nc.value, mode.value, slots.value, items[:cap]


def gqa_decode_selftest_timeout(timeout_us: int, stream=None) -> None:
    _check(lib().gqa_decode_selftest_timeout(int(timeout_us), _stream(stream)), "gqa_decode_selftest_timeout")


def decode(q, k_cache, v_cache, seqlens, *, num_splits: int = 0, scale: float = 0.0, causal: bool = False,
           out_dtype=None, reduction="auto", stream=None):
    """Allocates out / lse / workspace with torch and calls gqa_decode_attn."""
    import torch

    out_dtype = q.dtype if out_dtype is None else out_dtype
    B, nq, Hq, d = q.shape
    out = torch.empty(B, nq, Hq, d, dtype=out_dtype, device=q.device)
    lse = torch.empty(B, nq, Hq, dtype=torch.float32, device=q.device)
    ws_bytes = gqa_decode_workspace_size(q, k_cache, num_splits, causal=causal, out_dtype=out_dtype,
                                         reduction=reduction)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device) if ws_bytes else None
    gqa_decode_attn(q, k_cache, v_cache, seqlens, out, lse, num_splits, ws, scale=scale, causal=causal,
                    reduction=reduction, stream=stream)
    return out, lse
