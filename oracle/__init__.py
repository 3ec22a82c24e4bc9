"""fp64 CPU oracle for grouped-query attention decode.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` import this package.
It shares no code with ``gqa_decode_blackwell_gb300`` and never imports it.

The arithmetic lives in ``gqa_oracle.c`` (plain C, fp64, one thread per row
range); this module only compiles it with gcc and marshals arrays through
ctypes.  What each function computes, and which passage of the pages it
follows, is written at the top of ``gqa_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_LIB = os.path.join(_HERE, "libgqa_oracle.so")
_lock = threading.Lock()
_default = None


class _Shape(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int),
        ("q_tokens", ctypes.c_int),
        ("q_heads", ctypes.c_int),
        ("kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("max_seqlen", ctypes.c_int),
        ("scale", ctypes.c_double),
        ("causal", ctypes.c_int),
        ("in_fp16", ctypes.c_int),
    ]


def build(out_path: str = _LIB, mutant: int = 0) -> str:
    """Compile the oracle (or a mutant with one planted mistake) with gcc."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", out_path, "-lm"]
    subprocess.run(cmd, check=True)
    return out_path


def _np_u16(t):
    """Raw bf16 / fp16 bit patterns of a CPU tensor / array, as a contiguous uint16 array."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch

    assert t.dtype in (torch.bfloat16, torch.float16), "the oracle takes the exact bf16 or fp16 inputs"
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _is_fp16(t):
    import torch

    return (not isinstance(t, np.ndarray)) and t.dtype == torch.float16


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class Oracle:
    """ctypes handle on one build of ``gqa_oracle.c``."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.gqa_oracle_decode.restype = ctypes.c_int
        lib.gqa_oracle_decode.argtypes = [
            ctypes.POINTER(_Shape), ctypes.POINTER(ctypes.c_uint16), ctypes.POINTER(ctypes.c_uint16),
            ctypes.POINTER(ctypes.c_uint16), ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
            ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
            ctypes.c_int,
        ]
        lib.gqa_oracle_combine.restype = ctypes.c_int
        lib.gqa_oracle_combine.argtypes = [
            ctypes.c_int, ctypes.c_long, ctypes.c_int, ctypes.POINTER(ctypes.c_double),
            ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
        ]
        lib.gqa_oracle_elem.restype = ctypes.c_double
        lib.gqa_oracle_elem.argtypes = [ctypes.c_int, ctypes.c_uint16]
        self._lib = lib
        self.path = path

    def elem(self, bits: int, fp16: bool) -> float:
        """The value the oracle reads for one 16-bit input pattern."""
        return float(self._lib.gqa_oracle_elem(int(bool(fp16)), int(bits)))

    def decode(self, q, k, v, seqlens, *, scale=None, causal=False, pos_begin=None, pos_end=None,
               nthreads=None):
        """Exact attention per (b, t, hq) row.

        q: bf16 or fp16 [B, nq, Hq, d]; k, v: the same type, [B, S_max, Hkv, d];
        seqlens: int [B].
        pos_begin / pos_end: optional int [B] bounds on key positions (a split).
        Returns (out float64 [B, nq, Hq, d], lse float64 [B, nq, Hq]).
        """
        in_fp16 = _is_fp16(q)
        assert _is_fp16(k) == in_fp16 and _is_fp16(v) == in_fp16, "q, k and v share one element type"
        qa, ka, va = _np_u16(q), _np_u16(k), _np_u16(v)
        B, nq, Hq, d = qa.shape
        Bk, S_max, Hkv, dk = ka.shape
        assert va.shape == ka.shape and Bk == B and dk == d
        sl = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32).reshape(B))
        sh = _Shape(B, nq, Hq, Hkv, d, S_max, float(1.0 / np.sqrt(d) if scale is None else scale),
                    int(bool(causal)), int(in_fp16))
        pb = None if pos_begin is None else np.ascontiguousarray(np.asarray(pos_begin, dtype=np.int32).reshape(B))
        pe = None if pos_end is None else np.ascontiguousarray(np.asarray(pos_end, dtype=np.int32).reshape(B))
        out = np.empty((B, nq, Hq, d), dtype=np.float64)
        lse = np.empty((B, nq, Hq), dtype=np.float64)
        if nthreads is None:
            nthreads = len(os.sched_getaffinity(0))
        rc = self._lib.gqa_oracle_decode(
            ctypes.byref(sh), _ptr(qa, ctypes.c_uint16), _ptr(ka, ctypes.c_uint16), _ptr(va, ctypes.c_uint16),
            _ptr(sl, ctypes.c_int32), None if pb is None else _ptr(pb, ctypes.c_int32),
            None if pe is None else _ptr(pe, ctypes.c_int32), _ptr(out, ctypes.c_double),
            _ptr(lse, ctypes.c_double), int(nthreads))
        if rc != 0:
            raise ValueError(f"gqa_oracle_decode failed ({rc})")
        return out, lse

    def combine(self, o_part, lse_part):
        """Merge split partials: o_part [S, rows..., d], lse_part [S, rows...]."""
        o = np.ascontiguousarray(np.asarray(o_part, dtype=np.float64))
        l = np.ascontiguousarray(np.asarray(lse_part, dtype=np.float64))
        S = o.shape[0]
        d = o.shape[-1]
        rows = int(np.prod(o.shape[1:-1])) if o.ndim > 2 else 1
        assert l.shape[0] == S and int(np.prod(l.shape[1:])) == rows
        out = np.empty(o.shape[1:], dtype=np.float64)
        lse = np.empty(l.shape[1:], dtype=np.float64)
        rc = self._lib.gqa_oracle_combine(int(S), int(rows), int(d), _ptr(o, ctypes.c_double),
                                          _ptr(l, ctypes.c_double), _ptr(out, ctypes.c_double),
                                          _ptr(lse, ctypes.c_double))
        if rc != 0:
            raise ValueError(f"gqa_oracle_combine failed ({rc})")
        return out, lse


def load() -> Oracle:
    """The oracle built from the unmodified source (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            if not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
                build(_LIB)
            _default = Oracle(_LIB)
        return _default


def decode(*args, **kwargs):
    return load().decode(*args, **kwargs)


def combine(*args, **kwargs):
    return load().combine(*args, **kwargs)


def split_ranges(seqlens, num_splits, block=128, min_blocks=1):
    """Key-position ranges of the documented contiguous split partition.

    Sequence b has nblk = ceil(L_b / block) blocks and
    splits_b = clamp(ceil(nblk / min_blocks), 1, num_splits) splits; split s
    covers blocks [s*nblk // splits_b, (s+1)*nblk // splits_b) (empty for
    s >= splits_b).  Returns int32 arrays begin, end of shape [num_splits, B]
    in key positions.
    """
    sl = np.asarray(seqlens, dtype=np.int64)
    B = sl.shape[0]
    begin = np.zeros((num_splits, B), dtype=np.int32)
    end = np.zeros((num_splits, B), dtype=np.int32)
    for b in range(B):
        L = max(int(sl[b]), 0)
        nblk = (L + block - 1) // block
        splits = min(max((nblk + min_blocks - 1) // min_blocks, 1), num_splits)
        for s in range(num_splits):
            if s < splits:
                b0 = s * nblk // splits
                b1 = (s + 1) * nblk // splits
                begin[s, b] = b0 * block
                end[s, b] = min(b1 * block, L)
            else:
                begin[s, b] = 0
                end[s, b] = 0
    return begin, end
