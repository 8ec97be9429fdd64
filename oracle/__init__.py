"""CPU oracle for the DCP top-K merge -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library path
(``sparse_attention_indexer_stable_gb300``) never does, and shares no code
with it.

The arithmetic lives in ``dcp_topk_oracle.c`` (plain single-threaded C,
qsort over 64-bit keys); this module compiles it with the host C compiler on
first use and wraps it with numpy arrays.  Every function here is pinned by
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dcp_topk_oracle.c")
_HDR = os.path.join(_HERE, "dcp_topk_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libdcp_topk_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/ (host C compiler, -O2)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        cc = os.environ.get("CC", "gcc")
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call([cc, "-O2", "-std=c99", "-fPIC", "-shared", "-Wall", "-Wextra",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_merge_rows.argtypes = [P, P, I, I, I, P, P, I, P, P]
            lib.oracle_merge.argtypes = [P, P, I, I, I, P, P, P]
            lib.oracle_local_topk.argtypes = [P, I, I, I, I, I, I, P, P, P]
            lib.oracle_fused_topk.argtypes = [P, I, I, I, I, I, P, P, P]
            lib.oracle_local_topk_ids.argtypes = [P, I, I, I, I, I, I, P, I, P, P]
            lib.oracle_fused_topk_ids.argtypes = [P, I, I, I, I, I, P, I, P, P]
            for f in (lib.oracle_merge_rows, lib.oracle_merge, lib.oracle_local_topk,
                      lib.oracle_fused_topk):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def merge(scores, ids, row_starts=None, rows=None):
    """Global top-K per row of rank-major candidates ``(dcp, T, K)``.

    Returns ``(out_ids, out_scores)``, each ``(T, K)`` (or ``(len(rows), K)``
    when ``rows`` selects a subset of rows).
    """
    scores = _c(scores, np.float32)
    ids = _c(ids, np.int32)
    dcp, T, K = scores.shape
    assert ids.shape == scores.shape
    rs = _c(row_starts, np.int32)
    rows = _c(rows, np.int32)
    n = T if rows is None else len(rows)
    out_ids = np.empty((n, K), np.int32)
    out_scores = np.empty((n, K), np.float32)
    rc = _load().oracle_merge_rows(_ptr(scores), _ptr(ids), T, dcp, K, _ptr(rs), _ptr(rows), n,
                                   _ptr(out_ids), _ptr(out_scores))
    if rc != 0:
        raise ValueError(f"oracle_merge_rows failed with {rc}")
    return out_ids, out_scores


def local_topk(logits, K, rank, dcp, L=None, row_starts=None, interleaved=False):
    """One rank's top-K over logits rows ``(T, ld)`` (first ``L`` columns).

    Ids are ``row_starts + rank*L + c`` (contiguous shards) or, with
    ``interleaved``, ``row_starts + c*dcp + rank``.
    Returns ``(out_scores, out_ids)``, each ``(T, K)``.
    """
    logits = _c(logits, np.float32)
    T, ld = logits.shape
    L = ld if L is None else L
    rs = _c(row_starts, np.int32)
    out_scores = np.empty((T, K), np.float32)
    out_ids = np.empty((T, K), np.int32)
    rc = _load().oracle_local_topk_ids(_ptr(logits), T, L, ld, K, rank, dcp, _ptr(rs),
                                       int(bool(interleaved)), _ptr(out_scores), _ptr(out_ids))
    if rc != 0:
        raise ValueError(f"oracle_local_topk_ids failed with {rc}")
    return out_scores, out_ids


def fused_topk(logits, K, L=None, row_starts=None, interleaved=False):
    """Top-K over all shards' logits ``(dcp, T, ld)`` at once, ids as in
    ``local_topk``.

    Returns ``(out_scores, out_ids)``, each ``(T, K)``.
    """
    logits = _c(logits, np.float32)
    dcp, T, ld = logits.shape
    L = ld if L is None else L
    rs = _c(row_starts, np.int32)
    out_scores = np.empty((T, K), np.float32)
    out_ids = np.empty((T, K), np.int32)
    rc = _load().oracle_fused_topk_ids(_ptr(logits), T, dcp, L, ld, K, _ptr(rs),
                                       int(bool(interleaved)), _ptr(out_scores), _ptr(out_ids))
    if rc != 0:
        raise ValueError(f"oracle_fused_topk_ids failed with {rc}")
    return out_scores, out_ids
