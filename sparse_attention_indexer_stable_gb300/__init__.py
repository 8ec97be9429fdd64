"""GB300-native DCP sparse-indexer top-K: a thin Python binding of the C ABI.

The compute lives in ``_build/libdcp_topk.so`` (CUDA, sm_103a), declared in
``include/dcp_topk.h``.  This module only marshals torch tensors (device
memory) and the current CUDA stream into that ABI; every step of the top-K
runs in the library's kernels.  There is no CPU fallback: if the library is
missing or fails to load, every call raises.

Functions with the ABI's names take raw device pointers and sizes, exactly like
the C functions.  ``merge`` and ``local_topk`` are tensor conveniences on top
of them that check shapes and dtypes and allocate outputs with torch.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

__all__ = [
    "DCP_OK", "DCP_ERR_INVALID", "DCP_ERR_UNSUPPORTED", "DCP_ERR_CUDA",
    "DCP_MAX_K", "DCP_MAX_CANDIDATES", "DcpError",
    "dcp_topk_merge", "dcp_topk_merge_workspace_size", "dcp_local_topk", "dcp_status_string",
    "dcp_topk_merge_shards", "merge_shards", "DCP_DEVICE_BAD_SHARD_ALIGNMENT",
    "dcp_fused_topk", "dcp_topk_device_status", "dcp_topk_selftest_wait_timeout",
    "DCP_DEVICE_COPY_TIMEOUT", "DCP_ID_UNWRITTEN", "fused_topk", "dcp_local_topk_ex", "dcp_fused_topk_ex",
    "DCP_IDS_CONTIGUOUS", "DCP_IDS_INTERLEAVED",
    "merge", "local_topk", "library", "library_path",
]

DCP_OK, DCP_ERR_INVALID, DCP_ERR_UNSUPPORTED, DCP_ERR_CUDA = 0, 1, 2, 3
DCP_MAX_K = 4096
DCP_MAX_CANDIDATES = 16384
DCP_DEVICE_COPY_TIMEOUT = 1
DCP_DEVICE_BAD_SHARD_ALIGNMENT = 2
DCP_ID_UNWRITTEN = -(1 << 31)  # id of an output slot left by a CTA whose copy timed out
DCP_IDS_CONTIGUOUS, DCP_IDS_INTERLEAVED = 0, 1

_lock = threading.Lock()
_lib = None


class DcpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {dcp_status_string(status)} ({status})")


def library_path() -> str:
    return _build.LIB_PATH


def library():
    """Load (building first if missing or stale) the CUDA library."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if _build.is_stale():
                if os.environ.get("DCP_TOPK_NO_BUILD"):
                    raise RuntimeError(f"{path} is missing or stale and DCP_TOPK_NO_BUILD is set")
                _build.build()
            lib = ctypes.CDLL(path)
            P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            lib.dcp_topk_merge.argtypes = [P, P, I, I, I, P, P, P, P, S, P]
            lib.dcp_topk_merge.restype = I
            lib.dcp_topk_merge_shards.argtypes = [P, P, I, I, I, P, P, P, P]
            lib.dcp_topk_merge_shards.restype = I
            lib.dcp_topk_merge_workspace_size.argtypes = [I, I, I, ctypes.POINTER(S)]
            lib.dcp_topk_merge_workspace_size.restype = I
            lib.dcp_local_topk.argtypes = [P, I, I, I, I, I, I, P, P, P, P]
            lib.dcp_local_topk.restype = I
            lib.dcp_fused_topk.argtypes = [P, I, I, I, I, I, P, P, P, P]
            lib.dcp_fused_topk.restype = I
            lib.dcp_local_topk_ex.argtypes = [P, I, I, I, I, I, I, P, I, P, P, P]
            lib.dcp_local_topk_ex.restype = I
            lib.dcp_fused_topk_ex.argtypes = [P, I, I, I, I, I, P, I, P, P, P]
            lib.dcp_fused_topk_ex.restype = I
            lib.dcp_topk_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint)]
            lib.dcp_topk_device_status.restype = I
            lib.dcp_topk_selftest_wait_timeout.argtypes = [ctypes.c_uint, P]
            lib.dcp_topk_selftest_wait_timeout.restype = I
            lib.dcp_status_string.argtypes = [I]
            lib.dcp_status_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


# ------------------------------------------------------------ raw ABI mirrors
def dcp_status_string(status: int) -> str:
    return library().dcp_status_string(int(status)).decode()


def dcp_topk_merge(scores, ids, T, dcp, K, row_starts, out_ids, out_scores,
                   workspace=None, workspace_bytes=0, stream=None) -> int:
    return library().dcp_topk_merge(scores, ids, T, dcp, K, row_starts, out_ids, out_scores,
                                    workspace, workspace_bytes, stream)


def dcp_topk_merge_shards(shard_scores, shard_ids, T, dcp, K, row_starts, out_ids, out_scores,
                          stream=None) -> int:
    return library().dcp_topk_merge_shards(shard_scores, shard_ids, T, dcp, K, row_starts, out_ids,
                                           out_scores, stream)


def dcp_topk_merge_workspace_size(T, dcp, K):
    n = ctypes.c_size_t(0)
    st = library().dcp_topk_merge_workspace_size(T, dcp, K, ctypes.byref(n))
    if st != DCP_OK:
        raise DcpError(st, "dcp_topk_merge_workspace_size")
    return n.value


def dcp_local_topk(logits, T, L, ld, K, rank, dcp, row_starts, out_scores, out_ids,
                   stream=None) -> int:
    return library().dcp_local_topk(logits, T, L, ld, K, rank, dcp, row_starts, out_scores,
                                    out_ids, stream)


def dcp_fused_topk(logits, T, dcp, L, ld, K, row_starts, out_scores, out_ids,
                   stream=None) -> int:
    return library().dcp_fused_topk(logits, T, dcp, L, ld, K, row_starts, out_scores, out_ids,
                                    stream)


def dcp_local_topk_ex(logits, T, L, ld, K, rank, dcp, row_starts, layout, out_scores, out_ids,
                      stream=None) -> int:
    return library().dcp_local_topk_ex(logits, T, L, ld, K, rank, dcp, row_starts, layout,
                                       out_scores, out_ids, stream)


def dcp_fused_topk_ex(logits, T, dcp, L, ld, K, row_starts, layout, out_scores, out_ids,
                      stream=None) -> int:
    return library().dcp_fused_topk_ex(logits, T, dcp, L, ld, K, row_starts, layout, out_scores,
                                       out_ids, stream)


def dcp_topk_device_status():
    """Read and clear the device status word (synchronises the device)."""
    v = ctypes.c_uint(0)
    st = library().dcp_topk_device_status(ctypes.byref(v))
    if st != DCP_OK:
        raise DcpError(st, "dcp_topk_device_status")
    return v.value


def dcp_topk_selftest_wait_timeout(wait_cycles, stream=None) -> int:
    return library().dcp_topk_selftest_wait_timeout(int(wait_cycles), stream)


# ------------------------------------------------------- tensor conveniences
def _torch():
    import torch
    return torch


def _stream_handle(stream, dev=None):
    """The cudaStream_t to launch on: `stream` (a torch stream or a raw
    handle), else the current stream of device index `dev`."""
    if stream is None:
        torch = _torch()
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:  # the handle itself, without a Stream object
            return raw(torch.cuda.current_device() if dev is None else dev)
        stream = torch.cuda.current_stream(dev)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ok(t, dtype, device):
    """Fast form of _check: True when t needs no complaint (device: an index
    or None)."""
    return (t.dtype == dtype and t.is_cuda and t.is_contiguous()
            and (device is None or t.get_device() == device))


def _check(t, name, dtype, device):
    torch = _torch()
    if isinstance(t, torch.Tensor) and _ok(t, dtype, device):
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda or (device is not None and t.get_device() != device):
        where = "a CUDA device" if device is None else f"cuda:{device}"
        raise ValueError(f"{name} must be on {where}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _on_device(dev, fn):
    """Run fn with device index dev current (the library works on the
    current device)."""
    torch = _torch()
    if dev == torch.cuda.current_device():
        return fn()
    with torch.cuda.device(dev):
        return fn()


def merge(scores, ids, row_starts=None, out_ids=None, out_scores=None, stream=None):
    """Global top-K of rank-major candidates.

    scores: float32 (dcp, T, K) CUDA tensor; ids: int32 of the same shape;
    row_starts: optional int32 (T,).  Returns (out_ids int32 (T, K),
    out_scores float32 (T, K)).
    """
    torch = _torch()
    _check(scores, "scores", torch.float32, None)
    dev = scores.get_device()
    _check(ids, "ids", torch.int32, dev)
    if scores.dim() != 3 or ids.shape != scores.shape:
        raise ValueError("scores and ids must both be (dcp, T, K)")
    dcp, T, K = scores.shape
    if row_starts is not None:
        _check(row_starts, "row_starts", torch.int32, dev)
        if row_starts.shape != (T,):
            raise ValueError("row_starts must be (T,)")
    if out_ids is None:
        out_ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    if out_scores is None:
        out_scores = torch.empty((T, K), dtype=torch.float32, device=dev)
    _check(out_ids, "out_ids", torch.int32, dev)
    _check(out_scores, "out_scores", torch.float32, dev)
    if out_ids.shape != (T, K) or out_scores.shape != (T, K):
        raise ValueError("outputs must be (T, K)")
    st = _on_device(dev, lambda: library().dcp_topk_merge(
        scores.data_ptr(), ids.data_ptr(), T, dcp, K,
        None if row_starts is None else row_starts.data_ptr(),
        out_ids.data_ptr(), out_scores.data_ptr(), None, 0,
        _stream_handle(stream, dev)))
    if st != DCP_OK:
        raise DcpError(st, "dcp_topk_merge")
    return out_ids, out_scores


def merge_shards(shard_scores, shard_ids, row_starts=None, out_ids=None, out_scores=None,
                 stream=None, pointer_arrays=None):
    """Global top-K of shards held in separate tensors (read in place).

    shard_scores: sequence of dcp float32 (T, K) CUDA tensors; shard_ids: the
    matching int32 (T, K) tensors.  pointer_arrays: optional pair of int64
    CUDA tensors of length dcp to hold the shards' addresses (filled here);
    by default they are allocated per call.  The arrays are read on the
    device, so they must outlive the stream's use of the call.  Returns
    (out_ids int32 (T, K), out_scores float32 (T, K)).
    """
    torch = _torch()
    dcp = len(shard_scores)
    if dcp < 1 or len(shard_ids) != dcp:
        raise ValueError("need the same number (>= 1) of score and id shards")
    _check(shard_scores[0], "shard_scores[0]", torch.float32, None)
    dev = shard_scores[0].get_device()
    T, K = shard_scores[0].shape
    for r in range(dcp):
        _check(shard_scores[r], f"shard_scores[{r}]", torch.float32, dev)
        _check(shard_ids[r], f"shard_ids[{r}]", torch.int32, dev)
        if shard_scores[r].shape != (T, K) or shard_ids[r].shape != (T, K):
            raise ValueError("every shard must be (T, K)")
    if row_starts is not None:
        _check(row_starts, "row_starts", torch.int32, dev)
        if row_starts.shape != (T,):
            raise ValueError("row_starts must be (T,)")
    if out_ids is None:
        out_ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    if out_scores is None:
        out_scores = torch.empty((T, K), dtype=torch.float32, device=dev)
    _check(out_ids, "out_ids", torch.int32, dev)
    _check(out_scores, "out_scores", torch.float32, dev)
    if out_ids.shape != (T, K) or out_scores.shape != (T, K):
        raise ValueError("outputs must be (T, K)")
    if pointer_arrays is None:
        ps = torch.tensor([x.data_ptr() for x in shard_scores], dtype=torch.int64).to(dev)
        pi = torch.tensor([x.data_ptr() for x in shard_ids], dtype=torch.int64).to(dev)
    else:
        ps, pi = pointer_arrays
        ps.copy_(torch.tensor([x.data_ptr() for x in shard_scores], dtype=torch.int64))
        pi.copy_(torch.tensor([x.data_ptr() for x in shard_ids], dtype=torch.int64))
    st = _on_device(dev, lambda: library().dcp_topk_merge_shards(
        ps.data_ptr(), pi.data_ptr(), T, dcp, K,
        None if row_starts is None else row_starts.data_ptr(),
        out_ids.data_ptr(), out_scores.data_ptr(), _stream_handle(stream, dev)))
    if st != DCP_OK:
        raise DcpError(st, "dcp_topk_merge_shards")
    return out_ids, out_scores


def _layout(layout):
    if layout in (DCP_IDS_CONTIGUOUS, "contiguous"):
        return DCP_IDS_CONTIGUOUS
    if layout in (DCP_IDS_INTERLEAVED, "interleaved"):
        return DCP_IDS_INTERLEAVED
    raise ValueError(f"unknown shard id layout {layout!r}")


def local_topk(logits, K, rank, dcp, L=None, row_starts=None, out_scores=None, out_ids=None,
               stream=None, layout="contiguous"):
    """One rank's top-K over its logits rows.

    logits: float32 (T, ld) CUDA tensor with unit column stride (row stride
    ld >= L); the first L columns are the rank's shard.  layout: "contiguous"
    (ids row_starts + rank*L + c) or "interleaved" (row_starts + c*dcp + rank).
    Returns (out_scores float32 (T, K), out_ids int32 (T, K)).
    """
    torch = _torch()
    if not isinstance(logits, torch.Tensor) or logits.dtype != torch.float32 or not logits.is_cuda:
        raise TypeError("logits must be a float32 CUDA tensor")
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be 2-D with unit column stride")
    dev = logits.get_device()
    T = logits.shape[0]
    ld = logits.stride(0) if T > 1 else logits.shape[1]
    L = logits.shape[1] if L is None else int(L)
    if L > logits.shape[1]:
        raise ValueError("L exceeds the logits' columns")
    if row_starts is not None:
        _check(row_starts, "row_starts", torch.int32, dev)
        if row_starts.shape != (T,):
            raise ValueError("row_starts must be (T,)")
    if out_scores is None:
        out_scores = torch.empty((T, K), dtype=torch.float32, device=dev)
    if out_ids is None:
        out_ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    _check(out_scores, "out_scores", torch.float32, dev)
    _check(out_ids, "out_ids", torch.int32, dev)
    if out_ids.shape != (T, K) or out_scores.shape != (T, K):
        raise ValueError("outputs must be (T, K)")
    st = _on_device(dev, lambda: library().dcp_local_topk_ex(
        logits.data_ptr(), T, L, ld, K, rank, dcp,
        None if row_starts is None else row_starts.data_ptr(),
        _layout(layout), out_scores.data_ptr(), out_ids.data_ptr(),
        _stream_handle(stream, dev)))
    if st != DCP_OK:
        raise DcpError(st, "dcp_local_topk_ex")
    return out_scores, out_ids


def fused_topk(logits, K, L=None, row_starts=None, out_scores=None, out_ids=None, stream=None,
               layout="contiguous"):
    """Top-K over all shards' logits at once (local top-K + merge in one pass).

    logits: float32 (dcp, T, ld) CUDA tensor, contiguous in its last two dims;
    the first L columns of each row are candidates.  layout as for
    local_topk.  Returns (out_scores float32 (T, K), out_ids int32 (T, K)).
    """
    torch = _torch()
    if not isinstance(logits, torch.Tensor) or logits.dtype != torch.float32 or not logits.is_cuda:
        raise TypeError("logits must be a float32 CUDA tensor")
    if logits.dim() != 3 or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous (dcp, T, ld) tensor")
    dev = logits.get_device()
    dcp, T, ld = logits.shape
    L = ld if L is None else int(L)
    if L > ld:
        raise ValueError("L exceeds the logits' columns")
    if row_starts is not None:
        _check(row_starts, "row_starts", torch.int32, dev)
        if row_starts.shape != (T,):
            raise ValueError("row_starts must be (T,)")
    if out_scores is None:
        out_scores = torch.empty((T, K), dtype=torch.float32, device=dev)
    if out_ids is None:
        out_ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    _check(out_scores, "out_scores", torch.float32, dev)
    _check(out_ids, "out_ids", torch.int32, dev)
    if out_ids.shape != (T, K) or out_scores.shape != (T, K):
        raise ValueError("outputs must be (T, K)")
    st = _on_device(dev, lambda: library().dcp_fused_topk_ex(
        logits.data_ptr(), T, dcp, L, ld, K,
        None if row_starts is None else row_starts.data_ptr(),
        _layout(layout), out_scores.data_ptr(), out_ids.data_ptr(),
        _stream_handle(stream, dev)))
    if st != DCP_OK:
        raise DcpError(st, "dcp_fused_topk_ex")
    return out_scores, out_ids
