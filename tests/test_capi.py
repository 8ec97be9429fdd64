"""Host-side checks of the C ABI, no GPU needed: the library builds and loads,
exports every function include/dcp_topk.h declares, and rejects bad
arguments before it touches the device."""
import ctypes
import os
import re

import pytest

import sparse_attention_indexer_stable_gb300 as dk
from sparse_attention_indexer_stable_gb300 import _build

HEADERS = [os.path.join(_build.INCLUDE, f) for f in os.listdir(_build.INCLUDE) if f.endswith(".h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([a-z_][a-z0-9_]*)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("dcp_topk_merge", "dcp_topk_merge_workspace_size", "dcp_local_topk",
              "dcp_status_string"):
        assert n in names


@pytest.mark.parametrize("name", declared_functions())
def test_library_exports_declared_symbol(name):
    lib = ctypes.CDLL(dk.library()._name)
    assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_status_strings():
    assert dk.dcp_status_string(dk.DCP_OK) == "DCP_OK"
    assert dk.dcp_status_string(dk.DCP_ERR_INVALID) == "DCP_ERR_INVALID"
    assert dk.dcp_status_string(dk.DCP_ERR_UNSUPPORTED) == "DCP_ERR_UNSUPPORTED"
    assert dk.dcp_status_string(dk.DCP_ERR_CUDA) == "DCP_ERR_CUDA"
    assert dk.dcp_status_string(99) == "DCP_UNKNOWN_STATUS"


def test_workspace_size_is_zero():
    assert dk.dcp_topk_merge_workspace_size(8192, 4, 2048) == 0
    assert dk.dcp_topk_merge_workspace_size(0, 1, 1) == 0
    with pytest.raises(dk.DcpError):
        dk.dcp_topk_merge_workspace_size(-1, 4, 2048)
    with pytest.raises(dk.DcpError):
        dk.dcp_topk_merge_workspace_size(16, 4, 8192)


FAKE = 0x1000  # never dereferenced: every case below fails validation first


@pytest.mark.parametrize("args,want", [
    ((FAKE, FAKE, -1, 4, 16, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, FAKE, 4, 0, 16, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, FAKE, 4, 4, 0, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((None, FAKE, 4, 4, 16, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, None, 4, 4, 16, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, FAKE, 4, 4, 16, None, None, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, FAKE, 4, 4, 16, None, FAKE, None), dk.DCP_ERR_INVALID),
    ((FAKE, FAKE, 4, 1, 4097, None, FAKE, FAKE), dk.DCP_ERR_UNSUPPORTED),
    ((FAKE, FAKE, 4, 5, 4096, None, FAKE, FAKE), dk.DCP_ERR_UNSUPPORTED),
    ((None, None, 0, 4, 16, None, None, None), dk.DCP_OK),  # T == 0 is a no-op
])
def test_merge_argument_errors(args, want):
    assert dk.dcp_topk_merge(*args, None, 0, None) == want


@pytest.mark.parametrize("args,want", [
    ((FAKE, -1, 8, 8, 4, 0, 1, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, 2, 0, 8, 4, 0, 1, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, 2, 8, 7, 4, 0, 1, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, 2, 8, 8, 0, 0, 1, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, 2, 8, 8, 4, 1, 1, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, 2, 8, 8, 4, -1, 2, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, 2, 8, 8, 4, 0, 0, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((None, 2, 8, 8, 4, 0, 1, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, 2, 8, 8, 4, 0, 1, None, None, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, 2, 16385, 16385, 4, 0, 1, None, FAKE, FAKE), dk.DCP_ERR_UNSUPPORTED),
    ((FAKE, 2, 8, 8, 4097, 0, 1, None, FAKE, FAKE), dk.DCP_ERR_UNSUPPORTED),
    ((None, 0, 8, 8, 4, 0, 1, None, None, None), dk.DCP_OK),
])
def test_local_argument_errors(args, want):
    assert dk.dcp_local_topk(*args, None) == want


def test_device_status_rejects_null():
    assert dk.library().dcp_topk_device_status(None) == dk.DCP_ERR_INVALID


@pytest.mark.parametrize("args,want", [
    ((FAKE, -1, 4, 8, 8, 4, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, 2, 0, 8, 8, 4, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, 2, 4, 8, 7, 4, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, 2, 4, 8, 8, 0, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((None, 2, 4, 8, 8, 4, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, 2, 5, 4096, 4096, 4, None, FAKE, FAKE), dk.DCP_ERR_UNSUPPORTED),
    ((FAKE, 2, 4, 8, 8, 4097, None, FAKE, FAKE), dk.DCP_ERR_UNSUPPORTED),
    ((None, 0, 4, 8, 8, 4, None, None, None), dk.DCP_OK),
])
def test_fused_argument_errors(args, want):
    assert dk.dcp_fused_topk(*args, None) == want


@pytest.mark.parametrize("layout,want", [(-1, dk.DCP_ERR_INVALID), (2, dk.DCP_ERR_INVALID)])
def test_layout_argument_errors(layout, want):
    assert dk.dcp_local_topk_ex(FAKE, 2, 8, 8, 4, 0, 1, None, layout, FAKE, FAKE, None) == want
    assert dk.dcp_fused_topk_ex(FAKE, 2, 4, 8, 8, 4, None, layout, FAKE, FAKE, None) == want
    # T == 0 still validates the layout first
    assert dk.dcp_local_topk_ex(None, 0, 8, 8, 4, 0, 1, None, layout, None, None, None) == want


def test_layout_names():
    assert dk._layout("contiguous") == dk.DCP_IDS_CONTIGUOUS
    assert dk._layout("interleaved") == dk.DCP_IDS_INTERLEAVED
    with pytest.raises(ValueError):
        dk._layout("striped")


@pytest.mark.parametrize("args,want", [
    ((FAKE, FAKE, -1, 4, 16, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, FAKE, 4, 0, 16, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, FAKE, 4, 4, 0, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((None, FAKE, 4, 4, 16, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, None, 4, 4, 16, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, FAKE, 4, 4, 16, None, None, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, FAKE, 4, 4, 16, None, FAKE, None), dk.DCP_ERR_INVALID),
    # pointer arrays the device cannot read (here: not memory of any device)
    ((FAKE, FAKE, 4, 4, 16, None, FAKE, FAKE), dk.DCP_ERR_INVALID),
    ((FAKE, FAKE, 4, 1, 4097, None, FAKE, FAKE), dk.DCP_ERR_UNSUPPORTED),
    ((FAKE, FAKE, 4, 5, 4096, None, FAKE, FAKE), dk.DCP_ERR_UNSUPPORTED),
    ((None, None, 0, 4, 16, None, None, None), dk.DCP_OK),  # T == 0 is a no-op
])
def test_merge_shards_argument_errors(args, want):
    assert dk.dcp_topk_merge_shards(*args, None) == want


def test_merge_shards_rejects_host_pointer_arrays():
    """Pointer arrays in ordinary host memory would fault the kernel: the
    call refuses them before launching anything."""
    arr = (ctypes.c_uint64 * 4)(FAKE, FAKE, FAKE, FAKE)
    p = ctypes.addressof(arr)
    assert dk.dcp_topk_merge_shards(p, p, 2, 4, 16, None, FAKE, FAKE, None) == dk.DCP_ERR_INVALID
