"""Barrier tests on the race-check build of the library.

The review of "[Kernel] Optimize CuTeDSL DCP top-k merge" reports a race: a
threshold read from shared memory and the shared state reset with no barrier
in between, so late warps read the reset value and drop tied winners.  In the
ordinary build a missing barrier shows only when warp timing happens to
expose it.  The race-check build (compiled with -DDCP_DEBUG_POISON) makes it
show: after every barrier of the row loops the odd warps wait a while, every
reset of shared state is preceded by an overwrite with garbage and a barrier,
and indices taken from shared state are clamped (and the clamp recorded in
the device status word) so garbage cannot fault.  Every kernel and its
fallback paths run here, bit-exact against the oracle, with no clamp
recorded.
"""
import ctypes
import zlib

import numpy as np
import pytest

import oracle
import workloads
from tests import helpers

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import sparse_attention_indexer_stable_gb300 as dk  # noqa: E402
from sparse_attention_indexer_stable_gb300 import _build  # noqa: E402

CLAMP_BIT = 4  # kStatusPoisonClamp


@pytest.fixture(scope="module")
def rlib():
    lib = ctypes.CDLL(_build.build_race_check())
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.dcp_topk_merge.argtypes = [P, P, I, I, I, P, P, P, P, S, P]
    lib.dcp_local_topk_ex.argtypes = [P, I, I, I, I, I, I, P, I, P, P, P]
    lib.dcp_fused_topk_ex.argtypes = [P, I, I, I, I, I, P, I, P, P, P]
    lib.dcp_topk_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    for f in (lib.dcp_topk_merge, lib.dcp_local_topk_ex, lib.dcp_fused_topk_ex,
              lib.dcp_topk_device_status):
        f.restype = I
    return lib


def _status(lib):
    v = ctypes.c_uint(0)
    assert lib.dcp_topk_device_status(ctypes.byref(v)) == 0
    return v.value


def _bits(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def _merge(lib, m):
    s = torch.from_numpy(m.scores).cuda()
    i = torch.from_numpy(m.ids).cuda()
    rs = None if m.row_starts is None else torch.from_numpy(m.row_starts).cuda()
    oi = torch.empty((m.T, m.K), dtype=torch.int32, device="cuda")
    os_ = torch.empty((m.T, m.K), dtype=torch.float32, device="cuda")
    st = lib.dcp_topk_merge(s.data_ptr(), i.data_ptr(), m.T, m.dcp, m.K,
                            None if rs is None else rs.data_ptr(), oi.data_ptr(), os_.data_ptr(),
                            None, 0, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    return oi.cpu().numpy(), os_.cpu().numpy()


def _check_merge(lib, m, what):
    gi, gs = _merge(lib, m)
    wi, ws = helpers.oracle_merge_all(m)
    assert np.array_equal(gi, wi), what
    assert np.array_equal(_bits(gs), _bits(ws)), what
    assert _status(lib) & CLAMP_BIT == 0, f"{what}: an index from shared state was clamped"


@pytest.mark.parametrize("seed", range(24))
def test_race_check_tieheavy(rlib, seed):
    """Ties at the threshold: the case the review's race breaks."""
    _check_merge(rlib, workloads.tieheavy(seed=100 + seed), f"seed {seed}")


@pytest.mark.parametrize("T", [300, 700])
def test_race_check_prefill_slice(rlib, T):
    """Prefill rows: two 512-thread CTAs per SM (300 rows) and the many-row
    merge's four 256-thread CTAs per SM (700 rows), several rows per CTA."""
    _check_merge(rlib, workloads.prefill(T=T), f"prefill {T}")


RACE_CASES = [
    # (T, dcp, K, mode, pad_frac)
    (200, 4, 2048, "bf16", 0.8),      # many rows, fewer real candidates than K: the fallback
    (16, 4, 2048, "normal", 0.8),     # one CTA per row, the same
    (120, 4, 2048, "normal", 0.8),
    (200, 4, 2048, "narrow", 0.0),    # the live set refined on the next key bits
    (8, 4, 2048, "narrow", 0.0),
    (100, 4, 2048, "narrow", 0.0),
    (153, 4, 2048, "cluster", 0.0),   # buckets too large: the radix-select fallback
    (5, 4, 2048, "cluster", 0.0),
    (90, 4, 2048, "cluster", 0.0),
    (16, 4, 2048, "neginf", 0.0),     # real -inf candidates below the winners
    (38, 4, 2048, "bf16", 0.1),
    (50, 4, 2048, "ties", 0.3),
    (8, 8, 2048, "bf16", 0.0),        # 16384 candidates per row
    (16, 4, 2048, "wide", 0.0),
    (300, 4, 2048, "normal", 0.0),    # fp32 scores: 64-bit rank keys
    (170, 2, 1024, "ties", 0.1),      # two 512-thread CTAs per SM
    (3, 4, 4096, "ties", 0.3),        # K up to 4096
    (6, 3, 1001, "ties", 0.1),        # the general path (K not a multiple of 4)
    (160, 4, 2048, "neginf", 0.7),
    # the many-row merge (more than two rows per SM)
    (700, 4, 2048, "bf16", 0.8),      # list sorts of the real candidates, padding after
    (420, 4, 2048, "narrow", 0.0),    # refinement
    (340, 4, 2048, "cluster", 0.0),   # the radix-select fallback
    (400, 4, 2048, "normal", 0.0),    # 64-bit rank keys
    (350, 4, 2048, "neginf", 0.7),    # real -inf winners ranked by id
]


@pytest.mark.parametrize("case", RACE_CASES, ids=lambda c: "-".join(map(str, c)))
def test_race_check_merge_shapes(rlib, case):
    T, dcp, K, mode, pad = case
    m = workloads.random_merge(zlib.crc32(repr(case).encode()) & 0xFFFF, T, dcp, K, mode=mode,
                               pad_frac=pad, with_row_starts=True)
    _check_merge(rlib, m, str(case))


@pytest.mark.parametrize("T,mode", [(160, "masked"), (8, "bf16"), (300, "bf16")])
def test_race_check_local(rlib, T, mode):
    x = workloads.random_logits(77 + T, T, 4096, mode=mode)
    xd = torch.from_numpy(x).cuda()
    K = 2048
    os_ = torch.empty((T, K), dtype=torch.float32, device="cuda")
    oi = torch.empty((T, K), dtype=torch.int32, device="cuda")
    assert rlib.dcp_local_topk_ex(xd.data_ptr(), T, 4096, 4096, K, 1, 4, None, 0, os_.data_ptr(),
                                  oi.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    ws, wi = oracle.local_topk(x, K, 1, 4)
    assert np.array_equal(oi.cpu().numpy(), wi)
    assert np.array_equal(_bits(os_.cpu().numpy()), _bits(ws))
    assert _status(rlib) & CLAMP_BIT == 0


@pytest.mark.parametrize("T,layout", [(8, 0), (64, 1), (200, 0)])
def test_race_check_fused(rlib, T, layout):
    x = workloads.sweep_logits(T)
    xd = torch.from_numpy(x).cuda()
    dcp, _, L = x.shape
    K = 2048
    os_ = torch.empty((T, K), dtype=torch.float32, device="cuda")
    oi = torch.empty((T, K), dtype=torch.int32, device="cuda")
    assert rlib.dcp_fused_topk_ex(xd.data_ptr(), T, dcp, L, L, K, None, layout, os_.data_ptr(),
                                  oi.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    ws, wi = oracle.fused_topk(x, K, interleaved=layout == 1)
    assert np.array_equal(oi.cpu().numpy(), wi)
    assert np.array_equal(_bits(os_.cpu().numpy()), _bits(ws))
    assert _status(rlib) & CLAMP_BIT == 0
