"""The merge over shards in separate allocations (dcp_topk_merge_shards):
bit-exact against the oracle run on the same shards stacked rank-major,
in every launch configuration, plus the device-side alignment check.

Reading shards where they lie is the Top-K path of "[DCP][Performance] Add
Shared-DCP peer-addressable decode data paths" (Summary; Top-K performance);
here every shard is a separate buffer on one GPU.
"""
import zlib

import numpy as np
import pytest

import oracle
import workloads
from tests import helpers

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import sparse_attention_indexer_stable_gb300 as dk  # noqa: E402


def _bits(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def _shards(m):
    # one allocation per shard, each (T, K) row-major
    s = [torch.from_numpy(np.ascontiguousarray(m.scores[r])).cuda() for r in range(m.dcp)]
    i = [torch.from_numpy(np.ascontiguousarray(m.ids[r])).cuda() for r in range(m.dcp)]
    return s, i


SHARD_CASES = [
    # (T, dcp, K, mode, pad_frac): the launch configuration they reach
    (16, 4, 2048, "normal", 0.0),     # one 1024-thread CTA per row
    (100, 4, 2048, "normal", 0.0),
    (8, 4, 2048, "ties", 0.3),
    (400, 4, 2048, "bf16", 0.0),      # the many-row merge, four CTAs per SM
    (330, 3, 2048, "bf16", 0.8),      # the same, padding-heavy
    (160, 4, 2048, "normal", 0.0),    # two 512-thread CTAs per SM
    (200, 2, 1024, "ties", 0.1),      # two 512-thread CTAs per SM
    (5, 3, 1001, "normal", 0.1),      # K not a multiple of 4: the general path
    (3, 8, 2048, "normal", 0.0),      # 16384 candidates per row
    (4, 4, 4096, "bf16", 0.0),        # K up to 4096
]


@pytest.mark.parametrize("case", SHARD_CASES, ids=lambda c: "-".join(map(str, c)))
def test_merge_shards_matches_oracle(case):
    T, dcp, K, mode, pad = case
    m = workloads.random_merge(zlib.crc32(repr(case).encode()) & 0xFFFF, T, dcp, K, mode=mode,
                               pad_frac=pad,
                               with_row_starts=True)
    s, i = _shards(m)
    rs = torch.from_numpy(m.row_starts).cuda()
    oi, os_ = dk.merge_shards(s, i, rs)
    torch.cuda.synchronize()
    wi, ws = helpers.oracle_merge_all(m)
    assert np.array_equal(oi.cpu().numpy(), wi)
    assert np.array_equal(_bits(os_.cpu().numpy()), _bits(ws))


def test_merge_shards_prefill_equals_stacked_merge():
    """The full prefill workload with every shard in its own allocation gives
    the same bits as the merge of the rank-major buffer."""
    m = workloads.prefill()
    s, i = _shards(m)
    rs = torch.from_numpy(m.row_starts).cuda()
    oi, os_ = dk.merge_shards(s, i, rs)
    ri, rsc = dk.merge(torch.from_numpy(m.scores).cuda(), torch.from_numpy(m.ids).cuda(), rs)
    torch.cuda.synchronize()
    assert torch.equal(oi, ri) and torch.equal(os_.view(torch.int32), rsc.view(torch.int32))


def test_merge_shards_graph_replay_repointed():
    """Captured once, replayed after the pointer arrays are rewritten to other
    shards: the replay merges the new shards."""
    m1 = workloads.decode(seed=31)
    m2 = workloads.tieheavy(seed=32)
    s1, i1 = _shards(m1)
    s2, i2 = _shards(m2)
    ps = torch.empty(m1.dcp, dtype=torch.int64, device="cuda")
    pi = torch.empty(m1.dcp, dtype=torch.int64, device="cuda")
    oi = torch.empty((m1.T, m1.K), dtype=torch.int32, device="cuda")
    os_ = torch.empty((m1.T, m1.K), dtype=torch.float32, device="cuda")
    dk.merge_shards(s1, i1, out_ids=oi, out_scores=os_, pointer_arrays=(ps, pi))  # first call
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dk.dcp_topk_merge_shards(ps.data_ptr(), pi.data_ptr(), m1.T, m1.dcp, m1.K, None,
                                 oi.data_ptr(), os_.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    ps.copy_(torch.tensor([x.data_ptr() for x in s2], dtype=torch.int64))
    pi.copy_(torch.tensor([x.data_ptr() for x in i2], dtype=torch.int64))
    g.replay()
    torch.cuda.synchronize()
    wi, ws = oracle.merge(m2.scores, m2.ids)
    assert np.array_equal(oi.cpu().numpy(), wi)
    assert np.array_equal(_bits(os_.cpu().numpy()), _bits(ws))


@pytest.mark.parametrize("T", [16, 300, 400])
def test_merge_shards_misaligned_is_reported(T):
    """A shard 4 bytes off a 16-byte boundary (K % 4 == 0): the kernel checks
    the pointers before reading any shard, reports
    DCP_DEVICE_BAD_SHARD_ALIGNMENT and fills the rows with the unwritten
    sentinel; the context stays usable."""
    assert dk.dcp_topk_device_status() == 0
    m = workloads.decode(seed=33, T=T)
    s, i = _shards(m)
    buf = torch.empty(m.T * m.K + 4, dtype=torch.float32, device="cuda")
    view = buf[1:1 + m.T * m.K].view(m.T, m.K)
    view.copy_(s[1])
    s[1] = view  # data_ptr() is 4 bytes past a 16-byte boundary
    oi, os_ = dk.merge_shards(s, i)
    torch.cuda.synchronize()
    assert dk.dcp_topk_device_status() == dk.DCP_DEVICE_BAD_SHARD_ALIGNMENT
    assert torch.all(oi == dk.DCP_ID_UNWRITTEN)
    assert torch.all(torch.isnan(os_))
    # the device still computes correctly afterwards
    oi, os_ = dk.merge_shards(*_shards(m))
    torch.cuda.synchronize()
    wi, ws = oracle.merge(m.scores, m.ids)
    assert np.array_equal(oi.cpu().numpy(), wi)
    assert dk.dcp_topk_device_status() == 0
