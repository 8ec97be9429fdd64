"""Randomized parity: merge, local and fused top-K on seeded random shapes.

Shapes, score distributions, padding fractions and shard layouts are drawn
from one seeded generator, so every run checks the same cases; each draws a
fresh problem, runs the CUDA path and compares every output row bit for bit
with the oracle.  Covers every kernel instantiation and
the fallback's shorter ways (padding-heavy merge rows, masked logit rows).
"""
import numpy as np
import pytest

import oracle
import workloads
from tests import helpers

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import sparse_attention_indexer_stable_gb300 as dk  # noqa: E402

MODES = ["normal", "bf16", "ties", "const", "zeros", "neginf", "wide", "cluster", "narrow"]
N_CASES = 300


def _bits(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def _case(rng):
    kind = str(rng.choice(["merge", "merge", "local", "fused"]))
    if kind == "merge":
        dcp = int(rng.integers(1, 9))
        K = int(rng.choice([int(rng.integers(1, 300)), 4 * int(rng.integers(1, 1025)), 2048, 4096]))
        if dcp * K > dk.DCP_MAX_CANDIDATES:
            K = max(4, dk.DCP_MAX_CANDIDATES // dcp // 4 * 4)
        T = int(rng.choice([1, 3, 16, 150, 160, 300]))
        mode = str(rng.choice(MODES))
        pad = float(rng.choice([0.0, 0.3, 0.7, 0.9, 0.99]))
        m = workloads.random_merge(int(rng.integers(1 << 30)), T, dcp, K, mode=mode, pad_frac=pad,
                                   with_row_starts=bool(rng.integers(2)))
        return kind, m, None, f"merge T={T} dcp={dcp} K={K} {mode} pad={pad}"
    L = int(rng.choice([60, 1000, 2048, 4096]))
    K = int(rng.choice([64, 200, 1024, 2048]))
    T = int(rng.choice([1, 8, 160, 300]))
    mode = str(rng.choice(["bf16", "normal", "ties", "masked"]))
    layout = str(rng.choice(["contiguous", "interleaved"]))
    if kind == "local":
        x = workloads.random_logits(int(rng.integers(1 << 30)), T, L, mode=mode)
        return kind, (x, K, L, layout), None, f"local T={T} L={L} K={K} {mode} {layout}"
    dcp = int(rng.choice([2, 4]))
    x = np.stack([workloads.random_logits(int(rng.integers(1 << 30)), T, L, mode=mode)
                  for _ in range(dcp)])
    return kind, (x, K, L, layout), None, f"fused T={T} dcp={dcp} L={L} K={K} {mode} {layout}"


def test_randomized_parity():
    rng = np.random.default_rng(20261202)
    bad = []
    for _ in range(N_CASES):
        kind, prob, rows, desc = _case(rng)
        if kind == "merge":
            m = prob
            oi, os_ = dk.merge(torch.from_numpy(m.scores).cuda(), torch.from_numpy(m.ids).cuda(),
                               None if m.row_starts is None else torch.from_numpy(m.row_starts).cuda())
            torch.cuda.synchronize()
            wi, ws = helpers.oracle_merge_all(m)
            gi, gs = oi.cpu().numpy(), os_.cpu().numpy()
        elif kind == "local":
            x, K, L, layout = prob
            s_, i_ = dk.local_topk(torch.from_numpy(x).cuda(), K, 1, 4, L=L, layout=layout)
            torch.cuda.synchronize()
            ws, wi = oracle.local_topk(x, K, 1, 4, L=L, interleaved=layout == "interleaved")
            gi, gs = i_.cpu().numpy(), s_.cpu().numpy()
        else:
            x, K, L, layout = prob
            s_, i_ = dk.fused_topk(torch.from_numpy(x).cuda(), K, L=L, layout=layout)
            torch.cuda.synchronize()
            ws, wi = oracle.fused_topk(x, K, L=L, interleaved=layout == "interleaved")
            gi, gs = i_.cpu().numpy(), s_.cpu().numpy()
        if not (np.array_equal(gi, wi) and np.array_equal(_bits(gs), _bits(ws))):
            bad.append(desc)
    assert not bad, f"{len(bad)} of {N_CASES} cases differ, first: {bad[:5]}"
