"""Pins for the CPU oracle, against facts fixed by the pages and by the
mathematics rather than by the oracle itself:

* hand-worked examples (tests/golden/), derived from the selection rule of
  "[Kernel] Optimize CuTeDSL DCP top-k merge" (Summary) and the row_starts
  of "Reserve the sparse indexer's DCP top-k merge scratch through the
  workspace manager" (Purpose);
* brute force over every K-subset on tiny inputs, with a float-comparison
  order that uses no bit keys;
* permutation invariance over every arrangement of the candidates;
* row independence (the second page's chunking claim);
* the composition identity: per-shard local top-K followed by the merge
  equals the top-K over all shards' logits at once, with contiguous and with
  interleaved shard ids;
* the two shard id layouts give different, hand-worked orders
  (tests/golden/fused_examples.txt);
* a library cross-check: numpy's sort of the same 64-bit keys selects and
  orders the same K winners at full row sizes.

A plausible mistake in the oracle (a missing inversion of negative keys, a
signed instead of unsigned id order, row_starts on padding, a dropped shard,
a transposed rank/row index) fails at least one of these.
"""
import itertools
import math

import numpy as np
import pytest

import oracle
import workloads
from tests import helpers


def _bits(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


@pytest.mark.parametrize("ex", helpers.parse_merge_examples(), ids=lambda e: e["name"])
def test_merge_golden(ex):
    out_ids, out_scores = oracle.merge(ex["scores_in"], ex["ids_in"], ex["rs"])
    assert out_ids[0].tolist() == ex["ids"]
    assert np.array_equal(_bits(out_scores[0]), _bits(np.array(ex["scores"], np.float32)))


@pytest.mark.parametrize("ex", helpers.parse_local_examples(), ids=lambda e: e["name"])
def test_local_golden(ex):
    rs = None if ex["row_starts"] is None else np.array([ex["row_starts"]], np.int32)
    out_scores, out_ids = oracle.local_topk(ex["row"], ex["K"], ex["rank"], ex["dcp"],
                                            L=ex["L"], row_starts=rs,
                                            interleaved=ex["interleaved"])
    assert out_ids[0].tolist() == ex["ids"]
    assert np.array_equal(_bits(out_scores[0]), _bits(np.array(ex["scores"], np.float32)))


@pytest.mark.parametrize("ex", helpers.parse_fused_examples(), ids=lambda e: e["name"])
def test_fused_golden(ex):
    rs = None if ex["row_starts"] is None else np.array([ex["row_starts"]], np.int32)
    out_scores, out_ids = oracle.fused_topk(ex["logits"], ex["K"], row_starts=rs,
                                            interleaved=ex["interleaved"])
    assert out_ids[0].tolist() == ex["ids"]
    assert np.array_equal(_bits(out_scores[0]), _bits(np.array(ex["scores"], np.float32)))


# Values chosen to force ties, +-0, -inf and padding into tiny problems.
POOL = [0.5, 0.5, 0.25, -0.25, 0.0, -0.0, -math.inf, 1.0]


def _tiny_problem(rng, dcp, K, pool):
    n = dcp * K
    scores = np.array([pool[i] for i in rng.integers(0, len(pool), n)], np.float32)
    ids = rng.choice(40, n, replace=False).astype(np.int32)
    pad = rng.random(n) < 0.2
    scores[pad] = -np.inf
    ids[pad] = -1
    return scores.reshape(dcp, 1, K), ids.reshape(dcp, 1, K)


@pytest.mark.parametrize("seed", range(60))
def test_merge_brute_force(seed):
    rng = np.random.default_rng(1000 + seed)
    dcp = int(rng.integers(1, 4))
    K = int(rng.integers(1, 4))
    pool = POOL if seed % 2 else [0.5, 0.25, -1.0]  # 3 distinct values -> heavy ties
    scores, ids = _tiny_problem(rng, dcp, K, pool)
    rs = np.array([int(rng.integers(0, 1000))], np.int32) if seed % 3 == 0 else None
    out_ids, out_scores = oracle.merge(scores, ids, rs)
    cands = [(float(scores[r, 0, k]), int(ids[r, 0, k])) for r in range(dcp) for k in range(K)]
    want = helpers.brute_force_topk(cands, K)
    off = 0 if rs is None else int(rs[0])
    assert out_ids[0].tolist() == [(i if i == -1 else i + off) for _, i in want]
    assert np.array_equal(_bits(out_scores[0]), _bits(np.array([s for s, _ in want], np.float32)))


def test_merge_nan_order():
    """NaNs take the place their bits give them in the score key order (a
    reading: the pages never meet a NaN): sign clear above +inf, sign set
    below -inf and below padding.  Worked by hand for one row, K = 6."""
    bits = np.array([0xFFC00000, 0x3F800000, 0xFF800000, 0x7FC00001, 0xFF800000, 0x7F800000],
                    np.uint32)
    scores = bits.view(np.float32).reshape(1, 1, 6)
    ids = np.array([4, 9, -1, 2, 5, 7], np.int32).reshape(1, 1, 6)
    out_ids, out_scores = oracle.merge(scores, ids)
    # +NaN (2), +inf (7), 1.0 (9), real -inf (5), padding, -NaN (4)
    assert out_ids[0].tolist() == [2, 7, 9, 5, -1, 4]
    assert _bits(out_scores[0]).tolist() == [0x7FC00001, 0x7F800000, 0x3F800000, 0xFF800000,
                                             0xFF800000, 0xFFC00000]


@pytest.mark.parametrize("mode,pad", [("ties", 0.1), ("normal", 0.8), ("zeros", 0.0), ("neginf", 0.3)])
def test_merge_matches_library_sort(mode, pad):
    """The oracle's selection and order against numpy's sort of the same
    64-bit keys (the keys themselves are pinned by the hand-worked examples
    and the float-comparison brute force above): a mistake in the oracle's
    gather, comparator, cut at K or id mapping fails here at full size."""
    m = workloads.random_merge(77, 5, 4, 512, mode=mode, pad_frac=pad, with_row_starts=True)
    out_ids, out_scores = oracle.merge(m.scores, m.ids, m.row_starts)
    bits = _bits(m.scores).astype(np.uint64)
    key32 = np.where(bits >> np.uint64(31), ~bits & np.uint64(0xFFFFFFFF), bits | np.uint64(0x80000000))
    inv = (~m.ids.astype(np.int64)) & 0xFFFFFFFF
    key64 = (key32 << np.uint64(32)) | inv.astype(np.uint64)
    for t in range(m.T):
        k = key64[:, t, :].reshape(-1)
        order = np.argsort(k, kind="stable")[::-1][: m.K]
        ids = m.ids[:, t, :].reshape(-1)[order].astype(np.int64)
        want_ids = np.where(ids == -1, -1, ids + int(m.row_starts[t]))
        want_scores = m.scores[:, t, :].reshape(-1)[order]
        assert out_ids[t].tolist() == want_ids.tolist()
        assert np.array_equal(_bits(out_scores[t]), _bits(want_scores))


@pytest.mark.parametrize("seed", range(6))
def test_merge_permutation_invariance(seed):
    rng = np.random.default_rng(2000 + seed)
    dcp, K = (2, 3) if seed % 2 == 0 else (3, 2)
    scores, ids = _tiny_problem(rng, dcp, K, [0.5, 0.25, -0.0, 0.0])
    flat_s, flat_i = scores.ravel(), ids.ravel()
    ref = oracle.merge(scores, ids)
    for perm in itertools.permutations(range(dcp * K)):
        p = np.array(perm)
        got = oracle.merge(flat_s[p].reshape(dcp, 1, K), flat_i[p].reshape(dcp, 1, K))
        assert np.array_equal(got[0], ref[0])
        assert np.array_equal(_bits(got[1]), _bits(ref[1]))


@pytest.mark.parametrize("seed", range(40))
def test_local_brute_force(seed):
    rng = np.random.default_rng(3000 + seed)
    L = int(rng.integers(1, 7))
    ld = L + int(rng.integers(0, 3))
    K = int(rng.integers(1, 6))
    dcp = int(rng.integers(1, 4))
    rank = int(rng.integers(0, dcp))
    inter = seed % 2 == 1
    row = np.array([POOL[i] for i in rng.integers(0, len(POOL), ld)], np.float32)[None, :]
    rs = np.array([int(rng.integers(0, 500))], np.int32)
    out_scores, out_ids = oracle.local_topk(row, K, rank, dcp, L=L, row_starts=rs,
                                            interleaved=inter)
    rs0 = int(rs[0])
    cands = [(float(row[0, c]), rs0 + (c * dcp + rank if inter else rank * L + c))
             for c in range(L)]
    want = helpers.brute_force_topk(cands, min(K, L)) + [(-math.inf, -1)] * max(0, K - L)
    assert out_ids[0].tolist() == [i for _, i in want]
    assert np.array_equal(_bits(out_scores[0]), _bits(np.array([s for s, _ in want], np.float32)))


def test_rows_are_independent():
    """Row t's result depends only on row t (chunking cannot change it)."""
    m = workloads.random_merge(7, T=9, dcp=3, K=16, mode="ties", pad_frac=0.1, with_row_starts=True)
    full = oracle.merge(m.scores, m.ids, m.row_starts)
    for t in range(m.T):
        one = oracle.merge(m.scores[:, t:t + 1], m.ids[:, t:t + 1], m.row_starts[t:t + 1])
        assert np.array_equal(one[0][0], full[0][t])
        sub = oracle.merge(m.scores, m.ids, m.row_starts, rows=[t])
        assert np.array_equal(sub[0][0], full[0][t])
        assert np.array_equal(_bits(sub[1][0]), _bits(full[1][t]))


@pytest.mark.parametrize("inter", [False, True], ids=["contiguous", "interleaved"])
@pytest.mark.parametrize("mode", ["bf16", "ties", "normal"])
def test_composition_local_then_merge(mode, inter):
    """Every global winner is in its own shard's top-K, and the id map is
    monotone in the column (in both shard layouts), so the merge of the
    per-shard top-K equals the top-K over all shards' logits."""
    dcp, T, L, K = 4, 3, 96, 40
    rng_logits = np.stack([workloads.random_logits(50 + r, T, L, mode=mode) for r in range(dcp)])
    rs = np.array([0, 7, 1000], np.int32)
    loc_s = np.empty((dcp, T, K), np.float32)
    loc_i = np.empty((dcp, T, K), np.int32)
    for r in range(dcp):
        loc_s[r], loc_i[r] = oracle.local_topk(rng_logits[r], K, r, dcp, row_starts=None,
                                               interleaved=inter)
    m_ids, m_scores = oracle.merge(loc_s, loc_i, rs)
    f_scores, f_ids = oracle.fused_topk(rng_logits, K, row_starts=rs, interleaved=inter)
    assert np.array_equal(m_ids, f_ids)
    assert np.array_equal(_bits(m_scores), _bits(f_scores))


@pytest.mark.parametrize("seed", range(12))
def test_fused_equals_brute_force(seed):
    rng = np.random.default_rng(77 + seed)
    dcp = int(rng.integers(1, 4))
    L = int(rng.integers(1, 4))
    K = int(rng.integers(1, 5))
    inter = seed % 2 == 1
    logits = np.array([POOL[i] for i in rng.integers(0, len(POOL), dcp * L)],
                      np.float32).reshape(dcp, 1, L)
    out_scores, out_ids = oracle.fused_topk(logits, K, interleaved=inter)
    cands = [(float(logits[r, 0, c]), c * dcp + r if inter else r * L + c)
             for r in range(dcp) for c in range(L)]
    want = helpers.brute_force_topk(cands, min(K, dcp * L)) + [(-math.inf, -1)] * max(0, K - dcp * L)
    assert out_ids[0].tolist() == [i for _, i in want]
    assert np.array_equal(_bits(out_scores[0]), _bits(np.array([s for s, _ in want], np.float32)))


@pytest.mark.parametrize("name", ["tiny", "decode", "tieheavy"])
def test_invariants_named(name):
    m = workloads.NAMED[name]()
    out_ids, out_scores = oracle.merge(m.scores, m.ids, m.row_starts)
    helpers.check_merge_invariants(m.scores, m.ids, m.row_starts, out_ids, out_scores)
    if name == "tieheavy":
        # rows whose last shard is empty still have 3*K >= K real candidates
        assert np.all(out_ids != -1)


def test_invariants_prefill_sample():
    m = workloads.prefill(T=512)
    rows = [0, 1, 255, 256, 511]
    out_ids, out_scores = oracle.merge(m.scores, m.ids, m.row_starts, rows=rows)
    helpers.check_merge_invariants(m.scores, m.ids, m.row_starts, out_ids, out_scores, rows=rows)


def test_invariant_checker_catches_mistakes():
    """The invariant checker itself rejects plausible wrong outputs."""
    m = workloads.random_merge(5, T=2, dcp=2, K=8, mode="ties")
    out_ids, out_scores = oracle.merge(m.scores, m.ids)
    bad = [out_ids.copy(), out_ids.copy()]
    bad[0][0, [0, 1]] = bad[0][0, [1, 0]]          # swapped order
    bad[1][0, -1] = 10 ** 6                          # an id not among the candidates
    for b in bad:
        with pytest.raises(AssertionError):
            helpers.check_merge_invariants(m.scores, m.ids, None, b, out_scores)
