"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

The path only compares and copies, so the bar is bit-exact: ids equal and
score bit patterns equal, element by element.  Inputs come from the seeded
generators in ``workloads``; expected values from ``oracle``.
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


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _bits(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def run_merge(m, stream=None):
    out_ids, out_scores = dk.merge(_dev(m.scores), _dev(m.ids),
                                   None if m.row_starts is None else _dev(m.row_starts),
                                   stream=stream)
    torch.cuda.synchronize()
    return out_ids.cpu().numpy(), out_scores.cpu().numpy()


def assert_same(got, want, what=""):
    gi, gs = got
    wi, ws = want
    assert gi.shape == wi.shape, what
    bad = np.argwhere((gi != wi) | (_bits(gs) != _bits(ws)))
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first at {bad[0].tolist()}"


@pytest.mark.parametrize("name", ["tiny", "decode", "tieheavy"])
def test_named_workloads(name):
    m = workloads.NAMED[name]()
    assert_same(run_merge(m), oracle.merge(m.scores, m.ids, m.row_starts), name)


# The hand-worked examples of tests/golden/, run through the CUDA path and
# compared with their worked-out values (not only with the oracle).
@pytest.mark.parametrize("ex", helpers.parse_merge_examples(), ids=lambda e: e["name"])
def test_merge_golden_on_gpu(ex):
    out_ids, out_scores = dk.merge(_dev(ex["scores_in"]), _dev(ex["ids_in"]),
                                   None if ex["rs"] is None else _dev(ex["rs"]))
    torch.cuda.synchronize()
    assert out_ids.cpu().numpy()[0].tolist() == ex["ids"]
    assert np.array_equal(_bits(out_scores.cpu().numpy()[0]), _bits(np.array(ex["scores"], np.float32)))


@pytest.mark.parametrize("ex", helpers.parse_local_examples(), ids=lambda e: e["name"])
def test_local_golden_on_gpu(ex):
    rs = None if ex["row_starts"] is None else _dev(np.array([ex["row_starts"]], np.int32))
    out_scores, out_ids = dk.local_topk(_dev(ex["row"]), ex["K"], ex["rank"], ex["dcp"], L=ex["L"],
                                        row_starts=rs,
                                        layout="interleaved" if ex.get("interleaved") else "contiguous")
    torch.cuda.synchronize()
    assert out_ids.cpu().numpy()[0].tolist() == ex["ids"]
    assert np.array_equal(_bits(out_scores.cpu().numpy()[0]), _bits(np.array(ex["scores"], np.float32)))


@pytest.mark.parametrize("ex", helpers.parse_fused_examples(), ids=lambda e: e["name"])
def test_fused_golden_on_gpu(ex):
    rs = None if ex["row_starts"] is None else _dev(np.array([ex["row_starts"]], np.int32))
    out_scores, out_ids = dk.fused_topk(_dev(ex["logits"]), ex["K"], L=ex["L"], row_starts=rs,
                                        layout="interleaved" if ex.get("interleaved") else "contiguous")
    torch.cuda.synchronize()
    assert out_ids.cpu().numpy()[0].tolist() == ex["ids"]
    assert np.array_equal(_bits(out_scores.cpu().numpy()[0]), _bits(np.array(ex["scores"], np.float32)))


@pytest.mark.parametrize("seed", range(24))
def test_tieheavy_many_seeds(seed):
    """Heavy ties at the threshold across many seeds: the regression check for
    a missing barrier between reading the shared threshold and resetting it
    (the race the first page's review describes), which drops tied winners."""
    m = workloads.tieheavy(seed=100 + seed)
    assert_same(run_merge(m), oracle.merge(m.scores, m.ids), f"seed {seed}")


def test_prefill_full_size():
    """The full prefill workload (T=8192, dcp=4, K=2048) in the launch
    configuration the bench times: every row bit-exact against the oracle
    (the oracle's rows split between host threads), and the invariants that
    hold for any correct output on every row."""
    m = workloads.prefill()
    gi, gs = run_merge(m)
    wi, ws = helpers.oracle_merge_all(m)
    assert_same((gi, gs), (wi, ws), "prefill")
    k = helpers.key64(gs, np.where(gi == -1, -1, gi - m.row_starts[:, None]).astype(np.int32))
    assert np.all(k[:, :-1] >= k[:, 1:])


def test_chunk_boundaries():
    """2*1024 + 5 rows: the persistent walk crosses two chunk boundaries."""
    m = workloads.random_merge(11, T=2 * 1024 + 5, dcp=2, K=64, mode="bf16", pad_frac=0.05,
                               with_row_starts=True)
    assert_same(run_merge(m), oracle.merge(m.scores, m.ids, m.row_starts), "chunks")


CASES = [
    # (T, dcp, K, mode, pad_frac)
    (1, 1, 1, "normal", 0.0),
    (3, 1, 7, "ties", 0.0),
    (5, 3, 5, "zeros", 0.0),
    (7, 2, 33, "neginf", 0.2),
    (4, 8, 128, "ties", 0.1),
    (9, 4, 2048, "bf16", 0.0),
    (2, 4, 4096, "normal", 0.0),
    (2, 4, 4096, "ties", 0.3),
    (3, 8, 2048, "bf16", 0.05),
    (2, 1, 4096, "const", 0.0),
    (2, 16, 1024, "ties", 0.0),
    (6, 3, 1000, "normal", 0.0),
    (6, 3, 1001, "ties", 0.1),
    (4, 5, 999, "wide", 0.0),
    (3, 4, 2048, "const", 0.5),
    (200, 4, 2048, "bf16", 0.0),
    (5, 4, 2048, "cluster", 0.0),
    (3, 2, 1024, "cluster", 0.1),
    (300, 4, 2048, "ties", 0.02),
    (160, 3, 2048, "zeros", 0.0),
    (4, 4, 2048, "neginf", 0.0),
    (4, 4, 2048, "wide", 0.0),
    (2, 2, 2, "cluster", 0.0),
    # every candidate a winner (K equals the row's candidates), many rows
    (200, 1, 2048, "normal", 0.0),
    (170, 2, 1024, "ties", 0.1),
    # every candidate in one L1 bin: the live set is refined on the next bits
    (200, 4, 2048, "narrow", 0.0),    # two CTAs per SM
    (8, 4, 2048, "narrow", 0.0),      # one CTA per row
    (100, 4, 2048, "narrow", 0.0),
    (3, 4, 4096, "narrow", 0.0),      # K up to 4096
    # K above 2048: the one-CTA-per-row instantiation for K up to 4096
    (5, 2, 4096, "zeros", 0.0),
    (160, 4, 2560, "bf16", 0.0),      # more rows than SMs
    (4, 4, 4096, "cluster", 0.0),     # pathological buckets: the fallback
    (3, 4, 4096, "neginf", 0.5),
    (6, 3, 4096, "ties", 0.05),
    (2, 4, 3072, "wide", 0.0),
    # fewer real candidates than K (short shards): the K-th key is padding
    (16, 4, 2048, "normal", 0.8),     # one CTA per row
    (120, 4, 2048, "normal", 0.8),
    (90, 4, 2048, "cluster", 0.0),    # the same, buckets too large
    (110, 4, 2048, "neginf", 0.0),
    (200, 4, 2048, "bf16", 0.8),      # two CTAs per SM
    (200, 4, 2048, "normal", 0.95),
    (4, 4, 2048, "neginf", 0.8),      # real -inf candidates above the padding
    (160, 4, 2048, "neginf", 0.7),
    (3, 4, 4096, "ties", 0.8),        # K up to 4096
    (3, 8, 2048, "normal", 0.9),      # 16384 candidates per row
    (5, 4, 1024, "const", 0.9),
    # few rows: each row's sort split over parts = min(8, SMs / T) CTAs,
    # slices of the output not all of one size
    (20, 4, 2048, "bf16", 0.0),       # 7 parts
    (25, 4, 2048, "ties", 0.2),       # 6 parts
    (30, 3, 2048, "normal", 0.5),     # 5 parts, padding in the last slices
    (45, 8, 2048, "narrow", 0.0),     # 3 parts, 16384 candidates, b1 refined
    (7, 4, 4096, "bf16", 0.0),        # 8 parts of K = 4096
    (2, 4, 2048, "cluster", 0.3),     # 8 parts, oversized buckets in some slices
    # the many-row merge at K = 2048 (more than two rows per SM, four CTAs
    # per SM)
    (305, 4, 2048, "cluster", 0.0),   # buckets too large: the fallback's radix select
    (330, 2, 2048, "wide", 0.0),      # ids over all of int32: 64-bit rank keys
    (400, 4, 2048, "normal", 0.0),    # fp32 scores: 64-bit rank keys
    (320, 4, 2048, "const", 0.0),     # one score: the id decides everything
    (321, 4, 2048, "neginf", 0.0),    # real -inf candidates among the winners
    (611, 3, 2048, "bf16", 0.1),      # several rows per CTA, padding in some slots
    (420, 4, 2048, "narrow", 0.3),    # bin b1 refined on the next key bits
    (335, 2, 2048, "ties", 0.5),
    (337, 1, 2048, "zeros", 0.0),
    (700, 4, 2048, "bf16", 0.8),      # fewer real candidates than K: list sorts + padding
    (650, 4, 2048, "normal", 0.95),
    (310, 4, 2048, "neginf", 0.7),    # real -inf winners ranked by id
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_random_shapes(case):
    T, dcp, K, mode, pad = case
    m = workloads.random_merge(zlib.crc32(repr(case).encode()) & 0xFFFF, T, dcp, K, mode=mode, pad_frac=pad,
                               with_row_starts=(T % 2 == 0))
    assert_same(run_merge(m), oracle.merge(m.scores, m.ids, m.row_starts), str(case))


def _nan_padding_merge(T, dcp=4, K=2048, seed=7):
    """Rows mixing real candidates, padding and NaNs of both signs.

    Per row (cycling): only real finite candidates and padding; plus negative
    NaNs (which rank below padding) where the padding still fills K; so many
    negative NaNs that the padding does not (the NaNs are winners); positive
    NaNs (which rank above +inf); real -inf candidates above the padding.
    """
    rng = np.random.default_rng(seed)
    n = dcp * K
    ids = workloads.distinct_ids(rng, dcp, T, K, 1 << 20)
    flat_s = np.empty((T, n), np.float32)
    flat_i = ids.transpose(1, 0, 2).reshape(T, n).copy()
    neg_nan = lambda m: (np.uint32(0xFF800001) + rng.integers(0, 0x7FFFFE, m).astype(np.uint32)).view(np.float32)
    pos_nan = lambda m: (np.uint32(0x7F800001) + rng.integers(0, 0x7FFFFE, m).astype(np.uint32)).view(np.float32)
    for t in range(T):
        real = int(rng.integers(1, K // 2))
        kind = t % 5
        row = np.full(n, -np.inf, np.float32)
        pad = np.ones(n, bool)
        perm = rng.permutation(n)
        row[perm[:real]] = rng.standard_normal(real).astype(np.float32)
        pad[perm[:real]] = False
        rest = perm[real:]
        if kind == 1:    # a few negative NaNs, padding still fills K
            m = 50
        elif kind == 2:  # negative NaNs leave padding just enough
            m = n - K
        elif kind == 3:  # padding falls short: negative NaNs are winners
            m = n - real - (K - real) // 2
        else:
            m = 0
        if m:
            row[rest[:m]] = neg_nan(m)
            pad[rest[:m]] = False
        if kind == 4:    # positive NaNs and real -inf candidates
            row[rest[:40]] = pos_nan(40)
            pad[rest[:40]] = False
            pad[rest[40:40 + K // 2]] = False  # real -inf: keep their ids
        flat_s[t] = row
        flat_i[t] = np.where(pad, -1, flat_i[t])
    scores = np.ascontiguousarray(flat_s.reshape(T, dcp, K).transpose(1, 0, 2))
    ids = np.ascontiguousarray(flat_i.reshape(T, dcp, K).transpose(1, 0, 2))
    return workloads.Merge("nan-padding", scores, ids, np.arange(T, dtype=np.int32) * 3)


@pytest.mark.parametrize("T", [10, 200])
def test_nans_and_padding(T):
    m = _nan_padding_merge(T)
    assert_same(run_merge(m), oracle.merge(m.scores, m.ids, m.row_starts), f"T={T}")


def _neginf_rows(T, seed, dcp=4, K=2048):
    """Rows whose K-th key is -inf, cycling over four shapes: every candidate
    a real -inf; 1500 finite candidates and real -inf after them; real -inf
    ids repeated across shards (outside the contract: identical keys, which
    give identical outputs whichever is taken); finite, real -inf and padding
    mixed."""
    rng = np.random.default_rng(seed)
    ids = workloads.distinct_ids(rng, dcp, T, K, 1 << 20)
    scores = np.full((dcp, T, K), -np.inf, np.float32)
    for t in range(T):
        kind = t % 4
        flat_s = scores[:, t, :].reshape(-1)
        flat_i = ids[:, t, :].reshape(-1)
        if kind == 1:
            pos = rng.choice(dcp * K, 1500, replace=False)
            flat_s[pos] = rng.standard_normal(1500).astype(np.float32)
        elif kind == 2:
            ids[1, t, :] = ids[0, t, :]
            flat_i = ids[:, t, :].reshape(-1)
            pos = rng.choice(dcp * K, 300, replace=False)
            flat_s[pos] = rng.standard_normal(300).astype(np.float32)
        elif kind == 3:
            pos = rng.permutation(dcp * K)
            flat_s[pos[:900]] = rng.standard_normal(900).astype(np.float32)
            flat_i[pos[900 + 2500:]] = -1  # padding after 2500 real -inf candidates
        scores[:, t, :] = flat_s.reshape(dcp, K)
        ids[:, t, :] = flat_i.reshape(dcp, K)
    return workloads.Merge("neginf-rows", scores, ids,
                           rng.integers(0, 1 << 20, T).astype(np.int32))


@pytest.mark.parametrize("T", [16, 160, 320])
def test_neginf_threshold_rows(T):
    """Rows whose winners include real -inf candidates chosen by id: the
    split kernel (16 rows), the 512-thread kernel (160) and the many-row
    kernel's shared-memory select on ~id (320)."""
    m = _neginf_rows(T, seed=600 + T)
    assert_same(run_merge(m), helpers.oracle_merge_all(m), f"T={T}")
    assert dk.dcp_topk_device_status() == 0


def _finite_minus_one_rows(T, seed, dcp=4, K=2048):
    """bf16-valued rows (the narrow bucket keys of the many-row merge) with
    slots whose id is -1 but whose score is finite, cycling over four
    shapes: a few such slots; such slots beside (-inf, -1) padding; every id
    of the row -1 (finite scores); ids from a narrow offset range (so the ids'
    top bits agree) with a few -1 slots.  Only (-inf, -1) is padding under
    the contract; these rows check that the kernels, whose id statistics
    leave padding out and which rebuild ids from the bits the row's ids
    share, still give the oracle's bits."""
    rng = np.random.default_rng(seed)
    ids = workloads.distinct_ids(rng, dcp, T, K, 65536)
    scores = workloads.round_to_bf16(rng.standard_normal((dcp, T, K)).astype(np.float32))
    for t in range(T):
        kind = t % 4
        flat_s = scores[:, t, :].reshape(-1)
        flat_i = ids[:, t, :].reshape(-1)
        if kind == 0:
            flat_i[rng.choice(dcp * K, 40, replace=False)] = -1
        elif kind == 1:
            pos = rng.permutation(dcp * K)
            flat_i[pos[:30]] = -1
            flat_s[pos[30:530]] = -np.inf
            flat_i[pos[30:530]] = -1
        elif kind == 2:
            flat_i[:] = -1
        else:
            flat_i += 1 << 24
            flat_i[rng.choice(dcp * K, 25, replace=False)] = -1
        scores[:, t, :] = flat_s.reshape(dcp, K)
        ids[:, t, :] = flat_i.reshape(dcp, K)
    return workloads.Merge("finite-minus-one", scores, ids,
                           rng.integers(0, 1 << 20, T).astype(np.int32))


@pytest.mark.parametrize("T", [16, 160, 320])
def test_finite_scores_with_id_minus_one(T):
    """The split kernel (16 rows), the 512-thread kernel (160) and the
    many-row merge (320) on rows holding finite-score slots with id -1."""
    m = _finite_minus_one_rows(T, seed=700 + T)
    assert_same(run_merge(m), helpers.oracle_merge_all(m), f"T={T}")
    assert dk.dcp_topk_device_status() == 0


def test_all_padding_rows():
    dcp, T, K = 4, 3, 256
    scores = np.full((dcp, T, K), -np.inf, np.float32)
    ids = np.full((dcp, T, K), -1, np.int32)
    m = workloads.Merge("allpad", scores, ids, np.arange(T, dtype=np.int32) * 10)
    got = run_merge(m)
    assert np.all(got[0] == -1) and np.all(np.isneginf(got[1]))
    assert_same(got, oracle.merge(scores, ids, m.row_starts), "all padding")


def test_unaligned_views():
    """Inputs whose rows are not 16-byte aligned take the scalar load path."""
    m = workloads.random_merge(3, T=5, dcp=3, K=40, mode="ties")
    s = torch.zeros(m.scores.size + 1, dtype=torch.float32, device="cuda")
    i = torch.zeros(m.ids.size + 1, dtype=torch.int32, device="cuda")
    s[1:] = _dev(m.scores.ravel())
    i[1:] = _dev(m.ids.ravel())
    out_ids, out_scores = dk.merge(s[1:].view(m.scores.shape), i[1:].view(m.ids.shape))
    torch.cuda.synchronize()
    assert_same((out_ids.cpu().numpy(), out_scores.cpu().numpy()),
                oracle.merge(m.scores, m.ids), "unaligned")


def test_empty_T():
    s = torch.empty((4, 0, 16), dtype=torch.float32, device="cuda")
    i = torch.empty((4, 0, 16), dtype=torch.int32, device="cuda")
    out_ids, out_scores = dk.merge(s, i)
    assert out_ids.shape == (0, 16)


def test_deterministic_repeat():
    m = workloads.prefill(T=300)
    a = run_merge(m)
    b = run_merge(m)
    assert np.array_equal(a[0], b[0]) and np.array_equal(_bits(a[1]), _bits(b[1]))


def test_stream_and_graph_replay():
    """The merge runs on a side stream and inside a captured CUDA graph; replay
    with changed inputs gives the new inputs' result (first page, Tests:
    replay correctness under CUDA-graph capture)."""
    m1 = workloads.decode(seed=21)
    m2 = workloads.tieheavy(seed=22)
    s = _dev(m1.scores)
    i = _dev(m1.ids)
    out_ids = torch.empty((m1.T, m1.K), dtype=torch.int32, device="cuda")
    out_scores = torch.empty((m1.T, m1.K), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        dk.merge(s, i, out_ids=out_ids, out_scores=out_scores)  # uncaptured first call
    side.synchronize()
    assert_same((out_ids.cpu().numpy(), out_scores.cpu().numpy()), oracle.merge(m1.scores, m1.ids))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dk.merge(s, i, out_ids=out_ids, out_scores=out_scores)
    s.copy_(_dev(m2.scores))
    i.copy_(_dev(m2.ids))
    g.replay()
    torch.cuda.synchronize()
    assert_same((out_ids.cpu().numpy(), out_scores.cpu().numpy()), oracle.merge(m2.scores, m2.ids),
                "replay")


def test_stream_order_around_serialized_launches():
    """Kernels are launched so that they may be scheduled while the stream's
    previous kernel finishes; each must still see the inputs a preceding
    torch kernel writes, and a following torch kernel must see its outputs.
    Back-to-back iterations on one stream, no host sync in between."""
    ms = [workloads.decode(seed=40 + j) if j % 2 == 0 else workloads.tieheavy(seed=40 + j)
          for j in range(6)]
    neg_s = [_dev(-m.scores) for m in ms]
    ids = [_dev(m.ids) for m in ms]
    s = torch.empty_like(neg_s[0])
    i = torch.empty_like(ids[0])
    out_ids = torch.empty((ms[0].T, ms[0].K), dtype=torch.int32, device="cuda")
    out_scores = torch.empty((ms[0].T, ms[0].K), dtype=torch.float32, device="cuda")
    got_ids, got_scores = [], []
    for j in range(len(ms)):
        torch.neg(neg_s[j], out=s)           # a kernel writes the scores
        torch.add(ids[j], 0, out=i)          # and the ids
        dk.merge(s, i, out_ids=out_ids, out_scores=out_scores)
        got_ids.append(out_ids + 0)          # kernels read the outputs
        got_scores.append(out_scores * 1.0)
    torch.cuda.synchronize()
    for j, m in enumerate(ms):
        assert_same((got_ids[j].cpu().numpy(), got_scores[j].cpu().numpy()),
                    oracle.merge(m.scores, m.ids), f"iteration {j}")


# --------------------------------------------------------------- local top-K
def run_local(logits, K, rank, dcp, L=None, row_starts=None):
    x = _dev(logits)
    out_scores, out_ids = dk.local_topk(x, K, rank, dcp, L=L,
                                        row_starts=None if row_starts is None else _dev(row_starts))
    torch.cuda.synchronize()
    return out_scores.cpu().numpy(), out_ids.cpu().numpy()


LOCAL_CASES = [
    # (T, L, ld, K, mode)
    (4, 4096, 4096, 2048, "bf16"),
    (3, 4096, 4100, 2048, "normal"),
    (5, 1000, 1003, 64, "ties"),
    (2, 16384, 16384, 4096, "bf16"),
    (3, 100, 100, 200, "normal"),   # L < K: padded
    (2, 7, 7, 7, "ties"),
    (33, 4096, 4096, 2048, "ties"),
    (160, 4096, 4096, 2048, "normal"),  # more rows than SMs
    (8, 4096, 4096, 2048, "masked"),    # causal mask: real -inf candidates
    (160, 4096, 4096, 2048, "masked"),
    (4, 16384, 16384, 4096, "masked"),
]


@pytest.mark.parametrize("case", LOCAL_CASES, ids=lambda c: "-".join(map(str, c)))
def test_local_topk(case):
    T, L, ld, K, mode = case
    logits = workloads.random_logits(zlib.crc32(repr(case).encode()) & 0xFFFF, T, L, ld=ld, mode=mode)
    rs = np.arange(T, dtype=np.int32) * 3
    got = run_local(logits, K, 1, 4, L=L, row_starts=rs)
    want = oracle.local_topk(logits, K, 1, 4, L=L, row_starts=rs)
    assert_same((got[1], got[0]), (want[1], want[0]), str(case))


@pytest.mark.parametrize("T", workloads.SWEEP_T)
def test_sweep_local_then_merge(T):
    """The fused decode sweep: per-shard local top-2048 of 4096 logits, then the
    merge; equal to the oracle's top-2048 over all 16384 logits at once."""
    logits = workloads.sweep_logits(T)
    dcp, _, L = logits.shape
    K = 2048
    x = _dev(logits)
    cand_s = torch.empty((dcp, T, K), dtype=torch.float32, device="cuda")
    cand_i = torch.empty((dcp, T, K), dtype=torch.int32, device="cuda")
    for r in range(dcp):
        dk.local_topk(x[r], K, r, dcp, out_scores=cand_s[r], out_ids=cand_i[r])
    out_ids, out_scores = dk.merge(cand_s, cand_i)
    torch.cuda.synchronize()
    want_s, want_i = oracle.fused_topk(logits, K)
    assert_same((out_ids.cpu().numpy(), out_scores.cpu().numpy()), (want_i, want_s), f"T={T}")
    # and the intermediate candidates equal the oracle's local top-K
    for r in range(dcp):
        ls, li = oracle.local_topk(logits[r], K, r, dcp)
        assert_same((cand_i[r].cpu().numpy(), cand_s[r].cpu().numpy()), (li, ls), f"local r={r}")


def test_staging_wait_timeout_reports_status():
    """The bounded wait on a row's copy barrier gives up and reports it: a
    self-test kernel arms the barrier for a copy it never issues.  The
    context stays usable afterwards."""
    assert dk.dcp_topk_device_status() == 0
    assert dk.dcp_topk_selftest_wait_timeout(200000, torch.cuda.current_stream().cuda_stream) == dk.DCP_OK
    assert dk.dcp_topk_device_status() == dk.DCP_DEVICE_COPY_TIMEOUT
    assert dk.dcp_topk_device_status() == 0  # read clears it
    m = workloads.decode(seed=5, T=3)
    assert_same(run_merge(m), oracle.merge(m.scores, m.ids), "after timeout")
    assert dk.dcp_topk_device_status() == 0


def test_no_device_status_after_runs():
    m = workloads.prefill(T=400)
    run_merge(m)
    assert dk.dcp_topk_device_status() == 0


FUSED_CASES = [
    # (T, dcp, L, ld, K, mode)
    (4, 4, 4096, 4096, 2048, "bf16"),
    (3, 4, 4096, 4100, 2048, "normal"),
    (5, 2, 1000, 1000, 64, "ties"),
    (2, 3, 1001, 1003, 200, "normal"),
    (2, 2, 60, 60, 200, "bf16"),       # fewer candidates than K: padded
    (160, 4, 4096, 4096, 2048, "bf16"),  # more rows than SMs
    (3, 8, 2048, 2048, 2048, "ties"),
    (6, 4, 4096, 4096, 2048, "masked"),  # real -inf candidates
    (160, 2, 4096, 4096, 2048, "masked"),
]


@pytest.mark.parametrize("case", FUSED_CASES, ids=lambda c: "-".join(map(str, c)))
def test_fused_topk(case):
    """Top-K over all shards' logits in one call equals the oracle's fused
    top-K (and so, by the pinned composition identity, local top-K + merge)."""
    T, dcp, L, ld, K, mode = case
    seed = zlib.crc32(repr(case).encode()) & 0xFFFF
    logits = np.stack([workloads.random_logits(seed + r, T, L, ld=ld, mode=mode) for r in range(dcp)])
    rs = (np.arange(T, dtype=np.int32) * 5) if T % 2 else None
    out_s, out_i = dk.fused_topk(_dev(logits), K, L=L, row_starts=None if rs is None else _dev(rs))
    torch.cuda.synchronize()
    want_s, want_i = oracle.fused_topk(logits, K, L=L, row_starts=rs)
    assert_same((out_i.cpu().numpy(), out_s.cpu().numpy()), (want_i, want_s), str(case))


@pytest.mark.parametrize("T", workloads.SWEEP_T)
def test_sweep_fused(T):
    logits = workloads.sweep_logits(T)
    out_s, out_i = dk.fused_topk(_dev(logits), 2048)
    torch.cuda.synchronize()
    want_s, want_i = oracle.fused_topk(logits, 2048)
    assert_same((out_i.cpu().numpy(), out_s.cpu().numpy()), (want_i, want_s), f"T={T}")


# ------------------------------------------------- interleaved shard ids
INTERLEAVED_LOCAL = [
    # (T, L, ld, K, rank, dcp, mode)
    (4, 4096, 4096, 2048, 2, 4, "bf16"),
    (3, 1000, 1003, 64, 1, 3, "ties"),
    (2, 100, 100, 200, 0, 2, "normal"),  # L < K: padded
    (170, 4096, 4096, 2048, 3, 4, "ties"),  # more rows than SMs
]


@pytest.mark.parametrize("case", INTERLEAVED_LOCAL, ids=lambda c: "-".join(map(str, c)))
def test_local_topk_interleaved(case):
    T, L, ld, K, rank, dcp, mode = case
    logits = workloads.random_logits(zlib.crc32(repr(case).encode()) & 0xFFFF, T, L, ld=ld, mode=mode)
    rs = np.arange(T, dtype=np.int32) * 7
    out_s, out_i = dk.local_topk(_dev(logits), K, rank, dcp, L=L, row_starts=_dev(rs),
                                 layout="interleaved")
    torch.cuda.synchronize()
    want_s, want_i = oracle.local_topk(logits, K, rank, dcp, L=L, row_starts=rs, interleaved=True)
    assert_same((out_i.cpu().numpy(), out_s.cpu().numpy()), (want_i, want_s), str(case))


INTERLEAVED_FUSED = [
    # (T, dcp, L, ld, K, mode)
    (4, 4, 4096, 4096, 2048, "bf16"),
    (3, 4, 4096, 4100, 2048, "ties"),
    (5, 3, 1000, 1000, 64, "ties"),
    (2, 3, 1001, 1003, 200, "normal"),  # L % 4 != 0: the general path
    (160, 4, 4096, 4096, 2048, "bf16"),
    (2, 2, 8192, 8192, 2048, "ties"),   # 16384 candidates per row
]


@pytest.mark.parametrize("case", INTERLEAVED_FUSED, ids=lambda c: "-".join(map(str, c)))
def test_fused_topk_interleaved(case):
    T, dcp, L, ld, K, mode = case
    seed = zlib.crc32(repr(case).encode()) & 0xFFFF
    logits = np.stack([workloads.random_logits(seed + r, T, L, ld=ld, mode=mode) for r in range(dcp)])
    rs = (np.arange(T, dtype=np.int32) * 5) if T % 2 else None
    out_s, out_i = dk.fused_topk(_dev(logits), K, L=L, row_starts=None if rs is None else _dev(rs),
                                 layout="interleaved")
    torch.cuda.synchronize()
    want_s, want_i = oracle.fused_topk(logits, K, L=L, row_starts=rs, interleaved=True)
    assert_same((out_i.cpu().numpy(), out_s.cpu().numpy()), (want_i, want_s), str(case))


def test_interleaved_local_then_merge():
    """Interleaved shards: per-shard local top-K on the GPU, then the merge,
    equals the oracle's fused top-K with interleaved ids."""
    logits = workloads.sweep_logits(32, seed=11)
    dcp, T, L = logits.shape
    K = 2048
    x = _dev(logits)
    cand_s = torch.empty((dcp, T, K), dtype=torch.float32, device="cuda")
    cand_i = torch.empty((dcp, T, K), dtype=torch.int32, device="cuda")
    for r in range(dcp):
        dk.local_topk(x[r], K, r, dcp, out_scores=cand_s[r], out_ids=cand_i[r], layout="interleaved")
    out_ids, out_scores = dk.merge(cand_s, cand_i)
    torch.cuda.synchronize()
    want_s, want_i = oracle.fused_topk(logits, K, interleaved=True)
    assert_same((out_ids.cpu().numpy(), out_scores.cpu().numpy()), (want_i, want_s), "interleaved")


def test_graph_captured_prefill_chunks():
    """Prefill merges captured in CUDA graphs and replayed with new inputs
    ("Reserve the sparse indexer's DCP top-k merge scratch through the
    workspace manager", Purpose: the merge walks the rows in 1024-row chunks
    and reserves its scratch up front; rows are independent):
    * one call over T=3000 rows, whose kernel walks the chunks itself;
    * one call per 1024-row chunk on chunk buffers, as a caller holding them
      would make.
    Sampled rows equal the oracle's, and the library asks for no workspace."""
    T, dcp, K, chunk = 3000, 4, 2048, 1024
    assert dk.dcp_topk_merge_workspace_size(T, dcp, K) == 0
    m1 = workloads.prefill(seed=31, T=T)
    m2 = workloads.prefill(seed=32, T=T)
    rows = [0, 1, 1023, 1024, 1025, 2047, 2048, 2999]
    want = oracle.merge(m2.scores, m2.ids, m2.row_starts, rows=rows)

    # one call
    s, i, rs = _dev(m1.scores), _dev(m1.ids), _dev(m1.row_starts)
    out_ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
    out_scores = torch.empty((T, K), dtype=torch.float32, device="cuda")
    dk.merge(s, i, rs, out_ids=out_ids, out_scores=out_scores)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dk.merge(s, i, rs, out_ids=out_ids, out_scores=out_scores)
    s.copy_(_dev(m2.scores))
    i.copy_(_dev(m2.ids))
    rs.copy_(_dev(m2.row_starts))
    g.replay()
    torch.cuda.synchronize()
    assert_same((out_ids.cpu().numpy()[rows], out_scores.cpu().numpy()[rows]), want, "one call")

    # one call per chunk, on chunk buffers
    bounds = [(c0, min(T, c0 + chunk)) for c0 in range(0, T, chunk)]
    bufs = [(_dev(np.ascontiguousarray(m1.scores[:, a:b])), _dev(np.ascontiguousarray(m1.ids[:, a:b])),
             _dev(m1.row_starts[a:b])) for a, b in bounds]
    out_ids.zero_()
    out_scores.zero_()

    def chunks():
        for (a, b), (cs, ci, cr) in zip(bounds, bufs):
            dk.merge(cs, ci, cr, out_ids=out_ids[a:b], out_scores=out_scores[a:b])

    chunks()
    torch.cuda.synchronize()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2):
        chunks()
    for (a, b), (cs, ci, cr) in zip(bounds, bufs):
        cs.copy_(_dev(np.ascontiguousarray(m2.scores[:, a:b])))
        ci.copy_(_dev(np.ascontiguousarray(m2.ids[:, a:b])))
        cr.copy_(_dev(m2.row_starts[a:b]))
    g2.replay()
    torch.cuda.synchronize()
    assert_same((out_ids.cpu().numpy()[rows], out_scores.cpu().numpy()[rows]), want, "per chunk")


@pytest.mark.parametrize("T", [16, 300, 640])
def test_masked_sweep_merge(T):
    """The merge of the local top-Ks of causally masked rows (rows of
    differing context length): shards seeing fewer than K tokens contribute
    real -inf candidates, and rows seeing fewer than K tokens in all have a
    K-th key of -inf.  The merge must equal the oracle's merge of the same
    candidates, and (composition) the fused top-K of the logits."""
    x = workloads.masked_logits(T, seed=6 + T)
    dcp, _, L = x.shape
    K = 2048
    cs = np.empty((dcp, T, K), np.float32)
    ci = np.empty((dcp, T, K), np.int32)
    for r in range(dcp):
        cs[r], ci[r] = oracle.local_topk(x[r], K, r, dcp)
    m = workloads.Merge("masked", cs, ci)
    got = run_merge(m)
    assert_same(got, oracle.merge(cs, ci), "masked merge")
    fs, fi = oracle.fused_topk(x, K)
    assert_same(got, (fi, fs), "masked merge vs fused")
