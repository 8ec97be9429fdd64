"""Test-side helpers: golden-file parsing, a comparison-based brute force, and
invariant checks that hold for any correct top-K output at any size.

Nothing here is used by the library; the invariant checks apply equally to the
oracle's and to the CUDA path's outputs.
"""
from __future__ import annotations

import concurrent.futures
import itertools
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _f(tok: str) -> float:
    return float(tok)


def parse_merge_examples(path=os.path.join(GOLDEN, "merge_examples.txt")):
    out = []
    cur = None
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, _, rest = line.partition(" ")
        if head == "example":
            cur = {"name": rest, "shards": [], "row_starts": None}
            out.append(cur)
        elif head == "dcp":
            a = rest.split()
            cur["dcp"], cur["K"] = int(a[0]), int(a[2])
        elif head == "shard":
            _, _, pairs = rest.partition(":")
            row = [(_f(p.split(":")[0]), int(p.split(":")[1])) for p in pairs.split()]
            cur["shards"].append(row)
        elif head == "row_starts":
            cur["row_starts"] = int(rest)
        elif head == "ids":
            cur["ids"] = [int(x) for x in rest.split()]
        elif head == "scores":
            cur["scores"] = [_f(x) for x in rest.split()]
    for ex in out:
        dcp, K = ex["dcp"], ex["K"]
        assert len(ex["shards"]) == dcp and all(len(s) == K for s in ex["shards"])
        ex["scores_in"] = np.array([[[p[0] for p in s]] for s in ex["shards"]], np.float32)
        ex["ids_in"] = np.array([[[p[1] for p in s]] for s in ex["shards"]], np.int32)
        ex["rs"] = None if ex["row_starts"] is None else np.array([ex["row_starts"]], np.int32)
    return out


def parse_local_examples(path=os.path.join(GOLDEN, "local_examples.txt")):
    out = []
    cur = None
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, _, rest = line.partition(" ")
        if head == "example":
            cur = {"name": rest, "row_starts": None, "interleaved": False}
            out.append(cur)
        elif head == "layout":
            cur["interleaved"] = rest.strip() == "interleaved"
        elif head == "L":
            a = rest.split()
            cur["L"] = int(a[0])
            kv = dict(zip(a[1::2], a[2::2]))
            cur["ld"], cur["K"], cur["rank"], cur["dcp"] = (int(kv["ld"]), int(kv["K"]),
                                                            int(kv["rank"]), int(kv["dcp"]))
        elif head == "row":
            cur["row"] = np.array([[_f(x) for x in rest.split()]], np.float32)
        elif head == "row_starts":
            cur["row_starts"] = int(rest)
        elif head == "ids":
            cur["ids"] = [int(x) for x in rest.split()]
        elif head == "scores":
            cur["scores"] = [_f(x) for x in rest.split()]
    return out


def parse_fused_examples(path=os.path.join(GOLDEN, "fused_examples.txt")):
    out = []
    cur = None
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, _, rest = line.partition(" ")
        if head == "example":
            cur = {"name": rest, "row_starts": None, "shards": []}
            out.append(cur)
        elif head == "dcp":
            a = rest.split()
            cur["dcp"], cur["L"], cur["K"] = int(a[0]), int(a[2]), int(a[4])
        elif head == "layout":
            cur["interleaved"] = rest.strip() == "interleaved"
        elif head == "shard":
            _, _, vals = rest.partition(":")
            cur["shards"].append([_f(x) for x in vals.split()])
        elif head == "row_starts":
            cur["row_starts"] = int(rest)
        elif head == "ids":
            cur["ids"] = [int(x) for x in rest.split()]
        elif head == "scores":
            cur["scores"] = [_f(x) for x in rest.split()]
    for ex in out:
        assert len(ex["shards"]) == ex["dcp"] and all(len(r) == ex["L"] for r in ex["shards"])
        ex["logits"] = np.array([[r] for r in ex["shards"]], np.float32)  # (dcp, 1, L)
    return out


# ---------------------------------------------------------------- brute force
def beats(a, b) -> bool:
    """True if candidate a = (score, id) ranks strictly before b.

    Written from the order rule with float comparisons (no bit keys): higher
    score first; +0.0 before -0.0; among equal scores the lower id, taken as
    an unsigned 32-bit number (so padding id -1 comes last).
    """
    sa, ia = a
    sb, ib = b
    if sa != sb:
        return sa > sb
    if sa == 0.0:
        na = math.copysign(1.0, sa) < 0
        nb = math.copysign(1.0, sb) < 0
        if na != nb:
            return nb
    return (ia & 0xFFFFFFFF) < (ib & 0xFFFFFFFF)


def brute_force_topk(cands, K):
    """Top-K of a small candidate list by enumerating every K-subset.

    The selected set is the K-subset in which no member is beaten by a
    non-member; candidates identical in score bits and id are
    interchangeable.  Its order is found by counting, for each member, how
    many members beat it.  Returns a list of (score, id).
    """
    n = len(cands)
    found = None
    for S in itertools.combinations(range(n), K):
        inside = set(S)
        ok = all(not beats(cands[o], cands[i]) for i in S for o in range(n) if o not in inside)
        if ok:
            sig = sorted((np.float32(cands[i][0]).tobytes(), cands[i][1]) for i in S)
            if found is None:
                found = (S, sig)
            else:
                assert sig == found[1], "two valid selections differ"
    assert found is not None
    S = found[0]
    slots = [None] * K
    for i in S:
        pos = sum(1 for j in S if beats(cands[j], cands[i]))
        while slots[pos] is not None:  # identical duplicates share a rank
            pos += 1
        slots[pos] = cands[i]
    return slots


# ----------------------------------------------------------------- invariants
def key32(scores: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(scores, np.float32).view(np.uint32)
    return np.where(b >> 31 == 1, ~b, b | np.uint32(0x80000000)).astype(np.uint32)


def key64(scores: np.ndarray, ids: np.ndarray) -> np.ndarray:
    k = key32(scores).astype(np.uint64) << np.uint64(32)
    inv = (~np.ascontiguousarray(ids, np.int32).view(np.uint32)).astype(np.uint64)
    return k | inv


def check_merge_invariants(scores, ids, row_starts, out_ids, out_scores, rows=None):
    """Properties every correct merge output has, checked row by row.

    * exactly K outputs per row;
    * outputs in non-increasing key order, strictly decreasing except for
      identical (score bits, id) duplicates;
    * the output is a sub-multiset of the row's candidates, and every selected
      key is >= every rejected key (so selected scores >= rejected scores, and
      the tie rule holds at the threshold);
    * padding (id -1, -inf) only at the tail; ids carry row_starts except
      padding.
    """
    dcp, T, K = scores.shape
    rows = range(T) if rows is None else rows
    assert out_ids.shape[1] == K and out_scores.shape[1] == K
    for i, t in enumerate(rows):
        rs = 0 if row_starts is None else int(row_starts[t])
        oid = out_ids[i].astype(np.int64)
        raw = np.where(oid == -1, -1, oid - rs).astype(np.int64)
        assert np.all((raw >= -(2 ** 31)) & (raw < 2 ** 31)), f"row {t}: id overflow"
        ko = key64(out_scores[i], raw.astype(np.int32))
        assert np.all(ko[:-1] >= ko[1:]), f"row {t}: output not in key order"
        cand = np.sort(key64(scores[:, t, :].ravel(), ids[:, t, :].ravel()))[::-1]
        assert np.array_equal(np.sort(ko)[::-1], cand[:K]), f"row {t}: not the top-K multiset"
        pad = (raw == -1) & np.isneginf(out_scores[i])
        if pad.any():
            first = int(np.argmax(pad))
            assert np.all(pad[first:]), f"row {t}: padding not only at the tail"


def merge_inputs_from_example(ex):
    return ex["scores_in"], ex["ids_in"], ex["rs"]


def oracle_merge_all(m, threads=None):
    """The oracle's merge of every row of merge problem ``m``, the rows split
    between host threads (rows are independent; the C call releases Python's
    lock).  Same result as one ``oracle.merge`` call over all rows."""
    import oracle

    threads = threads or os.cpu_count() or 1
    T = m.T
    chunk = max(1, -(-T // (4 * threads)))
    starts = list(range(0, T, chunk))

    def part(a):
        rows = np.arange(a, min(T, a + chunk), dtype=np.int32)
        return oracle.merge(m.scores, m.ids, m.row_starts, rows=rows)

    with concurrent.futures.ThreadPoolExecutor(threads) as pool:
        parts = list(pool.map(part, starts))
    return (np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts]))
