"""Seeded synthetic inputs for the DCP top-K merge and the per-shard local top-K.

This module only draws random numbers and lays them out; it holds none of the
selection arithmetic.  Both the CPU oracle (tests) and the CUDA path (tests,
bench, smoke) take their inputs from here, so neither side generates data for
the other.

Layouts follow the candidate exchange described in "Reserve the sparse
indexer's DCP top-k merge scratch through the workspace manager" (Purpose): the
gathered candidates are rank-major, ``scores[r][t][k]`` and ``ids[r][t][k]``
with shape ``(dcp, T, K)``; a padding slot is ``(score=-inf, id=-1)``.

The five named workloads:

* ``tiny``      T=4, dcp=2, K=64; shard r draws 64 distinct ids from
                [r*1024, (r+1)*1024); scores uniform in [-1, 1); seed 0.
* ``decode``    T=16, dcp=4, K=2048; shard r draws distinct ids from
                [r*65536, (r+1)*65536); scores standard normal; seed 1.
* ``tieheavy``  as ``decode`` but scores uniform over the 16 values
                (i - 7.5)/8, i = 0..15 (exact in fp32), and shard 3 is all
                padding for rows t >= T/2; seed 2.
* ``sweep``     per-shard logits, shape (dcp=4, T, L=4096), standard normal
                rounded to bf16 (round to nearest even) and stored as fp32;
                T in {1, 8, 32, 64, 256}; seed 3 (+T).
* ``prefill``   T=8192, dcp=4, K=2048; distinct ids per shard as in
                ``decode``; scores N(mu_t, 1) with mu_t = (t mod 64)/8 - 4,
                rounded to bf16; row_starts[t] = 262144 * (t // 256); seed 4.
"""
from __future__ import annotations

import numpy as np

NEG_INF = np.float32(-np.inf)
PAD_ID = np.int32(-1)

SWEEP_T = (1, 8, 32, 64, 256)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even), returned as fp32.

    Input generation only: makes the duplicate-heavy score distributions the
    sweep and prefill workloads ask for.  Finite inputs only.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = ((b + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)).astype(np.uint32)
    return r.view(np.float32)


def distinct_ids(rng: np.random.Generator, dcp: int, T: int, K: int, span: int) -> np.ndarray:
    """Per (shard, row): K distinct ids drawn without replacement from
    [r*span, (r+1)*span).  Shape (dcp, T, K), int32."""
    ids = np.empty((dcp, T, K), dtype=np.int32)
    for r in range(dcp):
        for t in range(T):
            ids[r, t] = r * span + rng.choice(span, K, replace=False)
    return ids


class Merge:
    """A merge problem: rank-major candidates plus optional row offsets."""

    def __init__(self, name, scores, ids, row_starts=None):
        self.name = name
        self.scores = np.ascontiguousarray(scores, dtype=np.float32)
        self.ids = np.ascontiguousarray(ids, dtype=np.int32)
        self.dcp, self.T, self.K = self.scores.shape
        assert self.ids.shape == self.scores.shape
        self.row_starts = None if row_starts is None else np.ascontiguousarray(row_starts, dtype=np.int32)

    @property
    def N(self):
        return self.dcp * self.K

    def algorithmic_bytes(self):
        """Bytes a merge must move: every candidate's score and id once,
        plus the K output (id, score) pairs per row."""
        return self.T * (self.N * 8 + self.K * 8) + (0 if self.row_starts is None else self.T * 4)


def tiny(seed: int = 0) -> Merge:
    rng = np.random.default_rng(seed)
    T, dcp, K = 4, 2, 64
    ids = distinct_ids(rng, dcp, T, K, 1024)
    scores = rng.uniform(-1.0, 1.0, size=(dcp, T, K)).astype(np.float32)
    return Merge("tiny", scores, ids)


def decode(seed: int = 1, T: int = 16, dcp: int = 4, K: int = 2048) -> Merge:
    rng = np.random.default_rng(seed)
    ids = distinct_ids(rng, dcp, T, K, 65536)
    scores = rng.standard_normal((dcp, T, K), dtype=np.float32)
    return Merge("decode", scores, ids)


TIE_VALUES = ((np.arange(16, dtype=np.float64) - 7.5) / 8.0).astype(np.float32)


def tieheavy(seed: int = 2, T: int = 16, dcp: int = 4, K: int = 2048) -> Merge:
    rng = np.random.default_rng(seed)
    ids = distinct_ids(rng, dcp, T, K, 65536)
    scores = TIE_VALUES[rng.integers(0, 16, size=(dcp, T, K))]
    empty = dcp - 1
    scores[empty, T // 2:, :] = NEG_INF
    ids[empty, T // 2:, :] = PAD_ID
    return Merge("tieheavy", scores, ids)


def sweep_logits(T: int, seed: int = 3, dcp: int = 4, L: int = 4096) -> np.ndarray:
    """Per-shard logits (dcp, T, L), bf16-valued fp32."""
    rng = np.random.default_rng(seed + T)
    return round_to_bf16(rng.standard_normal((dcp, T, L), dtype=np.float32))


def prefill(seed: int = 4, T: int = 8192, dcp: int = 4, K: int = 2048) -> Merge:
    rng = np.random.default_rng(seed)
    ids = distinct_ids(rng, dcp, T, K, 65536)
    mu = ((np.arange(T) % 64) / 8.0 - 4.0).astype(np.float32)
    z = rng.standard_normal((dcp, T, K), dtype=np.float32)
    z += mu[None, :, None]
    scores = round_to_bf16(z)
    row_starts = (262144 * (np.arange(T) // 256)).astype(np.int32)
    return Merge("prefill", scores, ids, row_starts)


NAMED = {"tiny": tiny, "decode": decode, "tieheavy": tieheavy, "prefill": prefill}


class FusedShape:
    """Sizes of a fused top-K over per-shard logits (dcp, T, L), K outputs."""

    def __init__(self, T, dcp, L, K):
        self.T, self.dcp, self.L, self.K = T, dcp, L, K
        self.row_starts = None

    def algorithmic_bytes(self):
        """Every logit once, plus the K output (id, score) pairs per row."""
        return self.T * (self.dcp * self.L * 4 + self.K * 8)


def random_merge(seed: int, T: int, dcp: int, K: int, mode: str = "normal",
                 pad_frac: float = 0.0, with_row_starts: bool = False) -> Merge:
    """Small random merge problems for parity sweeps.

    mode: ``normal`` (fp32 N(0,1)), ``bf16`` (N(0,1) rounded to bf16),
    ``ties`` (4 distinct values), ``const`` (one value), ``zeros`` (+0/-0 and
    a few +-1), ``neginf`` (many real -inf scores), ``wide`` (ids spread over
    the whole non-negative int32 range), ``cluster`` (most top scores within a
    few ulps of each other), ``narrow`` (fp32 scores uniform in [1, 1.0625)).
    pad_frac: fraction of slots, anywhere in each shard, replaced by padding.
    """
    rng = np.random.default_rng(seed)
    span = 1 << 20
    if mode == "wide":
        ids = np.empty((dcp, T, K), dtype=np.int32)
        for r in range(dcp):
            for t in range(T):
                ids[r, t] = rng.choice(np.iinfo(np.int32).max // dcp, K, replace=False) * dcp + r
    else:
        ids = distinct_ids(rng, dcp, T, K, span)
    shape = (dcp, T, K)
    if mode in ("normal", "wide"):
        scores = rng.standard_normal(shape, dtype=np.float32)
    elif mode == "bf16":
        scores = round_to_bf16(rng.standard_normal(shape, dtype=np.float32))
    elif mode == "ties":
        scores = np.array([0.75, 0.5, -0.25, 2.0], np.float32)[rng.integers(0, 4, shape)]
    elif mode == "const":
        scores = np.full(shape, 0.5, np.float32)
    elif mode == "zeros":
        scores = np.array([0.0, -0.0, 1.0, -1.0, 0.0, -0.0], np.float32)[rng.integers(0, 6, shape)]
    elif mode == "cluster":
        # most of each row's top candidates packed into a few ulps above 1.0,
        # plus one candidate at 1.2 in the same top-11-bit bin: keys that
        # agree on every bit but the lowest few, the hardest case for
        # bucketing on leading bits
        scores = rng.uniform(-1.0, 0.5, size=shape).astype(np.float32)
        n = dcp * K
        m = max(1, (3 * min(n, 4096)) // 8 + K // 2)
        m = min(m, n - 1) if n > 1 else 1
        base = np.uint32(np.float32(1.0).view(np.uint32))
        flat = scores.transpose(1, 0, 2).reshape(T, n)
        for t in range(T):
            pos = rng.choice(n, min(n, m + 1), replace=False)
            flat[t, pos[:m]] = (base + rng.choice(4096, m, replace=m > 4096).astype(np.uint32)).view(np.float32)
            if len(pos) > m:
                flat[t, pos[m]] = np.float32(1.2)
        scores = np.ascontiguousarray(flat.reshape(T, dcp, K).transpose(1, 0, 2))
    elif mode == "narrow":
        # fp32 scores uniform in [1, 1 + 1/16): one L1 bin holds every
        # candidate, with distinct keys below it (the live-set refinement)
        scores = rng.uniform(1.0, 1.0625, size=shape).astype(np.float32)
    elif mode == "neginf":
        scores = np.where(rng.random(shape) < 0.6, NEG_INF,
                          rng.standard_normal(shape, dtype=np.float32)).astype(np.float32)
    else:
        raise ValueError(mode)
    if pad_frac > 0:
        m = rng.random(shape) < pad_frac
        scores = np.where(m, NEG_INF, scores).astype(np.float32)
        ids = np.where(m, PAD_ID, ids).astype(np.int32)
    rs = None
    if with_row_starts:
        rs = rng.integers(0, 1 << 24, size=T).astype(np.int32)
    return Merge(f"random-{mode}", scores, ids, rs)


def masked_logits(T: int, seed: int = 5, dcp: int = 4, L: int = 4096) -> np.ndarray:
    """Per-shard logits (dcp, T, L) of prefill rows with differing context
    lengths: row t sees the first c_t tokens of the sequence (c_t uniform in
    [1, dcp*L], seeded), the tokens dealt to the shards contiguously (shard r
    holds tokens [r*L, (r+1)*L)), so shard r's row t has max(0, min(L,
    c_t - r*L)) finite logits (N(0,1) rounded to bf16) and -inf after them
    (the causal mask).  The local top-K of each shard then holds real -inf
    candidates wherever a shard sees fewer than K tokens, and the merge of
    those rows has a K-th key of -inf whenever the row sees fewer than K
    tokens in all."""
    rng = np.random.default_rng(seed)
    x = round_to_bf16(rng.standard_normal((dcp, T, L), dtype=np.float32))
    ctx = rng.integers(1, dcp * L + 1, T)
    for r in range(dcp):
        valid = np.clip(ctx - r * L, 0, L)
        x[r][np.arange(L)[None, :] >= valid[:, None]] = NEG_INF
    return np.ascontiguousarray(x, dtype=np.float32)


def random_logits(seed: int, T: int, L: int, ld: int | None = None, mode: str = "bf16") -> np.ndarray:
    """Logits rows (T, ld) with the first L columns meaningful.

    mode: ``bf16`` (N(0,1) rounded to bf16), ``normal`` (fp32 N(0,1)),
    ``ties`` (4 distinct values), ``masked`` (bf16 values in each row's first
    columns, a row-dependent count from 0 to L, and -inf after them: a causal
    mask).
    """
    rng = np.random.default_rng(seed)
    ld = L if ld is None else ld
    x = rng.standard_normal((T, ld), dtype=np.float32)
    if mode == "bf16":
        x = round_to_bf16(x)
    elif mode == "ties":
        x = np.array([0.75, 0.5, -0.25, 2.0], np.float32)[rng.integers(0, 4, (T, ld))]
    elif mode == "masked":
        x = round_to_bf16(x)
        valid = rng.integers(0, L + 1, T)
        x[np.arange(ld)[None, :] >= valid[:, None]] = NEG_INF
    elif mode != "normal":
        raise ValueError(mode)
    return np.ascontiguousarray(x, dtype=np.float32)
