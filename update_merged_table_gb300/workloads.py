"""Seeded synthetic inputs for the merged dynamic embedding table.

This module only draws random inputs (ID batches, gradients, erase sets).  It
holds none of the table's arithmetic: no key encoding, hashing, dedup, row
initialisation or optimizer step.  Both the CUDA path and the CPU oracle are
fed from here, so the two always see the same bytes.

The workloads follow the sparse-embedding workloads described in
"MTGenRec: An Efficient Distributed Training System for Generative
Recommendation Models in Meituan" (dynamic hash embedding table, feature tables
merged into one, ID deduplication in two stages) and the jagged user sequences of "MTGR:
Industrial-Scale Generative Recommendation Framework in Meituan" (section 5,
"Load Balance").  The pages measure on production data that is not available,
so every batch here is synthetic:

* ID frequencies are Zipf(s) over a finite vocabulary, drawn by
  rejection-inversion (W. Hormann and G. Derflinger, "Rejection-inversion to
  generate variates from monotone discrete distributions", ACM TOMACS 1996).
* Jagged sequence lengths are floor(lognormal(mu, sigma)), capped.
* Gradients are N(0, 1).

IDs are plain non-negative int64 feature IDs; the merged key of a position is
formed by the library from the feature segment it falls in.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# --------------------------------------------------------------------------
# Zipf sampling by rejection-inversion
# --------------------------------------------------------------------------


def _expm1_over_x(t: np.ndarray) -> np.ndarray:
    """(exp(t) - 1) / t, continuous at t = 0."""
    t = np.asarray(t, dtype=np.float64)
    out = np.ones_like(t)
    nz = np.abs(t) > 1e-8
    out[nz] = np.expm1(t[nz]) / t[nz]
    small = ~nz
    out[small] = 1.0 + t[small] * 0.5
    return out


def _log1p_over_x(t: np.ndarray) -> np.ndarray:
    """log(1 + t) / t, continuous at t = 0."""
    t = np.asarray(t, dtype=np.float64)
    out = np.ones_like(t)
    nz = np.abs(t) > 1e-8
    out[nz] = np.log1p(t[nz]) / t[nz]
    small = ~nz
    out[small] = 1.0 - t[small] * 0.5
    return out


class ZipfSampler:
    """Draws ranks k in [1, V] with P(k) proportional to k**-s (s > 0).

    The continuous envelope is h(x) = x**-s with antiderivative
    H(x) = (x**(1-s) - 1) / (1-s) (log x at s = 1).  A uniform point between
    H(V + 1/2) and H(3/2) - 1 is inverted through H, rounded to the nearest
    integer k, and accepted when it falls under the step of height h(k).
    """

    def __init__(self, s: float, V: int):
        if not (s > 0.0) or V < 1:
            raise ValueError("Zipf needs s > 0 and V >= 1")
        self.s = float(s)
        self.V = int(V)
        self._hx1 = float(self._H(np.array([1.5]))[0] - 1.0)
        self._hN = float(self._H(np.array([self.V + 0.5]))[0])
        self._cut = 2.0 - float(
            self._Hinv(np.array([self._H(np.array([2.5]))[0] - self._h(np.array([2.0]))[0]]))[0])

    def _h(self, x):
        return np.exp(-self.s * np.log(x))

    def _H(self, x):
        lx = np.log(x)
        return lx * _expm1_over_x((1.0 - self.s) * lx)

    def _Hinv(self, y):
        t = y * (1.0 - self.s)
        t = np.maximum(t, -1.0 + 1e-16)
        return np.exp(_log1p_over_x(t) * y)

    def sample(self, rng: np.random.Generator, n: int) -> np.ndarray:
        out = np.empty(n, dtype=np.int64)
        todo = np.arange(n)
        while todo.size:
            m = todo.size
            u = self._hN + rng.random(m) * (self._hx1 - self._hN)
            x = self._Hinv(u)
            k = np.clip(np.floor(x + 0.5), 1, self.V)
            ok = (k - x <= self._cut) | (u >= self._H(k + 0.5) - self._h(k))
            out[todo[ok]] = k[ok].astype(np.int64)
            todo = todo[~ok]
        return out


def zipf_ranks(rng: np.random.Generator, n: int, s: float, V: int) -> np.ndarray:
    return ZipfSampler(s, V).sample(rng, n)


def bijection32(x: np.ndarray) -> np.ndarray:
    """A fixed bijection of [0, 2**32) used to spread Zipf ranks over a 32-bit key space."""
    x = np.asarray(x, dtype=np.uint64) & np.uint64(0xFFFFFFFF)
    x = (x * np.uint64(0x9E3779B1)) & np.uint64(0xFFFFFFFF)
    x ^= x >> np.uint64(15)
    x = (x * np.uint64(0x85EBCA77)) & np.uint64(0xFFFFFFFF)
    x ^= x >> np.uint64(13)
    return x.astype(np.int64)


# --------------------------------------------------------------------------
# Batches
# --------------------------------------------------------------------------


@dataclasses.dataclass
class Batch:
    """One lookup batch: IDs grouped into feature segments.

    ids[feat_offsets[f]:feat_offsets[f+1]] belong to feature table table_ids[f].
    """
    ids: np.ndarray            # int64 [N]
    feat_offsets: np.ndarray   # int64 [F+1]
    table_ids: np.ndarray      # uint8 [F]
    user_offsets: np.ndarray | None = None   # int64 [users+1] (jagged batches only)

    @property
    def n(self) -> int:
        return int(self.ids.shape[0])


def single_feature(ids: np.ndarray, table_id: int = 0) -> Batch:
    ids = np.ascontiguousarray(ids, dtype=np.int64)
    return Batch(ids, np.array([0, ids.size], dtype=np.int64), np.array([table_id], dtype=np.uint8))


def grads_normal(seed: int, n: int, dim: int) -> np.ndarray:
    """N(0, 1) fp32 gradients [n, dim]."""
    return np.random.default_rng(seed).standard_normal((n, dim), dtype=np.float32)


def grads_small_int(seed: int, n: int, dim: int, lo: int = -4, hi: int = 4) -> np.ndarray:
    """Integer-valued fp32 gradients: every partial sum is exact in fp32."""
    return np.random.default_rng(seed).integers(lo, hi + 1, size=(n, dim)).astype(np.float32)


# ---- single table (4096 IDs, Zipf 1.1 over 1e5) ----------------------------

def single_table_batch(seed: int = 0, n: int = 4096, s: float = 1.1, vocab: int = 100_000) -> Batch:
    rng = np.random.default_rng(seed)
    return single_feature(zipf_ranks(rng, n, s, vocab) - 1)


# ---- merged tables (8 features, vocab 1e4..1e6, s 0.8..1.3) ----------------

MERGED_TABLES = 8


def merged_vocab(k: int) -> int:
    return int(round(10.0 ** (4.0 + 2.0 * k / 7.0)))


def merged_exponent(k: int) -> float:
    return 0.8 + 0.5 * k / 7.0


def merged_batch(seed: int, per_table: int = 8192, tables: int = MERGED_TABLES) -> Batch:
    parts = []
    for k in range(tables):
        rng = np.random.default_rng([seed, k])
        parts.append(zipf_ranks(rng, per_table, merged_exponent(k), merged_vocab(k)) - 1)
    ids = np.concatenate(parts)
    offs = np.arange(tables + 1, dtype=np.int64) * per_table
    return Batch(ids, offs, np.arange(tables, dtype=np.uint8))


# ---- GRM jagged sequences (2048 users, lognormal lengths, 4 ID features) ---

def jagged_lengths(seed: int, users: int = 2048, mu: float = 5.0, sigma: float = 1.0, cap: int = 3000) -> np.ndarray:
    rng = np.random.default_rng([seed, 0x5E9])
    lens = np.floor(rng.lognormal(mu, sigma, size=users)).astype(np.int64)
    return np.clip(lens, 1, cap)


def jagged_batch(seed: int, users: int = 2048, features: int = 4, s: float = 1.1,
                 vocab: int = 1_000_000, mu: float = 5.0, sigma: float = 1.0, cap: int = 3000,
                 lengths_seed: int | None = None) -> Batch:
    """Feature-major flattening of a jagged batch: F segments of T tokens each.

    The user sequence lengths are drawn once per lengths_seed (default: seed);
    each feature's token IDs are Zipf(s) over `vocab`.
    """
    lens = jagged_lengths(seed if lengths_seed is None else lengths_seed, users, mu, sigma, cap)
    T = int(lens.sum())
    parts = []
    for f in range(features):
        rng = np.random.default_rng([seed, 0xF00 + f])
        parts.append(zipf_ranks(rng, T, s, vocab) - 1)
    ids = np.concatenate(parts)
    offs = np.arange(features + 1, dtype=np.int64) * T
    uo = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    return Batch(ids, offs, np.arange(features, dtype=np.uint8), uo)


# ---- large table (Zipf 1.05 over a 2**32 key space) ------------------------

LARGE_KEYSPACE = 1 << 32


def large_table_batch(seed: int, n: int = 1 << 20, s: float = 1.05) -> Batch:
    rng = np.random.default_rng([seed, 0x1A6])
    ranks = zipf_ranks(rng, n, s, LARGE_KEYSPACE)
    return single_feature(bijection32(ranks - 1))


def large_table_prefill_ids(count: int) -> np.ndarray:
    """IDs of the `count` most popular ranks (the steady-state resident set)."""
    return bijection32(np.arange(count, dtype=np.int64))


# ---- online churn ----------------------------------------------------------

class ChurnStream:
    """Per step: n IDs, `new_frac` of them never seen before, plus an erase set.

    The hot universe is IDs [0, hot); fresh IDs count up from `hot`.  The
    stream assumes its prefill_ids() were inserted before step 0 and that
    every ID of a step is inserted by that step's lookup, so it knows which
    IDs are live: the erase set of a step is drawn uniformly, without
    replacement, from the IDs live after that step's lookup, and those IDs are
    live no longer.  Steps must be taken in order 0, 1, 2, ...
    """

    def __init__(self, seed: int, hot: int = 1 << 23, n: int = 1 << 18, new_frac: float = 0.1,
                 erase: int = 1 << 16, s: float = 1.1):
        self.seed, self.hot, self.n, self.new_frac, self.erase, self.s = seed, hot, n, new_frac, erase, s
        self.next_fresh = hot
        self._zipf = ZipfSampler(s, hot)
        self._live = np.ones(hot, dtype=bool)
        self._next_step = 0

    def prefill_ids(self) -> np.ndarray:
        return np.arange(self.hot, dtype=np.int64)

    def step(self, k: int) -> tuple[Batch, np.ndarray]:
        if k != self._next_step:
            raise ValueError(f"churn steps must be taken in order: expected step {self._next_step}, got {k}")
        self._next_step += 1
        rng = np.random.default_rng([self.seed, 0xC4, k])
        n_new = int(round(self.n * self.new_frac))
        hot_ids = self._zipf.sample(rng, self.n - n_new) - 1
        fresh = np.arange(self.next_fresh, self.next_fresh + n_new, dtype=np.int64)
        self.next_fresh += n_new
        ids = np.concatenate([hot_ids, fresh])
        ids = ids[rng.permutation(ids.size)]
        if self._live.size < self.next_fresh:
            grown = np.zeros(max(self.next_fresh, 2 * self._live.size), dtype=bool)
            grown[: self._live.size] = self._live
            self._live = grown
        self._live[ids] = True
        live_ids = np.flatnonzero(self._live[: self.next_fresh])
        erase_ids = rng.choice(live_ids, size=min(self.erase, live_ids.size), replace=False).astype(np.int64)
        self._live[erase_ids] = False
        return single_feature(ids), erase_ids

    def live_ids(self) -> np.ndarray:
        """The IDs live after the last step taken (prefill, then every step's inserts and erases)."""
        return np.flatnonzero(self._live[: self.next_fresh]).astype(np.int64)
