"""Seeded synthetic inputs for the exact top-k transform (shared by tests, smoke, bench).

This module draws random numbers and lays them out; it holds none of the
selection arithmetic, so that the CUDA path and the CPU oracle can both be fed
from it without sharing anything else. Every array is produced on the host
(numpy PCG64, draws in float64 rounded to nearest fp32), so both sides receive
identical bits.

The shapes and value distributions stand in for the decode-time indexer scores
of DeepSeek-V4 / GLM models that the sglang PR #36004 and #37591 pages measure
on; those real logits are not available, and these generators replace them:

* ``normal``     i.i.d. N(0, 1)                                   (unit-test shape of #36004)
* ``decode``     N(0, 1) plus one N(0, sigma=4) offset per row     (128k-context decode sweep)
* ``banded``     88% of values are 1.0f with random low 8 mantissa bits, the rest N(0, 1)
* ``narrow``     N(5, sigma=1e-6)
* ``subnormal``  random sign, exponent field 0, |x| <= 1e-38
* ``heavy_tail`` 99% N(0, 1), 1% N(8, 1) at random positions
* ``dup``        after any of the above, each element copies a random element of
                 its own row with probability 0.05 (exact duplicate values)

The concentrated generators follow the adversarial distributions that the #37591
page's exactness tests use (section "实现拆解" (implementation breakdown) item 3).
"""

from __future__ import annotations

import dataclasses

import numpy as np

BASE_SEED = 42  # the seed of the #36004 unit test; config n uses BASE_SEED + n - 1


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


# ---------------------------------------------------------------- value generators

def normal(g: np.random.Generator, shape) -> np.ndarray:
    return g.standard_normal(shape).astype(np.float32)


def decode(g: np.random.Generator, batch: int, n: int, offset_sigma: float = 4.0) -> np.ndarray:
    off = g.normal(0.0, offset_sigma, size=(batch, 1))
    return (g.standard_normal((batch, n)) + off).astype(np.float32)


def banded(g: np.random.Generator, n: int, frac: float = 0.88) -> np.ndarray:
    x = g.standard_normal(n).astype(np.float32)
    band = g.random(n) < frac
    low = g.integers(0, 256, size=n, dtype=np.uint32)
    bits = x.view(np.uint32).copy()
    bits[band] = np.uint32(0x3F800000) | low[band]
    return bits.view(np.float32)


def narrow(g: np.random.Generator, n: int, mean: float = 5.0, sigma: float = 1e-6) -> np.ndarray:
    return g.normal(mean, sigma, size=n).astype(np.float32)


# 1e-38 / 2**-149 rounded down: the largest subnormal mantissa with |x| <= 1e-38.
SUBNORMAL_MANTISSA_MAX = 7136238


def subnormal(g: np.random.Generator, n: int) -> np.ndarray:
    mant = g.integers(0, SUBNORMAL_MANTISSA_MAX + 1, size=n, dtype=np.uint32)
    sign = g.integers(0, 2, size=n, dtype=np.uint32) << np.uint32(31)
    return (sign | mant).view(np.float32)


def heavy_tail(g: np.random.Generator, shape, frac: float = 0.01, mean: float = 8.0) -> np.ndarray:
    x = g.standard_normal(shape)
    tail = g.random(shape) < frac
    x[tail] = g.normal(mean, 1.0, size=int(tail.sum()))
    return x.astype(np.float32)


def with_duplicates(g: np.random.Generator, row: np.ndarray, p: float = 0.05) -> np.ndarray:
    """Each element, with probability p, takes the value of a uniformly random
    element of the same (original) row."""
    row = np.asarray(row, dtype=np.float32)
    out = row.copy()
    hit = g.random(row.shape[0]) < p
    src = g.integers(0, row.shape[0], size=int(hit.sum()))
    out[hit] = row[src]
    return out


DISTRIBUTIONS = ("normal", "decode", "banded", "narrow", "subnormal", "heavy_tail")


def row_values(g: np.random.Generator, dist: str, n: int, dup: bool = False) -> np.ndarray:
    """One row of n values from a named distribution."""
    if dist == "normal":
        x = normal(g, n)
    elif dist == "decode":
        x = decode(g, 1, n)[0]
    elif dist == "banded":
        x = banded(g, n)
    elif dist == "narrow":
        x = narrow(g, n)
    elif dist == "subnormal":
        x = subnormal(g, n)
    elif dist == "heavy_tail":
        x = heavy_tail(g, n)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return with_duplicates(g, x) if dup else x


# ---------------------------------------------------------------- layout helpers

def identity_page_table(batch: int, n_pages: int) -> np.ndarray:
    return np.tile(np.arange(n_pages, dtype=np.int32), (batch, 1))


def permuted_page_table(g: np.random.Generator, batch: int, n_pages: int) -> np.ndarray:
    """Row b: an independent random permutation of the page ids 0 .. n_pages-1."""
    return np.stack([g.permutation(n_pages).astype(np.int32) for _ in range(batch)])


def pages_for(row_cap: int, page_size: int) -> int:
    return (row_cap + page_size - 1) // page_size


# ---------------------------------------------------------------- workloads

@dataclasses.dataclass
class Workload:
    """One batch of inputs. ``form`` is "raw", "paged", "ragged" or "window".

    window: row b of ``scores`` [B, row_stride] selects among its columns
    [row_starts[b], seq_lens[b]) (both clamped to the row)."""
    name: str
    form: str
    k: int
    scores: np.ndarray                 # [B, row_stride] (raw/paged) or packed 1-D (ragged)
    seq_lens: np.ndarray               # [B] int32
    page_table: np.ndarray | None = None   # [B, pages] int32 (paged)
    page_size: int = 64
    row_starts: np.ndarray | None = None   # [B] int32 (ragged: row offsets; window: starts)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def scored_elements(self) -> int:
        """Sum over rows of the valid length (the elements the selection scores)."""
        if self.form == "ragged":
            return int(np.maximum(self.seq_lens, 0).sum())
        cap = self.scores.shape[1]
        if self.form == "window":
            lo = np.clip(self.row_starts.astype(np.int64), 0, cap)
            hi = np.clip(self.seq_lens.astype(np.int64), 0, cap)
            return int(np.maximum(hi - lo, 0).sum())
        return int(np.clip(self.seq_lens, 0, cap).sum())

    @property
    def max_row_len(self) -> int:
        """The longest valid row (window) length, e.g. for a length hint."""
        if self.batch == 0:
            return 0
        if self.form == "ragged":
            return int(np.maximum(self.seq_lens, 0).max())
        cap = self.scores.shape[1]
        hi = np.clip(self.seq_lens.astype(np.int64), 0, cap)
        if self.form == "window":
            lo = np.clip(self.row_starts.astype(np.int64), 0, cap)
            return int(np.maximum(hi - lo, 0).max())
        return int(hi.max())

    def as_raw(self) -> "Workload":
        return dataclasses.replace(self, form="raw", page_table=None)


def unit_test_shape(batch: int, c4_len: int, seed: int = BASE_SEED, k: int = 1024,
                    page_size: int = 64) -> Workload:
    """The #36004 unit-test shape: N(0,1), full seq_lens, identity page table."""
    g = rng(seed)
    scores = normal(g, (batch, c4_len))
    seq = np.full(batch, c4_len, dtype=np.int32)
    pt = identity_page_table(batch, pages_for(c4_len, page_size))
    return Workload(f"unit_b{batch}_n{c4_len}", "paged", k, scores, seq, pt, page_size)


def config1() -> Workload:
    """B=1, c4_len=2048, k=1024, page_size=64, N(0,1), identity table [1,32], seed 42."""
    w = unit_test_shape(1, 2048, seed=BASE_SEED)
    w.name = "paged_b1_n2048_k1024"
    return w


def config2(c4_len: int, batch: int = 48, seed: int = BASE_SEED + 1) -> Workload:
    """B=48, c4_len in {8192, 32768}, seq_lens uniform in [1, c4_len], per-row
    permuted page tables, N(0,1), k=1024, page_size=64."""
    g = rng(seed + c4_len)
    scores = normal(g, (batch, c4_len))
    seq = g.integers(1, c4_len + 1, size=batch).astype(np.int32)
    pt = permuted_page_table(g, batch, pages_for(c4_len, 64))
    return Workload(f"paged_b{batch}_n{c4_len}_k1024_randlen", "paged", 1024, scores, seq, pt, 64)


def config3(batch: int, form: str = "paged", c4_len: int = 32768, seed: int = BASE_SEED + 2) -> Workload:
    """Decode sweep at 128k context: c4_len=32768, k=1024, page_size=64,
    N(0,1) plus a per-row N(0, sigma=4) offset, full seq_lens, permuted tables."""
    g = rng(seed + batch)
    scores = decode(g, batch, c4_len)
    seq = np.full(batch, c4_len, dtype=np.int32)
    pt = permuted_page_table(g, batch, pages_for(c4_len, 64))
    w = Workload(f"{form}_b{batch}_n{c4_len}_k1024_decode", "paged", 1024, scores, seq, pt, 64)
    return w.as_raw() if form == "raw" else w


def config4(dist: str, batch: int = 16, lo: int = 65536, hi: int = 262144,
            seed: int = BASE_SEED + 3) -> Workload:
    """Adversarial exactness, ragged: B=16 rows of length uniform in [lo, hi],
    packed back to back, values from a concentrated distribution with ~5% exact
    duplicates, k=2048."""
    g = rng(seed + DISTRIBUTIONS.index(dist))
    lens = g.integers(lo, hi + 1, size=batch).astype(np.int64)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int32)
    rows = [row_values(g, dist, int(n), dup=True) for n in lens]
    scores = np.concatenate(rows).astype(np.float32)
    return Workload(f"ragged_b{batch}_{dist}_k2048", "ragged", 2048, scores,
                    lens.astype(np.int32), None, 64, starts)


def config5(batch: int, c4_len: int = 262144, seed: int = BASE_SEED + 4) -> Workload:
    """Long rows, small batch (1M-token context at 4x compression): c4_len=262144,
    k=2048, page_size=64, 99% N(0,1) + 1% N(8,1), full seq_lens, permuted tables."""
    g = rng(seed + batch)
    scores = heavy_tail(g, (batch, c4_len))
    seq = np.full(batch, c4_len, dtype=np.int32)
    pt = permuted_page_table(g, batch, pages_for(c4_len, 64))
    return Workload(f"paged_b{batch}_n{c4_len}_k2048_heavytail", "paged", 2048, scores, seq, pt, 64)


def prefill_windows(batch: int, row_stride: int, window: int | None = None, k: int = 1024,
                    seed: int = BASE_SEED + 5) -> Workload:
    """Prefill-shaped rows: query b of the last ``batch`` tokens of a context of
    ``row_stride`` keys attends causally to keys [start_b, end_b), end_b =
    row_stride - batch + b + 1, start_b = max(0, end_b - window) (0 without a
    sliding window). Scores: N(0,1) plus a per-row N(0, sigma=4) offset."""
    g = rng(seed + batch + row_stride + (window or 0))
    scores = decode(g, batch, row_stride)
    ends = (row_stride - batch + np.arange(batch) + 1).clip(min=0).astype(np.int32)
    starts = (np.zeros(batch, np.int32) if window is None
              else np.maximum(ends - window, 0).astype(np.int32))
    name = f"window_b{batch}_n{row_stride}_k{k}" + (f"_w{window}" if window else "_causal")
    return Workload(name, "window", k, scores, ends, None, 64, starts)


def random_rows(g: np.random.Generator, batch: int, row_stride: int, dist: str,
                dup: bool = False) -> np.ndarray:
    return np.stack([row_values(g, dist, row_stride, dup) for _ in range(batch)])
