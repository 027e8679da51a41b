"""Pins of the CPU oracle to things other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError on
the first disagreement. The pins are:

* hand-worked fixtures (tests/golden/topk_cases.txt), values worked out from the
  definitions on the source pages;
* brute force over every k-subset of tiny rows (no key transform, no sort of
  (key, position) pairs: it maximises the descending list of values and takes the
  lexicographically smallest position set among the maxima);
* the closed form of short rows (L <= k: positions 0 .. L-1, then -1);
* the complete invariant check of tests/checks.py on medium rows of every
  generator, with and without exact duplicates;
* torch.topk (CPU) on continuous data without duplicate values;
* cross-form identities: identity page table == raw, un-mapped permuted table
  == raw, ragged row minus its start == raw of that row, window starting at 0 ==
  raw, window minus its start == raw of the window's columns;
* brute force over tiny windows (every k-subset of the window's columns).

Run as a script (``python tests/oracle_pins.py <liboracle.so>``) it runs every pin
but the torch one on the given library and exits 0 only if all pass; the
planted-mistake test uses that to show that each mistake is caught.
"""

from __future__ import annotations

import itertools
import math
import os
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
for _p in (_ROOT, _HERE):
    if _p not in sys.path:
        sys.path.insert(0, _p)

import workloads  # noqa: E402
from checks import check_selection, check_workload, unmap_paged  # noqa: E402
from golden import load_cases  # noqa: E402


def run_case(o, c):
    if c.form == "raw":
        return o.topk_raw(c.scores, c.seq_lens, c.k, 1)
    if c.form == "paged":
        return o.topk_paged(c.scores, c.seq_lens, c.page_table, c.page_size, c.k, 1)
    if c.form == "window":
        return o.topk_window(c.scores, c.row_starts, c.seq_lens, c.k, 1)
    return o.topk_ragged(c.scores, c.row_starts, c.seq_lens, c.k, 1)


def pin_golden(o):
    for c in load_cases():
        got = np.sort(run_case(o, c), axis=1)
        exp = np.sort(c.expect, axis=1)
        assert got.shape == exp.shape and (got == exp).all(), (
            f"golden case {c.name}: got {got.tolist()}, expected {exp.tolist()}")
        if c.expect_sorted is None:
            continue
        w = workloads.Workload(c.name, c.form, c.k, c.scores, c.seq_lens, c.page_table,
                               c.page_size, c.row_starts)
        pos, vals = o.run_values(w, 1)
        assert (pos == c.expect_sorted).all(), (
            f"golden case {c.name}: rank order {pos.tolist()}, expected {c.expect_sorted.tolist()}")
        assert (vals.view(np.uint32) == c.expect_values.view(np.uint32)).all(), (
            f"golden case {c.name}: values {vals.tolist()}, expected {c.expect_values.tolist()}")


def _value_order(x: float):
    # float order, with -0.0 just below +0.0
    return (float(x), 0 if (x == 0 and math.copysign(1.0, x) < 0) else 1)


def brute_force(values, k: int) -> set[int]:
    """The exact top-k by enumeration of every k-subset."""
    L = len(values)
    if k >= L:
        return set(range(L))
    best, best_set = None, None
    for comb in itertools.combinations(range(L), k):  # lexicographic order
        score = sorted((_value_order(values[i]) for i in comb), reverse=True)
        if best is None or score > best:
            best, best_set = score, comb
    return set(best_set)


_POOL = np.array([-1.5, -0.0, 0.0, 1e-45, -1e-45, 2.0, 3.0, np.inf, -np.inf, 2.0,
                  1.0000001, 1.0], dtype=np.float32)


def tiny_row(g: np.random.Generator, L: int) -> np.ndarray:
    kind = int(g.integers(0, 7))
    if kind < 5:
        dist = ("normal", "banded", "narrow", "subnormal", "heavy_tail")[kind]
        x = workloads.row_values(g, dist, L)
    elif kind == 5:
        x = _POOL[g.integers(0, _POOL.shape[0], size=L)]
    else:
        x = g.integers(-2, 3, size=L).astype(np.float32)  # heavy ties
    if g.random() < 0.5:
        x = workloads.with_duplicates(g, x, p=0.3)
    return np.asarray(x, dtype=np.float32)


def pin_brute_force(o, trials: int = 1500, seed: int = 7):
    g = np.random.Generator(np.random.PCG64(seed))
    for t in range(trials):
        L = int(g.integers(1, 10))
        k = int(g.integers(1, L + 1)) if g.random() < 0.85 else int(g.integers(L, L + 4))
        row = tiny_row(g, L)
        out = o.topk_raw(row[None, :], np.array([L], np.int32), k, 1)[0]
        exp = brute_force(row, k)
        got = set(int(v) for v in out if v >= 0)
        assert got == exp and int((out == -1).sum()) == k - len(exp), (
            f"trial {t}: row {row.tolist()} k={k}: oracle {out.tolist()}, brute force {sorted(exp)}")
        # rank order: larger value first, equal values by smaller position first,
        # then the padding; values are the selected scores, -inf pads
        ranked = sorted(exp, key=lambda i: (tuple(-x for x in _value_order(row[i])), i))
        assert out.tolist() == ranked + [-1] * (k - len(exp)), (
            f"trial {t}: row {row.tolist()} k={k}: oracle order {out.tolist()}, expected {ranked}")
        w = workloads.Workload("bf", "raw", k, row[None, :], np.array([L], np.int32))
        pos, vals = o.run_values(w, 1)
        want = np.array([row[i] for i in ranked] + [-np.inf] * (k - len(exp)), np.float32)
        assert (pos[0] == out).all() and (vals[0].view(np.uint32) == want.view(np.uint32)).all(), (
            f"trial {t}: values {vals[0].tolist()}, expected {want.tolist()}")


def pin_brute_force_window(o, trials: int = 600, seed: int = 29):
    """Windows [start, end) of tiny rows, including ends outside the row and empty
    windows, against enumeration over the window's columns."""
    g = np.random.Generator(np.random.PCG64(seed))
    for t in range(trials):
        stride = int(g.integers(1, 10))
        row = tiny_row(g, stride)
        start = int(g.integers(-2, stride + 2))
        end = int(g.integers(-1, stride + 3))
        k = int(g.integers(1, stride + 3))
        out = o.topk_window(row[None, :], np.array([start], np.int32), np.array([end], np.int32),
                            k, 1)[0]
        lo, hi = min(max(start, 0), stride), min(max(end, 0), stride)
        cols = list(range(lo, hi)) if hi > lo else []
        exp = {cols[i] for i in brute_force([row[c] for c in cols], k)} if cols else set()
        got = set(int(v) for v in out if v >= 0)
        assert got == exp and int((out == -1).sum()) == k - len(exp), (
            f"trial {t}: row {row.tolist()} [{start}, {end}) k={k}: oracle {out.tolist()}, "
            f"brute force {sorted(exp)}")


def pin_closed_form(o, seed: int = 11):
    g = np.random.Generator(np.random.PCG64(seed))
    for k in (1, 3, 1024, 2048):
        for L in sorted({0, 1, k // 2, k - 1, k}):
            if L < 0:
                continue
            stride = max(L, 1) + int(g.integers(0, 5))
            row = workloads.normal(g, (1, stride))
            out = o.topk_raw(row, np.array([L], np.int32), k, 1)[0]
            exp = np.concatenate([np.arange(L), np.full(k - L, -1)])
            assert (np.sort(out) == np.sort(exp)).all(), f"short row L={L} k={k}"


def pin_invariants(o, seed: int = 13):
    g = np.random.Generator(np.random.PCG64(seed))
    for dist in workloads.DISTRIBUTIONS:
        for dup in (False, True):
            for k in (1, 7, 100, 1024):
                B, stride = 3, int(g.integers(1100, 3000))
                scores = workloads.random_rows(g, B, stride, dist, dup)
                seq = g.integers(stride // 2, stride + 3, size=B).astype(np.int32)
                out = o.topk_raw(scores, seq, k, 2)
                for b in range(B):
                    L = min(int(seq[b]), stride)
                    msg = check_selection(scores[b], L, k, out[b])
                    assert msg is None, f"{dist} dup={dup} k={k} row {b}: {msg}"


def pin_torch_topk(o, seed: int = 17):
    import torch
    g = np.random.Generator(np.random.PCG64(seed))
    for (B, n, k) in ((1, 2048, 1024), (4, 8192, 1024), (2, 32768, 1024), (2, 20000, 2048)):
        # continuous values without repeats: distinct N(0,1) draws in random order
        x = np.stack([g.permutation(np.unique(workloads.normal(g, 2 * n)))[:n]
                      for _ in range(B)])
        for b in range(B):
            assert np.unique(x[b]).shape[0] == n, "fixture must hold no duplicate values"
        ref = torch.topk(torch.from_numpy(x), k, dim=-1, sorted=False).indices.numpy()
        got = o.topk_raw(x, np.full(B, n, np.int32), k, 0)
        assert (np.sort(ref, 1) == np.sort(got, 1)).all(), "index sets differ from torch.topk"
        vals_ref = np.sort(np.take_along_axis(x, ref, 1), 1)
        vals_got = np.sort(np.take_along_axis(x, got, 1), 1)
        assert (vals_ref.view(np.uint32) == vals_got.view(np.uint32)).all()


def pin_forms(o, seed: int = 19):
    g = np.random.Generator(np.random.PCG64(seed))
    B, stride, ps, k = 4, 3000, 64, 1024
    scores = workloads.random_rows(g, B, stride, "banded", dup=True)
    seq = np.array([stride, 2000, 500, 1025], np.int32)
    raw = o.topk_raw(scores, seq, k, 1)
    n_pages = workloads.pages_for(stride, ps)
    ident = workloads.identity_page_table(B, n_pages)
    assert (o.topk_paged(scores, seq, ident, ps, k, 1) == raw).all(), "identity paged != raw"
    perm = workloads.permuted_page_table(g, B, n_pages)
    paged = o.topk_paged(scores, seq, perm, ps, k, 1)
    for b in range(B):
        assert (unmap_paged(paged[b], perm[b], ps) == raw[b]).all(), f"paged row {b} != raw"
    # ragged: the same rows packed back to back at odd offsets
    lens = np.minimum(seq, stride)
    starts = np.concatenate([[3], 3 + np.cumsum(lens + 5)[:-1]]).astype(np.int32)
    packed = np.zeros(int(starts[-1] + lens[-1] + 7), np.float32)
    for b in range(B):
        packed[starts[b]:starts[b] + lens[b]] = scores[b, :lens[b]]
    rag = o.topk_ragged(packed, starts, lens.astype(np.int32), k, 1)
    for b in range(B):
        un = np.where(rag[b] >= 0, rag[b] - starts[b], -1)
        assert (un == raw[b]).all(), f"ragged row {b} != raw"
    w = workloads.Workload("forms", "ragged", k, packed, lens.astype(np.int32), None, ps, starts)
    assert not check_workload(w, rag)
    # window: starting at column 0 it is the raw form; otherwise, minus its start,
    # it is the raw form of the window's columns
    zero = np.zeros(B, np.int32)
    assert (o.topk_window(scores, zero, seq, k, 1) == raw).all(), "window from 0 != raw"
    wst = np.array([7, 1500, 0, 24], np.int32)
    wen = np.array([2900, 2000, 499, 3100], np.int32)
    win = o.topk_window(scores, wst, wen, k, 1)
    for b in range(B):
        hi = min(int(wen[b]), stride)
        part = o.topk_raw(scores[b:b + 1, wst[b]:hi], np.array([hi - wst[b]], np.int32), k, 1)[0]
        shifted = np.where(part >= 0, part + wst[b], -1)
        assert (win[b] == shifted).all(), f"window row {b} != raw of its columns"
    ww = workloads.Workload("forms", "window", k, scores, wen, None, ps, wst)
    assert not check_workload(ww, win)


def pin_threads(o, seed: int = 23):
    g = np.random.Generator(np.random.PCG64(seed))
    scores = workloads.random_rows(g, 9, 4000, "narrow", dup=True)
    seq = g.integers(1, 4001, size=9).astype(np.int32)
    assert (o.topk_raw(scores, seq, 1024, 1) == o.topk_raw(scores, seq, 1024, 4)).all()


CPU_PINS = (pin_golden, pin_brute_force, pin_brute_force_window, pin_closed_form, pin_invariants,
            pin_forms, pin_threads)


def main(argv):
    import oracle
    o = oracle.Oracle(argv[1])
    failed = []
    for pin in CPU_PINS:
        try:
            pin(o)
        except AssertionError as e:
            failed.append(f"{pin.__name__}: {str(e)[:200]}")
    for f in failed:
        print("FAIL", f)
    return 1 if failed else 0


if __name__ == "__main__":
    sys.exit(main(sys.argv))
