"""Independent checks of a top-k transform result (used on oracle and GPU outputs).

Nothing here reuses the oracle's key transform: values are compared as floats,
with -0.0 placed just below +0.0, which is the order the order-preserving key
induces on non-NaN values. For a row of valid length L and m = min(k, L), a
selection S (positions, before mapping) is the exact top-k with the
smaller-position-wins rule if and only if

  1. S has m distinct positions, all in [0, L);
  2. no unselected position holds a larger value than any selected one;
  3. at the threshold value tau = min(S), every unselected position holding tau
     comes after every selected position holding tau.

These three conditions determine S uniquely, so they are a complete check.
"""

from __future__ import annotations

import numpy as np


def _rank_values(v: np.ndarray) -> np.ndarray:
    """Dense ranks of fp32 values under float order with -0.0 < +0.0 (no NaN)."""
    v = np.asarray(v, dtype=np.float32)
    if np.isnan(v).any():
        raise ValueError("NaN values are outside the checked domain")
    neg_zero = (v == 0) & np.signbit(v)
    # lexsort: last key is primary. Sort by value, then -0 before +0.
    order = np.lexsort((~neg_zero, v.astype(np.float64)))
    sv = v[order].astype(np.float64)
    snz = neg_zero[order]
    new = np.ones(v.shape[0], dtype=bool)
    if v.shape[0] > 1:
        new[1:] = (sv[1:] != sv[:-1]) | (snz[1:] != snz[:-1])
    dense = np.cumsum(new) - 1
    ranks = np.empty(v.shape[0], dtype=np.int64)
    ranks[order] = dense
    return ranks


def check_selection(row: np.ndarray, L: int, k: int, sel: np.ndarray) -> str | None:
    """Return None if ``sel`` (unmapped positions, -1 padded, any order) is the
    exact top-k of row[:L]; otherwise a description of the first violation."""
    sel = np.asarray(sel, dtype=np.int64)
    m = min(k, max(L, 0))
    if sel.shape[0] != k:
        return f"expected {k} slots, got {sel.shape[0]}"
    pos = sel[sel >= 0]
    n_pad = int((sel == -1).sum())
    if pos.shape[0] != m or n_pad != k - m:
        return f"expected {m} positions and {k - m} x -1, got {pos.shape[0]} and {n_pad}"
    if (sel < -1).any():
        return "a slot holds a negative value other than -1"
    if m == 0:
        return None
    if pos.max() >= L:
        return f"position {int(pos.max())} outside [0, {L})"
    if np.unique(pos).shape[0] != m:
        return "repeated positions"
    if m == L:
        return None
    r = _rank_values(np.asarray(row[:L]))
    chosen = np.zeros(L, dtype=bool)
    chosen[pos] = True
    tau = r[chosen].min()
    best_rest = r[~chosen].max()
    if best_rest > tau:
        return "an unselected value is larger than a selected one"
    if best_rest == tau:
        idx = np.arange(L)
        last_sel = idx[chosen & (r == tau)].max()
        first_rest = idx[~chosen & (r == tau)].min()
        if first_rest < last_sel:
            return (f"tie at the threshold resolved wrongly: position {first_rest} left out, "
                    f"position {last_sel} taken")
    return None


def unmap_paged(out_row: np.ndarray, page_table_row: np.ndarray, page_size: int) -> np.ndarray:
    """Invert the paged mapping for a row whose page table is injective."""
    out_row = np.asarray(out_row, dtype=np.int64)
    pt = np.asarray(page_table_row, dtype=np.int64)
    if np.unique(pt).shape[0] != pt.shape[0]:
        raise ValueError("page table row is not injective")
    inv = {int(p): i for i, p in enumerate(pt)}
    res = np.full(out_row.shape, -1, dtype=np.int64)
    for i, v in enumerate(out_row):
        if v < 0:
            continue
        page, off = divmod(int(v), page_size)
        if page not in inv:
            res[i] = -2  # not a slot of this row's pages: reported as invalid
        else:
            res[i] = inv[page] * page_size + off
    return res


def check_workload(w, out: np.ndarray, max_rows: int | None = None) -> list[str]:
    """Check every row of one ``workloads.Workload`` result; return violations."""
    out = np.asarray(out)
    errors = []
    rows = range(w.batch) if max_rows is None else range(min(w.batch, max_rows))
    for b in rows:
        if w.form in ("ragged", "window"):
            if w.form == "ragged":
                L = max(int(w.seq_lens[b]), 0)
                start = int(w.row_starts[b])
                row = w.scores[start:start + L]
            else:  # columns [start, end) of row b, both clamped to the row
                stride = w.scores.shape[1]
                start = min(max(int(w.row_starts[b]), 0), stride)
                end = min(max(int(w.seq_lens[b]), 0), stride)
                L = max(end - start, 0)
                row = w.scores[b, start:start + L]
            sel = np.where(out[b] >= 0, out[b].astype(np.int64) - start, out[b])
            sel = np.where((out[b] >= 0) & (sel < 0), -2, sel)
        else:
            L = min(max(int(w.seq_lens[b]), 0), w.scores.shape[1])
            row = w.scores[b]
            if w.form == "paged":
                sel = unmap_paged(out[b], w.page_table[b], w.page_size)
            else:
                sel = out[b].astype(np.int64)
        msg = check_selection(row, L, w.k, sel)
        if msg:
            errors.append(f"row {b}: {msg}")
    return errors


def same_sets(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Per-row equality of the two outputs compared as sorted sets; bool [B]."""
    return (np.sort(np.asarray(a), axis=1) == np.sort(np.asarray(b), axis=1)).all(axis=1)
