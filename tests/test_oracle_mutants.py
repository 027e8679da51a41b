"""Planted mistakes in the oracle are caught by its pins.

Each case copies oracle/topk_oracle.cpp, changes one line into a plausible
mistake, builds it, and runs every CPU pin on it in a child process (a mistake
may read out of bounds, so it must not run in this process). The child must
fail. This shows that the pins constrain each part of the definition.
"""

import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))

MUTANTS = [
    ("negatives_not_inverted",
     "if (bits & 0x80000000u) return ~bits;", "if (bits & 0x80000000u) return bits ^ 0x80000000u;"),
    ("positives_sign_not_set", "return bits | 0x80000000u;", "return bits;"),
    ("ascending_order", "return a.key > b.key; });", "return a.key < b.key; });"),
    ("larger_position_wins_ties", "return a.key > b.key; });",
     "return a.key > b.key || (a.key == b.key && a.pos > b.pos); });"),
    ("unstable_sort", "std::stable_sort(", "std::sort("),
    ("paged_page_and_offset_swapped",
     "v = pt[j / job.page_size] * job.page_size + j % job.page_size;",
     "v = pt[j % job.page_size] * job.page_size + j / job.page_size;"),
    ("paged_missing_page_size", "v = pt[j / job.page_size] * job.page_size + j % job.page_size;",
     "v = pt[j / job.page_size] + j % job.page_size;"),
    ("ragged_offset_dropped", "v = job.row_starts[b] + j;", "v = j;"),
    ("pad_with_zero", "for (int64_t i = m; i < job.k; ++i) out[i] = -1;",
     "for (int64_t i = m; i < job.k; ++i) out[i] = 0;"),
    ("no_clamp_to_row", "L = std::min<int64_t>(std::max<int64_t>(s, 0), job.row_stride);",
     "L = std::max<int64_t>(s, 0);"),
    ("row_stride_ignored", "row = job.scores + b * job.row_stride;",
     "row = job.scores + b * job.k;"),
    ("window_offset_dropped", "v = static_cast<int32_t>(lo + j);", "v = j;"),
    ("window_length_is_end", "L = hi > lo ? hi - lo : 0;", "L = hi;"),
    ("window_start_below_zero_kept", "lo = std::clamp<int64_t>(job.row_starts[b], 0, job.row_stride);",
     "lo = std::min<int64_t>(job.row_starts[b], job.row_stride);"),
    ("window_row_not_offset", "row = job.scores + b * job.row_stride + lo;",
     "row = job.scores + b * job.row_stride;"),
    ("rank_order_reversed", "for (int64_t i = 0; i < m; ++i) chosen[i] = pairs[i].pos;",
     "for (int64_t i = 0; i < m; ++i) chosen[i] = pairs[m - 1 - i].pos;"),
    ("values_from_first_slot", "for (int64_t i = 0; i < m; ++i) v[i] = row[chosen[i]];",
     "for (int64_t i = 0; i < m; ++i) v[i] = row[chosen[0]];"),
    ("values_padding_zero", "for (int64_t i = m; i < job.k; ++i) v[i] = -INFINITY;",
     "for (int64_t i = m; i < job.k; ++i) v[i] = 0.0f;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "topk_oracle.cpp")).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant = tmp_path / "mutant.cpp"
    mutant.write_text(src.replace(old, new))
    lib = oracle.compile_library(str(mutant), str(tmp_path / "libmutant.so"))
    r = subprocess.run([sys.executable, os.path.join(HERE, "oracle_pins.py"), lib],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mistake {name} passed every pin:\n{r.stdout}\n{r.stderr}"
