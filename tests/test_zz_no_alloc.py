"""The grouped call that allocates nothing (topk_transform_grouped_static), on the GPU.

Some callers cannot allocate device memory while they run: a plug-in that a host
runtime gives only its input and output buffers, or a serving engine whose
caching allocator has reserved the device's memory, where a cudaMalloc would fail
or synchronise every stream mid-step. topk_transform_grouped_static stages the
sorted option's (key, position) pairs in a fixed 16 MiB array inside the library
instead of a caller workspace. This test calls it through the C ABI twice in a
row, on different problems each time (the array keeps the previous call's
contents), and checks every output and value against the entry point that takes
a caller-allocated workspace, topk_transform_grouped, on the same inputs. Both
are integer selections, so the comparison is exact.

The file is named so that pytest collects it last; it passes alone in a fresh
process too.
"""

from __future__ import annotations

import numpy as np
import pytest

import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_attention_indexer_sm_gb300 as p
    p.load_library()
    return p


def _problem(w, dev, sorted_):
    q = {"form": w.form, "k": w.k, "sorted": sorted_,
         "scores": torch.from_numpy(np.ascontiguousarray(w.scores)).to(dev),
         "seq_lens": torch.from_numpy(np.ascontiguousarray(w.seq_lens)).to(dev),
         "out": torch.full((w.batch, w.k), -7, dtype=torch.int32, device=dev),
         "values": torch.full((w.batch, w.k), 7.0, dtype=torch.float32, device=dev)}
    if w.form == "paged":
        q["page_table"] = torch.from_numpy(np.ascontiguousarray(w.page_table)).to(dev)
        q["page_size"] = w.page_size
    elif w.form == "ragged":
        q["row_starts"] = torch.from_numpy(np.ascontiguousarray(w.row_starts)).to(dev)
        q["max_row_len_hint"] = int(np.max(w.seq_lens, initial=0))
    elif w.form == "window":
        q["starts"] = torch.from_numpy(np.ascontiguousarray(w.row_starts)).to(dev)
        q["max_row_len_hint"] = w.max_row_len
    return q


def _run(pkg, ws, sorted_flags, static):
    dev = torch.device("cuda:0")
    probs = [_problem(w, dev, s) for w, s in zip(ws, sorted_flags)]
    pkg.topk_transform_grouped(probs, static_workspace=static)
    torch.cuda.synchronize()
    return [(q["out"].cpu().numpy(), q["values"].cpu().numpy()) for q in probs]


def _calls():
    """Two groups of problems: sorted ones of several forms, one unsorted. The
    second call stages fewer, shorter rows than the first, so a slot it failed to
    write would still hold the first call's pair."""
    g = np.random.Generator(np.random.PCG64(2024))
    ties = workloads.Workload("no_alloc_ties", "raw", 500, np.round(
        workloads.random_rows(g, 6, 4000, "normal"), 1).astype(np.float32),
        np.array([4000, 3999, 300, 0, 2500, 501], np.int32))
    first = ([workloads.config3(64), workloads.config4("banded", batch=3),
              workloads.prefill_windows(48, 6000, window=2000), ties, workloads.config2(8192, batch=8)],
             [True, True, True, True, False])
    second = ([workloads.config2(8192, batch=12, seed=77), workloads.config5(1),
               workloads.config3(8, "raw")],
              [True, True, True])
    return [first, second]


def test_no_alloc_call_matches_workspace_call_twice(pkg):
    pkg.topk_reset_guard_hits()
    for ws, flags in _calls():
        got = _run(pkg, ws, flags, static=True)
        exp = _run(pkg, ws, flags, static=False)
        for w, s, (o, v), (eo, ev) in zip(ws, flags, got, exp):
            if s:  # rank order: slot by slot
                assert np.array_equal(o, eo), f"{w.name}: outputs differ"
                assert np.array_equal(v.view(np.uint32), ev.view(np.uint32)), f"{w.name}: values differ"
            else:  # unspecified order: compare as sets, with each value following its slot
                oo, eo_ = np.argsort(o, axis=1), np.argsort(eo, axis=1)
                assert np.array_equal(np.sort(o, axis=1), np.sort(eo, axis=1)), f"{w.name}: outputs differ"
                assert np.array_equal(np.take_along_axis(v, oo, 1).view(np.uint32),
                                      np.take_along_axis(ev, eo_, 1).view(np.uint32)), f"{w.name}: values differ"
            assert (o >= -1).all() and (o != -7).all(), f"{w.name}: unwritten output slots"
    assert pkg.topk_guard_hits() == 0
