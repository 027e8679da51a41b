"""The C-ABI library builds, loads and exports every declared entry point (no GPU).

Only calls that the library rejects before touching CUDA are made here.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


def declared_functions():
    names = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(topk_\w+)\s*\(", text, flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_indexer_sm_gb300 import build
    build.build()
    import sparse_attention_indexer_sm_gb300 as pkg
    return pkg.load_library()


def test_header_declares_every_form():
    names = declared_functions()
    for n in ("topk_transform_raw", "topk_transform_paged", "topk_transform_ragged",
              "topk_transform_window", "topk_transform_grouped", "topk_problem_bytes",
              "topk_workspace_bytes", "topk_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_status_strings(lib):
    for st in range(5):
        assert lib.topk_status_string(st)
    assert b"unknown" in lib.topk_status_string(99)


def test_host_side_argument_checks(lib):
    one = ctypes.c_void_p(16)  # never dereferenced: each call is rejected on the host
    assert lib.topk_transform_raw(one, 8, one, 1, 0, one, None, 0, None) == 2      # k < 1
    assert lib.topk_transform_raw(one, 8, one, 1, 2049, one, None, 0, None) == 2   # k > max
    assert lib.topk_transform_raw(one, 8, one, -1, 16, one, None, 0, None) == 1    # batch < 0
    assert lib.topk_transform_raw(one, 8, one, 0, 16, one, None, 0, None) == 0     # empty batch
    assert lib.topk_transform_raw(None, 8, one, 1, 16, one, None, 0, None) == 1    # null scores
    assert lib.topk_transform_raw(ctypes.c_void_p(18), 8, one, 1, 16, one, None, 0, None) == 1
    assert lib.topk_transform_raw(one, 0, one, 1, 16, one, None, 0, None) == 1     # stride < 1
    assert lib.topk_transform_paged(one, 8, one, None, 1, 64, 1, 16, one, None, 0, None) == 1
    assert lib.topk_transform_paged(one, 8, one, one, 1, 0, 1, 16, one, None, 0, None) == 1
    assert lib.topk_transform_paged(one, 8, one, one, 0, 64, 1, 16, one, None, 0, None) == 1
    assert lib.topk_transform_ragged(one, None, one, 0, 1, 16, one, None, 0, None) == 1
    assert lib.topk_transform_ragged(one, one, one, -1, 1, 16, one, None, 0, None) == 1
    assert lib.topk_workspace_bytes(256, 262144, 2048) == 0  # no device here: no split
    assert lib.topk_workspace_bytes(1, 262144, 2048) == 0
    assert lib.topk_transform_window(one, 8, None, one, 0, 1, 16, one, None, 0, None) == 1
    assert lib.topk_transform_window(one, 0, one, one, 0, 1, 16, one, None, 0, None) == 1
    assert lib.topk_transform_window(one, 8, one, one, -1, 1, 16, one, None, 0, None) == 1
    assert lib.topk_transform_window(one, 8, one, one, 0, 1, 0, one, None, 0, None) == 2


def test_grouped_layout_and_host_checks(lib):
    import sparse_attention_indexer_sm_gb300 as pkg
    P = pkg.TopkProblem
    assert lib.topk_problem_bytes() == ctypes.sizeof(P)
    one = 16  # never dereferenced: every call below is rejected on the host

    def group(*probs):
        arr = (P * max(len(probs), 1))(*probs)
        return lib.topk_transform_grouped(ctypes.addressof(arr), len(probs), None, 0, None)

    ok_raw = P(form=0, batch=2, k=16, row_stride=64, scores=one, seq_lens=one, out=one)
    assert lib.topk_transform_grouped(None, 0, None, 0, None) == 0        # nothing to do
    assert lib.topk_transform_grouped(None, 1, None, 0, None) == 1        # null array
    assert lib.topk_transform_grouped(None, -1, None, 0, None) == 1
    assert lib.topk_transform_grouped(None, pkg.TOPK_MAX_GROUP + 1, None, 0, None) == 1
    assert group(P(form=0, batch=0, k=16)) == 0                           # empty problems only
    assert group(ok_raw, P(form=7, batch=1, k=16)) == 1                   # unknown form
    assert group(ok_raw, P(form=0, batch=1, k=0, row_stride=8, scores=one, seq_lens=one,
                           out=one)) == 2                                 # bad k, second problem
    assert group(ok_raw, P(form=1, batch=1, k=4, row_stride=8, scores=one, seq_lens=one,
                           out=one, page_size=64, page_table_stride=1)) == 1  # no page table
    assert group(ok_raw, P(form=2, batch=1, k=4, scores=one, seq_lens=one, out=one)) == 1
    assert group(ok_raw, P(form=3, batch=1, k=4, row_stride=8, scores=one, seq_lens=one,
                           out=one)) == 1                                 # window without starts
    assert group(P(form=0, batch=1, k=4, row_stride=8, scores=18, seq_lens=one,
                   out=one)) == 1                                         # misaligned scores
    assert group(P(form=0, batch=1, k=4, row_stride=8, scores=one, seq_lens=one, out=one,
                   flags=2)) == 1                                         # unknown flag
    sorted_raw = P(form=0, batch=3, k=100, row_stride=8, scores=one, seq_lens=one, out=one,
                   flags=pkg.TOPK_FLAG_SORTED)
    arr = (P * 2)(ok_raw, sorted_raw)
    need = lib.topk_problem_workspace_bytes(ctypes.addressof(arr), 2)
    assert need == 2560  # 3 * 100 pairs of 8 bytes, rounded up to 256
    assert lib.topk_problem_workspace_bytes(ctypes.addressof(arr), 1) == 0
    assert lib.topk_transform_grouped(ctypes.addressof(arr), 2, None, 0, None) == 3
    assert lib.topk_transform_grouped(ctypes.addressof(arr), 2, ctypes.c_void_p(256), need - 1,
                                      None) == 3
    assert lib.topk_transform_grouped(ctypes.addressof(arr), 2, ctypes.c_void_p(260), need,
                                      None) == 1                         # misaligned workspace
    # the static-scratch call: more staging than the library's array holds
    big = P(form=0, batch=(16 << 20) // (8 * 2048) + 1, k=2048, row_stride=8, scores=one,
            seq_lens=one, out=one, flags=pkg.TOPK_FLAG_SORTED)
    arr1 = (P * 1)(big)
    assert lib.topk_transform_grouped_static(ctypes.addressof(arr1), 1, None) == 3
    # every problem is checked before the array's limit: a problem's own status wins
    bad_k = P(form=0, batch=big.batch, k=2049, row_stride=8, scores=one, seq_lens=one,
              out=one, flags=pkg.TOPK_FLAG_SORTED)
    bad_form = P(form=5, batch=big.batch, k=2048, flags=pkg.TOPK_FLAG_SORTED)
    for probs, status in (((bad_k,), 2), ((bad_form,), 1), ((big, bad_k), 2), ((big, bad_form), 1),
                          ((bad_k, big), 2)):
        arr2 = (P * len(probs))(*probs)
        assert lib.topk_transform_grouped_static(ctypes.addressof(arr2), len(probs), None) == status
        assert lib.topk_transform_grouped(ctypes.addressof(arr2), len(probs), None, 0, None) == status
    assert lib.topk_transform_grouped_static(None, 1, None) == 1
    assert lib.topk_transform_grouped_static(None, 0, None) == 0


def test_cta_threads_control_round_trip(lib):
    prev = lib.topk_set_cta_threads(256)
    assert lib.topk_set_cta_threads(512) == 256
    assert lib.topk_set_cta_threads(7) == 512     # anything else: automatic
    assert lib.topk_set_cta_threads(prev) == 0


def test_tuning_controls_round_trip(lib):
    prev = lib.topk_set_tie_capacity(16)
    assert lib.topk_set_tie_capacity(prev) == 16
    assert lib.topk_set_tie_capacity(10**6) == prev
    assert lib.topk_set_tie_capacity(prev) == 4096
    prev_split = lib.topk_set_row_split(4)
    assert lib.topk_set_row_split(prev_split) == 4


def test_binding_rejects_cpu_tensors():
    torch = pytest.importorskip("torch")
    import sparse_attention_indexer_sm_gb300 as pkg
    x = torch.zeros(2, 8)
    with pytest.raises(ValueError, match="CUDA"):
        pkg.topk_transform_raw(x, torch.full((2,), 8, dtype=torch.int32), 4)
