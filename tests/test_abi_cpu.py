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


def test_header_declares_the_three_forms():
    names = declared_functions()
    for n in ("topk_transform_raw", "topk_transform_paged", "topk_transform_ragged",
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
    assert lib.topk_workspace_bytes(256, 262144, 2048) == 0


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
