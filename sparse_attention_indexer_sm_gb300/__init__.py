"""Exact per-row top-k transform of sparse-attention indexer scores on GB300.

A thin ctypes binding over the C ABI in ``include/topk_transform.h``: the Python
functions carry the C entry points' names, check and marshal torch tensors, and
call the library on the tensors' device and the current torch stream. All the
work runs in the library's sm_103a kernels; there is no fallback. If the library
has not been built, or a tensor is not on a CUDA device, the call raises.

    out = topk_transform_paged(scores, seq_lens, page_table, page_size=64, k=1024)

``scores`` is fp32 [B, row_stride] with unit inner stride (raw/paged) or a packed
1-D buffer (ragged). Rows of ``out`` hold the selected positions, mapped, in an
unspecified order, followed by -1 where a row has fewer than k positions.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

__all__ = [
    "TopkError", "TOPK_MAX_K", "TOPK_TIE_CAPACITY_MAX", "library_path", "load_library",
    "topk_transform_raw", "topk_transform_paged", "topk_transform_ragged", "topk_transform_window",
    "topk_transform_grouped", "TopkProblem", "TOPK_MAX_GROUP", "TOPK_FLAG_SORTED",
    "topk_set_cta_threads", "topk_guard_hits", "topk_reset_guard_hits",
    "topk_workspace_bytes", "topk_set_row_split", "topk_set_tie_capacity", "topk_set_fast_tier",
    "topk_set_staged_tier", "topk_set_chip_split",
]

TOPK_MAX_K = 2048
TOPK_TIE_CAPACITY_MAX = 4096

_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported k", 3: "workspace too small",
           4: "CUDA error"}

_lock = threading.Lock()
_lib = None


class TopkError(RuntimeError):
    """A non-OK status from the library."""


def library_path() -> str:
    return _build.LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it first (python -m "
                    "sparse_attention_indexer_sm_gb300.build, or __graft_entry__.build())")
            lib = ctypes.CDLL(path)
            vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
            lib.topk_workspace_bytes.restype = sz
            lib.topk_workspace_bytes.argtypes = [i32, i64, i32]
            lib.topk_transform_raw.restype = ctypes.c_int
            lib.topk_transform_raw.argtypes = [vp, i64, vp, i32, i32, vp, vp, sz, vp]
            lib.topk_transform_paged.restype = ctypes.c_int
            lib.topk_transform_paged.argtypes = [vp, i64, vp, vp, i64, i32, i32, i32, vp, vp, sz, vp]
            lib.topk_transform_ragged.restype = ctypes.c_int
            lib.topk_transform_ragged.argtypes = [vp, vp, vp, i64, i32, i32, vp, vp, sz, vp]
            lib.topk_transform_window.restype = ctypes.c_int
            lib.topk_transform_window.argtypes = [vp, i64, vp, vp, i64, i32, i32, vp, vp, sz, vp]
            lib.topk_transform_grouped.restype = ctypes.c_int
            lib.topk_transform_grouped.argtypes = [vp, i32, vp, sz, vp]
            lib.topk_problem_bytes.restype = sz
            lib.topk_problem_bytes.argtypes = []
            lib.topk_transform_grouped_static.restype = ctypes.c_int
            lib.topk_transform_grouped_static.argtypes = [vp, i32, vp]
            lib.topk_problem_workspace_bytes.restype = sz
            lib.topk_problem_workspace_bytes.argtypes = [vp, i32]
            if lib.topk_problem_bytes() != ctypes.sizeof(TopkProblem):
                raise RuntimeError("topk_problem_t layout differs between the library and "
                                   "this binding")
            lib.topk_status_string.restype = ctypes.c_char_p
            lib.topk_status_string.argtypes = [ctypes.c_int]
            lib.topk_last_cuda_error.restype = ctypes.c_int
            lib.topk_last_cuda_error.argtypes = []
            lib.topk_set_row_split.restype = ctypes.c_int
            lib.topk_set_row_split.argtypes = [ctypes.c_int]
            lib.topk_set_tie_capacity.restype = ctypes.c_int
            lib.topk_set_tie_capacity.argtypes = [ctypes.c_int]
            lib.topk_guard_hits.restype = ctypes.c_int
            lib.topk_guard_hits.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
            lib.topk_reset_guard_hits.restype = ctypes.c_int
            lib.topk_reset_guard_hits.argtypes = []
            lib.topk_set_cta_threads.restype = ctypes.c_int
            lib.topk_set_cta_threads.argtypes = [ctypes.c_int]
            lib.topk_set_fast_tier.restype = ctypes.c_int
            lib.topk_set_fast_tier.argtypes = [ctypes.c_int]
            lib.topk_set_staged_tier.restype = ctypes.c_int
            lib.topk_set_staged_tier.argtypes = [ctypes.c_int]
            lib.topk_set_chip_split.restype = ctypes.c_int
            lib.topk_set_chip_split.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def _check(status: int, what: str) -> None:
    if status != 0:
        lib = load_library()
        msg = lib.topk_status_string(status).decode()
        if status == 4:
            msg += f" (cudaError {lib.topk_last_cuda_error()})"
        raise TopkError(f"{what}: {msg}")


def _cuda_tensor(t: torch.Tensor, name: str, dtype: torch.dtype, device=None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device (the library has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _vector(t: torch.Tensor, name: str, n: int, device) -> None:
    _cuda_tensor(t, name, torch.int32, device)
    if t.dim() != 1 or t.shape[0] != n or (n > 1 and t.stride(0) != 1):
        raise ValueError(f"{name} must be a contiguous int32 vector of length {n}")


def _out(out, batch: int, k: int, device) -> torch.Tensor:
    if out is None:
        return torch.empty((batch, k), dtype=torch.int32, device=device)
    _cuda_tensor(out, "out", torch.int32, device)
    if tuple(out.shape) != (batch, k) or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous int32 tensor of shape ({batch}, {k})")
    return out


def _stream(stream, device) -> int:
    s = torch.cuda.current_stream(device) if stream is None else stream
    return int(s.cuda_stream)


def _workspace(lib, workspace, batch: int, max_row_len: int, k: int, device, stream):
    """(pointer, bytes) of the call's workspace: the caller's uint8 tensor, else one
    allocated here when topk_workspace_bytes asks for one (the chip-wide split)."""
    if workspace is not None:
        _cuda_tensor(workspace, "workspace", torch.uint8, device)
        if not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous uint8 tensor")
        return workspace.data_ptr(), int(workspace.numel()), workspace
    with torch.cuda.device(device):
        nbytes = int(lib.topk_workspace_bytes(batch, max_row_len, k))
    if nbytes == 0:
        return None, 0, None
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    if stream is not None:
        ws.record_stream(stream)  # in use on that stream until the call's kernels end
    return ws.data_ptr(), nbytes, ws


def _scores_2d(scores: torch.Tensor):
    _cuda_tensor(scores, "scores", torch.float32)
    if scores.dim() != 2 or not scores.is_contiguous() or scores.shape[1] < 1:
        raise ValueError("scores must be a contiguous [batch, row_stride] fp32 tensor, row_stride >= 1")
    return int(scores.shape[0]), int(scores.shape[1])


def topk_workspace_bytes(batch: int, max_row_len: int, k: int) -> int:
    return int(load_library().topk_workspace_bytes(batch, max_row_len, k))


def topk_transform_raw(scores: torch.Tensor, seq_lens: torch.Tensor, k: int,
                       out: torch.Tensor | None = None, stream=None,
                       workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Exact top-k positions of each row of ``scores`` (raw form). workspace: a uint8
    device tensor of topk_workspace_bytes (else allocated here when needed)."""
    lib = load_library()
    batch, row_stride = _scores_2d(scores)
    dev = scores.device
    _vector(seq_lens, "seq_lens", batch, dev)
    out = _out(out, batch, k, dev)
    ws, ws_bytes, _keep = _workspace(lib, workspace, batch, row_stride, k, dev, stream)
    with torch.cuda.device(dev):
        st = lib.topk_transform_raw(scores.data_ptr(), row_stride, seq_lens.data_ptr(), batch, k,
                                    out.data_ptr(), ws, ws_bytes, _stream(stream, dev))
    _check(st, "topk_transform_raw")
    return out


def topk_transform_paged(scores: torch.Tensor, seq_lens: torch.Tensor, page_table: torch.Tensor,
                         page_size: int, k: int, out: torch.Tensor | None = None,
                         stream=None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Exact top-k of each row, each position j written as
    page_table[b, j // page_size] * page_size + j % page_size."""
    lib = load_library()
    batch, row_stride = _scores_2d(scores)
    dev = scores.device
    _vector(seq_lens, "seq_lens", batch, dev)
    _cuda_tensor(page_table, "page_table", torch.int32, dev)
    if page_table.dim() != 2 or page_table.shape[0] != batch or (
            page_table.shape[1] > 1 and page_table.stride(1) != 1):
        raise ValueError("page_table must be [batch, pages] int32 with unit inner stride")
    pt_stride = int(page_table.stride(0)) if batch > 1 else int(page_table.shape[1])
    if pt_stride < max(int(page_table.shape[1]), 1):
        raise ValueError("page_table rows must not overlap (use .contiguous() on expanded tables)")
    if page_table.shape[1] * page_size < min(row_stride, scores.shape[1]):
        raise ValueError("page_table has too few pages for the rows")
    out = _out(out, batch, k, dev)
    ws, ws_bytes, _keep = _workspace(lib, workspace, batch, row_stride, k, dev, stream)
    with torch.cuda.device(dev):
        st = lib.topk_transform_paged(scores.data_ptr(), row_stride, seq_lens.data_ptr(),
                                      page_table.data_ptr(), pt_stride, page_size, batch, k,
                                      out.data_ptr(), ws, ws_bytes, _stream(stream, dev))
    _check(st, "topk_transform_paged")
    return out


def topk_transform_ragged(scores: torch.Tensor, row_starts: torch.Tensor, seq_lens: torch.Tensor,
                          k: int, max_row_len_hint: int = 0, out: torch.Tensor | None = None,
                          stream=None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Exact top-k of packed rows scores[row_starts[b] : row_starts[b] + seq_lens[b]];
    each position j is written as row_starts[b] + j."""
    lib = load_library()
    _cuda_tensor(scores, "scores", torch.float32)
    if scores.dim() != 1 or (scores.numel() > 1 and scores.stride(0) != 1):
        raise ValueError("ragged scores must be a contiguous 1-D fp32 tensor")
    dev = scores.device
    batch = int(row_starts.shape[0]) if row_starts.dim() == 1 else -1
    _vector(row_starts, "row_starts", batch, dev)
    _vector(seq_lens, "seq_lens", batch, dev)
    out = _out(out, batch, k, dev)
    ws, ws_bytes, _keep = _workspace(lib, workspace, batch, int(max_row_len_hint), k, dev, stream)
    with torch.cuda.device(dev):
        st = lib.topk_transform_ragged(scores.data_ptr(), row_starts.data_ptr(),
                                       seq_lens.data_ptr(), int(max_row_len_hint), batch, k,
                                       out.data_ptr(), ws, ws_bytes, _stream(stream, dev))
    _check(st, "topk_transform_ragged")
    return out


def topk_transform_window(scores: torch.Tensor, starts: torch.Tensor, seq_lens: torch.Tensor,
                          k: int, max_row_len_hint: int = 0, out: torch.Tensor | None = None,
                          stream=None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Exact top-k of each row's window of columns [starts[b], seq_lens[b]) (both
    clamped to the row); the selected columns are written. max_row_len_hint: an
    upper bound of the window lengths (0: the row length), used only to pick the
    kernel configuration."""
    lib = load_library()
    batch, row_stride = _scores_2d(scores)
    dev = scores.device
    _vector(starts, "starts", batch, dev)
    _vector(seq_lens, "seq_lens", batch, dev)
    out = _out(out, batch, k, dev)
    hint = int(max_row_len_hint) if 0 < int(max_row_len_hint) < row_stride else row_stride
    ws, ws_bytes, _keep = _workspace(lib, workspace, batch, hint, k, dev, stream)
    with torch.cuda.device(dev):
        st = lib.topk_transform_window(scores.data_ptr(), row_stride, starts.data_ptr(),
                                       seq_lens.data_ptr(), int(max_row_len_hint), batch, k,
                                       out.data_ptr(), ws, ws_bytes, _stream(stream, dev))
    _check(st, "topk_transform_window")
    return out


TOPK_MAX_GROUP = 32
_FORMS = {"raw": 0, "paged": 1, "ragged": 2, "window": 3}


class TopkProblem(ctypes.Structure):
    """ctypes copy of topk_problem_t (include/topk_transform.h)."""
    _fields_ = [("form", ctypes.c_int32), ("batch", ctypes.c_int32), ("k", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("row_stride", ctypes.c_int64),
                ("page_table_stride", ctypes.c_int64), ("max_row_len_hint", ctypes.c_int64),
                ("scores", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("row_starts", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("values", ctypes.c_void_p), ("flags", ctypes.c_uint32),
                ("reserved", ctypes.c_uint32)]


TOPK_FLAG_SORTED = 1


def topk_transform_grouped(problems: list[dict], stream=None, static_workspace: bool = False,
                           workspace: torch.Tensor | None = None) -> list[torch.Tensor]:
    """Several independent transforms in one call (one launch per form present).

    Each problem is a dict with "form" ("raw", "paged", "ragged" or "window"), "k",
    "scores", "seq_lens" and what its form needs: "page_table" and "page_size"
    (paged), "row_starts" and optionally "max_row_len_hint" (ragged), "starts" and
    optionally "max_row_len_hint" (window); "out" is optional. Options: "values", a
    [batch, k] fp32 device tensor that receives each slot's score (-inf in the
    padding slots), and "sorted": True for the slots in rank order (largest score
    first, equal scores by smaller position first). Sorted problems use a device
    workspace: `workspace` (a uint8 device tensor of at least
    topk_problem_workspace_bytes, owned by the caller), else one this function
    allocates; or, with static_workspace=True, the library's own scratch array
    (topk_transform_grouped_static: no allocation; such calls must not overlap on
    a device). Returns the output tensors, in order."""
    lib = load_library()
    if len(problems) > TOPK_MAX_GROUP:
        raise ValueError(f"at most {TOPK_MAX_GROUP} problems per grouped call")
    arr = (TopkProblem * max(len(problems), 1))()
    outs, dev = [], None
    for i, q in enumerate(problems):
        form = q["form"]
        if form not in _FORMS:
            raise ValueError(f"unknown form {form!r}")
        k = int(q["k"])
        scores = q["scores"]
        d = scores.device
        if dev is None:
            dev = d
        elif d != dev:
            raise ValueError("all problems of a grouped call must be on one device")
        if form == "ragged":
            _cuda_tensor(scores, "scores", torch.float32)
            if scores.dim() != 1 or (scores.numel() > 1 and scores.stride(0) != 1):
                raise ValueError("ragged scores must be a contiguous 1-D fp32 tensor")
            batch = int(q["row_starts"].shape[0])
            _vector(q["row_starts"], "row_starts", batch, d)
            arr[i].row_starts = q["row_starts"].data_ptr()
            arr[i].max_row_len_hint = int(q.get("max_row_len_hint", 0))
        else:
            batch, arr[i].row_stride = _scores_2d(scores)
        _vector(q["seq_lens"], "seq_lens", batch, d)
        if form == "paged":
            pt = q["page_table"]
            _cuda_tensor(pt, "page_table", torch.int32, d)
            if pt.dim() != 2 or pt.shape[0] != batch or (pt.shape[1] > 1 and pt.stride(1) != 1):
                raise ValueError("page_table must be [batch, pages] int32 with unit inner stride")
            pt_stride = int(pt.stride(0)) if batch > 1 else int(pt.shape[1])
            if pt_stride < max(int(pt.shape[1]), 1):
                raise ValueError("page_table rows must not overlap (use .contiguous() on expanded tables)")
            if pt.shape[1] * int(q["page_size"]) < scores.shape[1]:
                raise ValueError("page_table has too few pages for the rows")
            arr[i].page_table = pt.data_ptr()
            arr[i].page_table_stride = pt_stride
            arr[i].page_size = int(q["page_size"])
        elif form == "window":
            _vector(q["starts"], "starts", batch, d)
            arr[i].row_starts = q["starts"].data_ptr()
            arr[i].max_row_len_hint = int(q.get("max_row_len_hint", 0))
        out = _out(q.get("out"), batch, k, d)
        vals = q.get("values")
        if vals is not None:
            _cuda_tensor(vals, "values", torch.float32, d)
            if tuple(vals.shape) != (batch, k) or not vals.is_contiguous():
                raise ValueError(f"values must be a contiguous fp32 tensor of shape ({batch}, {k})")
            arr[i].values = vals.data_ptr()
        arr[i].flags = TOPK_FLAG_SORTED if q.get("sorted", False) else 0
        arr[i].form, arr[i].batch, arr[i].k = _FORMS[form], batch, k
        arr[i].scores, arr[i].seq_lens, arr[i].out = scores.data_ptr(), q["seq_lens"].data_ptr(), out.data_ptr()
        outs.append(out)
    if not problems:
        return outs
    if static_workspace:
        with torch.cuda.device(dev):
            st = lib.topk_transform_grouped_static(ctypes.addressof(arr), len(problems),
                                                   _stream(stream, dev))
        _check(st, "topk_transform_grouped_static")
        return outs
    ws_bytes = int(lib.topk_problem_workspace_bytes(ctypes.addressof(arr), len(problems)))
    if workspace is not None:
        _cuda_tensor(workspace, "workspace", torch.uint8, dev)
        if not workspace.is_contiguous() or workspace.numel() < ws_bytes:
            raise ValueError(f"workspace must be a contiguous uint8 tensor of at least {ws_bytes} bytes")
        with torch.cuda.device(dev):
            st = lib.topk_transform_grouped(ctypes.addressof(arr), len(problems),
                                            workspace.data_ptr() if ws_bytes else None,
                                            workspace.numel(), _stream(stream, dev))
        _check(st, "topk_transform_grouped")
        return outs
    with torch.cuda.device(dev):
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
        st = lib.topk_transform_grouped(ctypes.addressof(arr), len(problems),
                                        ws.data_ptr() if ws is not None else None, ws_bytes,
                                        _stream(stream, dev))
        if ws is not None:  # the launches on `stream` read it until they finish
            ws.record_stream(torch.cuda.current_stream(dev) if stream is None else stream)
    _check(st, "topk_transform_grouped")
    return outs


def topk_set_row_split(g: int) -> int:
    """CTAs per row (1, 2, 4, 8, 16); g < 1 restores the built-in choice."""
    return int(load_library().topk_set_row_split(int(g)))


def topk_set_tie_capacity(cap: int) -> int:
    """Entries of the shared tie buffer (0 .. TOPK_TIE_CAPACITY_MAX); for tests."""
    return int(load_library().topk_set_tie_capacity(int(cap)))


def topk_guard_hits() -> int:
    """Failed internal consistency checks on the current device (0 unless inputs
    changed while a kernel ran, or a bug); waits for the device's pending work."""
    n = ctypes.c_uint64(0)
    _check(load_library().topk_guard_hits(ctypes.byref(n)), "topk_guard_hits")
    return int(n.value)


def topk_reset_guard_hits() -> None:
    _check(load_library().topk_reset_guard_hits(), "topk_reset_guard_hits")


def topk_set_cta_threads(threads: int) -> int:
    """Which kernel build runs: 512 or 256 threads per CTA; anything else restores
    the built-in choice (returned as 0)."""
    return int(load_library().topk_set_cta_threads(int(threads)))


def topk_set_fast_tier(enable: bool) -> int:
    """1: try the sampled-threshold one-pass filter first (default); 0: exact tier only."""
    return int(load_library().topk_set_fast_tier(1 if enable else 0))


def topk_set_chip_split(mode: int) -> int:
    """When single-form calls take the chip-wide split (many CTAs per row, candidates
    through a device workspace): 1 automatic (default), 2 for every batch and row
    length, 0 never."""
    return int(load_library().topk_set_chip_split(int(mode)))


def topk_set_staged_tier(mode: int) -> int:
    """Where single-CTA rows of at most 32768 elements run on the staged tier (the row
    copied to shared memory from kernel start): 1 automatic (default), 2 always with
    the whole row staged, 3 always with half a row staged, 0 never."""
    return int(load_library().topk_set_staged_tier(int(mode)))
