"""CPU oracle for the exact per-row top-k transform (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
legs of ``bench.py`` may import this package. The product library never does: it
shares no code with the oracle and fails loudly when its own CUDA build is
missing.

The arithmetic lives in ``topk_oracle.cpp`` (the plain definition: order-preserving
key, stable sort by key descending, first min(k, L) positions, mapped, -1 padded).
This module only compiles it with the host C++ compiler and marshals numpy arrays.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "topk_oracle.cpp")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libtopk_oracle.so")

_lock = threading.Lock()
_default = None


def compile_library(src: str, out_path: str) -> str:
    """Compile one oracle source file into a shared library (g++, -O2)."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".{os.getpid()}.tmp"
    cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", "-o", tmp, src]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libtopk_oracle.so`` if stale."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        compile_library(_SRC, _LIB_PATH)
    return _LIB_PATH


def _f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


class Oracle:
    """numpy front end of one compiled oracle library."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        i32p = ctypes.POINTER(ctypes.c_int32)
        f32p = ctypes.POINTER(ctypes.c_float)
        lib.oracle_order_key.restype = ctypes.c_uint32
        lib.oracle_order_key.argtypes = [ctypes.c_float]
        lib.oracle_usable_cores.restype = ctypes.c_int
        lib.oracle_usable_cores.argtypes = []
        lib.oracle_topk_raw.restype = ctypes.c_int
        lib.oracle_topk_raw.argtypes = [f32p, ctypes.c_int64, i32p, ctypes.c_int32,
                                        ctypes.c_int32, i32p, ctypes.c_int]
        lib.oracle_topk_paged.restype = ctypes.c_int
        lib.oracle_topk_paged.argtypes = [f32p, ctypes.c_int64, i32p, i32p, ctypes.c_int64,
                                          ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                          i32p, ctypes.c_int]
        lib.oracle_topk_ragged.restype = ctypes.c_int
        lib.oracle_topk_ragged.argtypes = [f32p, i32p, i32p, ctypes.c_int32,
                                           ctypes.c_int32, i32p, ctypes.c_int]
        lib.oracle_topk_values.restype = ctypes.c_int
        lib.oracle_topk_values.argtypes = [ctypes.c_int32, f32p, ctypes.c_int64, i32p, i32p, i32p,
                                           ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_int32, i32p, f32p, ctypes.c_int]
        lib.oracle_topk_window.restype = ctypes.c_int
        lib.oracle_topk_window.argtypes = [f32p, ctypes.c_int64, i32p, i32p, ctypes.c_int32,
                                           ctypes.c_int32, i32p, ctypes.c_int]
        self.lib = lib
        self.path = lib_path

    def order_key(self, x: float) -> int:
        """Order-preserving 32-bit key of one fp32 value."""
        return int(self.lib.oracle_order_key(ctypes.c_float(x)))

    def usable_cores(self) -> int:
        return int(self.lib.oracle_usable_cores())

    def topk_raw(self, scores, seq_lens, k: int, threads: int = 0) -> np.ndarray:
        """scores [B, row_stride] fp32, seq_lens [B] int32 -> positions [B, k] int32."""
        s, sp = _f32(scores)
        if s.ndim != 2:
            raise ValueError("scores must be [batch, row_stride]")
        L, lp = _i32(seq_lens)
        if L.shape != (s.shape[0],):
            raise ValueError("seq_lens must be [batch]")
        out = np.empty((s.shape[0], k), dtype=np.int32)
        _, op = _i32(out)
        rc = self.lib.oracle_topk_raw(sp, s.shape[1], lp, s.shape[0], k, op, threads)
        if rc != 0:
            raise ValueError(f"oracle_topk_raw: invalid arguments (status {rc})")
        return out

    def topk_paged(self, scores, seq_lens, page_table, page_size: int, k: int,
                   threads: int = 0) -> np.ndarray:
        """As topk_raw, positions mapped through page_table [B, pages] (int32)."""
        s, sp = _f32(scores)
        if s.ndim != 2:
            raise ValueError("scores must be [batch, row_stride]")
        L, lp = _i32(seq_lens)
        pt, ptp = _i32(page_table)
        if pt.ndim != 2 or pt.shape[0] != s.shape[0] or L.shape != (s.shape[0],):
            raise ValueError("page_table must be [batch, pages] and seq_lens [batch]")
        if pt.shape[1] * page_size < min(s.shape[1], max(int(L.max(initial=0)), 0)):
            raise ValueError("page_table does not cover the rows")
        out = np.empty((s.shape[0], k), dtype=np.int32)
        _, op = _i32(out)
        rc = self.lib.oracle_topk_paged(sp, s.shape[1], lp, ptp, pt.shape[1], page_size,
                                        s.shape[0], k, op, threads)
        if rc != 0:
            raise ValueError(f"oracle_topk_paged: invalid arguments (status {rc})")
        return out

    def topk_ragged(self, scores, row_starts, seq_lens, k: int, threads: int = 0) -> np.ndarray:
        """scores: packed 1-D fp32; row b = scores[row_starts[b] : row_starts[b] + seq_lens[b]]."""
        s, sp = _f32(scores)
        rs, rsp = _i32(row_starts)
        L, lp = _i32(seq_lens)
        B = rs.shape[0]
        if L.shape != (B,):
            raise ValueError("row_starts and seq_lens must both be [batch]")
        if B and (rs.min() < 0 or (rs.astype(np.int64) + np.maximum(L, 0)).max() > s.size):
            raise ValueError("a ragged row runs outside the packed scores buffer")
        out = np.empty((B, k), dtype=np.int32)
        _, op = _i32(out)
        rc = self.lib.oracle_topk_ragged(sp, rsp, lp, B, k, op, threads)
        if rc != 0:
            raise ValueError(f"oracle_topk_ragged: invalid arguments (status {rc})")
        return out

    def topk_window(self, scores, starts, seq_lens, k: int, threads: int = 0) -> np.ndarray:
        """scores [B, row_stride] fp32; row b selects among columns [starts[b],
        seq_lens[b]) (clamped to the row) and emits those columns."""
        s, sp = _f32(scores)
        if s.ndim != 2:
            raise ValueError("scores must be [batch, row_stride]")
        st, stp = _i32(starts)
        L, lp = _i32(seq_lens)
        if st.shape != (s.shape[0],) or L.shape != (s.shape[0],):
            raise ValueError("starts and seq_lens must both be [batch]")
        out = np.empty((s.shape[0], k), dtype=np.int32)
        _, op = _i32(out)
        rc = self.lib.oracle_topk_window(sp, s.shape[1], stp, lp, s.shape[0], k, op, threads)
        if rc != 0:
            raise ValueError(f"oracle_topk_window: invalid arguments (status {rc})")
        return out

    def run_values(self, w, threads: int = 0) -> tuple[np.ndarray, np.ndarray]:
        """Run one ``workloads.Workload`` with the values output: (positions in rank
        order, fp32 values, -inf in the padding slots)."""
        forms = {"raw": 0, "paged": 1, "ragged": 2, "window": 3}
        s, sp = _f32(w.scores)
        B, k = w.batch, w.k
        L, lp = _i32(w.seq_lens)
        rs, rsp = _i32(w.row_starts if w.row_starts is not None else np.zeros(B, np.int32))
        pt, ptp = _i32(w.page_table if w.page_table is not None else np.zeros((B, 1), np.int32))
        if w.form == "ragged" and B and (rs.astype(np.int64) + np.maximum(L, 0)).max() > s.size:
            raise ValueError("a ragged row runs outside the packed scores buffer")
        if w.form == "paged" and pt.shape[1] * w.page_size < min(s.shape[1], max(int(L.max(initial=0)), 0)):
            raise ValueError("page_table does not cover the rows")
        out = np.empty((B, k), dtype=np.int32)
        vals = np.empty((B, k), dtype=np.float32)
        _, op = _i32(out)
        _, vp = _f32(vals)
        stride = s.shape[1] if s.ndim == 2 else 0
        rc = self.lib.oracle_topk_values(forms[w.form], sp, stride, rsp, lp, ptp, pt.shape[1],
                                         w.page_size, B, k, op, vp, threads)
        if rc != 0:
            raise ValueError(f"oracle_topk_values: invalid arguments (status {rc})")
        return out, vals

    def run(self, w, threads: int = 0) -> np.ndarray:
        """Run one ``workloads.Workload``."""
        if w.form == "raw":
            return self.topk_raw(w.scores, w.seq_lens, w.k, threads)
        if w.form == "paged":
            return self.topk_paged(w.scores, w.seq_lens, w.page_table, w.page_size, w.k, threads)
        if w.form == "ragged":
            return self.topk_ragged(w.scores, w.row_starts, w.seq_lens, w.k, threads)
        if w.form == "window":
            return self.topk_window(w.scores, w.row_starts, w.seq_lens, w.k, threads)
        raise ValueError(f"unknown form {w.form!r}")


def default() -> Oracle:
    """The oracle built from ``topk_oracle.cpp`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def order_key(x: float) -> int:
    return default().order_key(x)


def usable_cores() -> int:
    return default().usable_cores()


def topk_raw(scores, seq_lens, k: int, threads: int = 0) -> np.ndarray:
    return default().topk_raw(scores, seq_lens, k, threads)


def topk_paged(scores, seq_lens, page_table, page_size: int, k: int, threads: int = 0) -> np.ndarray:
    return default().topk_paged(scores, seq_lens, page_table, page_size, k, threads)


def topk_ragged(scores, row_starts, seq_lens, k: int, threads: int = 0) -> np.ndarray:
    return default().topk_ragged(scores, row_starts, seq_lens, k, threads)


def topk_window(scores, starts, seq_lens, k: int, threads: int = 0) -> np.ndarray:
    return default().topk_window(scores, starts, seq_lens, k, threads)


def run_values(w, threads: int = 0):
    return default().run_values(w, threads)


def run(w, threads: int = 0) -> np.ndarray:
    return default().run(w, threads)
