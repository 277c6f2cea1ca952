"""ctypes front end of ``topk_oracle.c`` (test infrastructure only).

The oracle is the plain definition of the result: a full sort of every row
(larger score first, IEEE comparison, the smaller position wins a tie),
the page-table transform ``page_table[b][i // P] * P + i % P`` and ``-1``
padding, after SGLang PR #26788 "[JIT Kernel] DeepSeek-V4 DSA indexer: faster
top-k + page-table transform (runtime k <= 2048)", sections "Motivation" and
"Feature".  See the C file's header for every reading taken.

Nothing here imports or calls the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "topk_oracle.c")
LIBRARY = os.path.join(HERE, "liboracle.so")

FLAG_SEQ_CLAMPED = 1
FLAG_SEQ_NEGATIVE = 2

_lock = threading.Lock()
_libs: dict[str, ctypes.CDLL] = {}


def build(output: str = LIBRARY, defines: tuple[str, ...] = ()) -> str:
    """Compile the oracle with gcc (host only, no CUDA) and return the path."""
    os.makedirs(os.path.dirname(output), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", "-pthread", SOURCE, "-o", output, "-lm"]
    cmd[1:1] = [f"-D{d}" for d in defines]
    subprocess.run(cmd, check=True)
    return output


def load(path: str = LIBRARY) -> ctypes.CDLL:
    """Load (building first if needed) the oracle shared library."""
    with _lock:
        if path in _libs:
            return _libs[path]
        if path == LIBRARY and (
            not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(SOURCE)
        ):
            build(path)
        lib = ctypes.CDLL(path)
        i32, i64, p = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
        lib.oracle_topk_transform.argtypes = [p, i64, p, i32, i32, p, i64, i32, i32, p, p, i32, p]
        lib.oracle_topk_transform.restype = ctypes.c_int
        lib.oracle_page_transform.argtypes = [p, i32, i32, p, i64, i32, p]
        lib.oracle_page_transform.restype = ctypes.c_int
        lib.oracle_plan_classify.argtypes = [p, i32, i32, i32, p, p, p]
        lib.oracle_plan_classify.restype = ctypes.c_int
        _libs[path] = lib
        return lib


def _ptr(a: np.ndarray | None) -> int | None:
    return None if a is None else a.ctypes.data


def topk_transform(
    scores: np.ndarray,
    seq_lens: np.ndarray,
    page_table: np.ndarray,
    page_size: int,
    k: int,
    max_seq_len: int | None = None,
    want_raw: bool = True,
    nthreads: int = 1,
    lib_path: str = LIBRARY,
):
    """Return ``(out, raw_or_None, flags)`` for a ``[batch, row_stride]`` fp32 matrix.

    ``out``/``raw`` are ``[batch, k]`` int32 in sort order (best first), padded
    with -1.  ``max_seq_len`` defaults to the row stride.
    """
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    page_table = np.ascontiguousarray(page_table, dtype=np.int32)
    batch, row_stride = scores.shape
    if max_seq_len is None:
        max_seq_len = row_stride
    out = np.empty((batch, k), dtype=np.int32)
    raw = np.empty((batch, k), dtype=np.int32) if want_raw else None
    flags = ctypes.c_uint32(0)
    lib = load(lib_path)
    rc = lib.oracle_topk_transform(
        _ptr(scores), row_stride, _ptr(seq_lens), batch, max_seq_len, _ptr(page_table),
        page_table.shape[1], page_size, k, _ptr(out), _ptr(raw), nthreads, ctypes.byref(flags),
    )
    if rc != 0:
        raise ValueError(f"oracle_topk_transform failed with status {rc}")
    return out, raw, int(flags.value)


def page_transform(raw: np.ndarray, page_table: np.ndarray, page_size: int, lib_path: str = LIBRARY):
    """The transform alone: ``[batch, k]`` raw positions (or -1) to page indices."""
    raw = np.ascontiguousarray(raw, dtype=np.int32)
    page_table = np.ascontiguousarray(page_table, dtype=np.int32)
    batch, k = raw.shape
    out = np.empty_like(raw)
    rc = load(lib_path).oracle_page_transform(
        _ptr(raw), batch, k, _ptr(page_table), page_table.shape[1], page_size, _ptr(out)
    )
    if rc != 0:
        raise ValueError(f"oracle_page_transform failed with status {rc}")
    return out


def plan_classify(seq_lens: np.ndarray, max_seq_len: int, long_threshold: int, lib_path: str = LIBRARY):
    """Return ``(effective_len, is_long, flags)`` of the plan step's row split."""
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    batch = seq_lens.shape[0]
    eff = np.empty(batch, dtype=np.int32)
    is_long = np.empty(batch, dtype=np.int32)
    flags = ctypes.c_uint32(0)
    rc = load(lib_path).oracle_plan_classify(
        _ptr(seq_lens), batch, max_seq_len, long_threshold, _ptr(eff), _ptr(is_long), ctypes.byref(flags)
    )
    if rc != 0:
        raise ValueError(f"oracle_plan_classify failed with status {rc}")
    return eff, is_long.astype(bool), int(flags.value)
