"""ctypes binding of ``libtopkidx.so`` (include/topkidx.h), argument marshalling only.

Every function has the C name.  Tensors are passed as raw device pointers;
the stream defaults to PyTorch's current stream on the tensors' device.  A
non-OK status raises :class:`TopkError`.  There is no fallback: if the CUDA
library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(_PKG, "libtopkidx.so")

TOPK_OK = 0
TOPK_EINVAL = -1
TOPK_EALIGN = -2
TOPK_ECUDA = -3
TOPK_ENOSPACE = -4
TOPK_EDEVICE = -5

TOPK_FLAG_SEQ_CLAMPED = 0x1
TOPK_FLAG_SEQ_NEGATIVE = 0x2
TOPK_FLAG_PLAN_MISMATCH = 0x4
TOPK_FLAG_TIMEOUT = 0x8
TOPK_FLAG_INTERNAL = 0x10

TOPK_NOALLOC_MAX_BATCH = 16384

EXPORTED = (
    "topk_plan_workspace_bytes",
    "topk_plan",
    "topk_transform",
    "topk_transform_noalloc",
    "topk_transform_launches",
    "topk_page_transform",
    "topk_key_map",
    "topk_read_flags",
    "topk_status_string",
    "topk_last_error_string",
    "topk_get_tuning",
    "topk_set_tuning",
)


class TopkError(RuntimeError):
    def __init__(self, fn: str, status: int):
        detail = f"; {topk_last_error_string()}" if status == TOPK_ECUDA else ""
        super().__init__(f"{fn} failed: {status} ({topk_status_string(status)}){detail}")
        self.status = status


class topk_tuning_t(ctypes.Structure):  # noqa: N801 - C name
    _fields_ = [
        ("long_threshold_small_batch", ctypes.c_int32),
        ("long_threshold", ctypes.c_int32),
        ("small_batch_max", ctypes.c_int32),
        ("cluster_size", ctypes.c_int32),
        ("force_two_pass", ctypes.c_int32),
        ("disable_gate", ctypes.c_int32),
        ("candidate_capacity", ctypes.c_int32),
        ("samples", ctypes.c_int32),
        ("gate_fill_percent", ctypes.c_int32),
        ("single_block_threads", ctypes.c_int32),
        ("single_block_copy_bytes", ctypes.c_int32),
        ("single_block_stages", ctypes.c_int32),
        ("gate_refresh_tiles", ctypes.c_int32),
        ("warp_rows", ctypes.c_int32),
        ("wait_limit_us", ctypes.c_int32),
        ("single_block_kernel", ctypes.c_int32),
        ("long_threshold_large_batch", ctypes.c_int32),
        ("large_batch_min", ctypes.c_int32),
        ("warp_batch_min", ctypes.c_int32),
        ("stream_batch_min", ctypes.c_int32),
        ("split_rows", ctypes.c_int32),
        ("split_segment", ctypes.c_int32),
        ("split_full_resolve", ctypes.c_int32),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIBRARY):
        raise ImportError(
            f"{LIBRARY} is missing: build it with `python -m sparse_attention_indexer_uint32_gb300.build` "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIBRARY)
    i32, i64, p, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    lib.topk_plan_workspace_bytes.argtypes = [i32]
    lib.topk_plan_workspace_bytes.restype = sz
    lib.topk_plan.argtypes = [p, i32, i32, p, sz, p]
    lib.topk_plan.restype = ctypes.c_int
    lib.topk_transform.argtypes = [p, i64, p, i32, i32, p, i64, i32, i32, p, p, p, p]
    lib.topk_transform.restype = ctypes.c_int
    lib.topk_transform_noalloc.argtypes = [p, i64, p, i32, i32, p, i64, i32, i32, p, p, p]
    lib.topk_transform_noalloc.restype = ctypes.c_int
    lib.topk_transform_launches.argtypes = [i32, i32, i32]
    lib.topk_transform_launches.restype = i32
    lib.topk_page_transform.argtypes = [p, i32, i32, p, i64, i32, p, p]
    lib.topk_page_transform.restype = ctypes.c_int
    lib.topk_key_map.argtypes = [p, i64, p, p]
    lib.topk_key_map.restype = ctypes.c_int
    lib.topk_read_flags.argtypes = [p, ctypes.POINTER(ctypes.c_uint32), i32, p]
    lib.topk_read_flags.restype = ctypes.c_int
    lib.topk_status_string.argtypes = [ctypes.c_int]
    lib.topk_status_string.restype = ctypes.c_char_p
    lib.topk_last_error_string.argtypes = []
    lib.topk_last_error_string.restype = ctypes.c_char_p
    lib.topk_get_tuning.argtypes = [ctypes.POINTER(topk_tuning_t)]
    lib.topk_get_tuning.restype = ctypes.c_int
    lib.topk_set_tuning.argtypes = [ctypes.POINTER(topk_tuning_t)]
    lib.topk_set_tuning.restype = ctypes.c_int
    return lib


_lib = _load()


def library() -> ctypes.CDLL:
    return _lib


def _check(fn: str, status: int) -> None:
    if status == TOPK_OK:
        return
    err = TopkError(fn, status)
    if status == TOPK_ECUDA:
        # Surface the CUDA runtime's own message (for example a fault left by
        # an earlier asynchronous launch) next to the library status.
        try:
            torch.cuda.synchronize()
        except Exception as e:  # noqa: BLE001
            raise err from e
    raise err


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(getattr(stream, "cuda_stream", stream) or 0)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def topk_status_string(status: int) -> str:
    return _lib.topk_status_string(status).decode()


def topk_last_error_string() -> str:
    return _lib.topk_last_error_string().decode()


def topk_plan_workspace_bytes(batch: int) -> int:
    return int(_lib.topk_plan_workspace_bytes(batch))


def topk_plan(seq_lens: torch.Tensor, batch: int, max_seq_len: int, workspace: torch.Tensor, stream=None) -> None:
    """Plan step on ``seq_lens`` (int32 cuda[batch]) into ``workspace`` (uint8 cuda)."""
    _check("topk_plan", _lib.topk_plan(_ptr(seq_lens), batch, max_seq_len, _ptr(workspace),
                                       workspace.numel() * workspace.element_size(),
                                       _stream(stream, seq_lens.device)))


def topk_transform(scores: torch.Tensor, row_stride: int, seq_lens: torch.Tensor, batch: int, max_seq_len: int,
                   page_table: torch.Tensor, page_table_stride: int, page_size: int, k: int,
                   out_indices: torch.Tensor, out_raw_indices_or_null: torch.Tensor | None,
                   workspace: torch.Tensor, stream=None) -> None:
    """Top-k + page-table transform into ``out_indices`` (and the raw positions)."""
    _check("topk_transform", _lib.topk_transform(
        _ptr(scores), row_stride, _ptr(seq_lens), batch, max_seq_len, _ptr(page_table), page_table_stride,
        page_size, k, _ptr(out_indices), _ptr(out_raw_indices_or_null), _ptr(workspace),
        _stream(stream, scores.device)))


def topk_transform_noalloc(scores: torch.Tensor, row_stride: int, seq_lens: torch.Tensor, batch: int,
                           max_seq_len: int, page_table: torch.Tensor, page_table_stride: int, page_size: int,
                           k: int, out_indices: torch.Tensor, out_raw_indices_or_null: torch.Tensor | None,
                           stream=None) -> None:
    """Plan + transform without a caller workspace (batch <= TOPK_NOALLOC_MAX_BATCH)."""
    _check("topk_transform_noalloc", _lib.topk_transform_noalloc(
        _ptr(scores), row_stride, _ptr(seq_lens), batch, max_seq_len, _ptr(page_table), page_table_stride,
        page_size, k, _ptr(out_indices), _ptr(out_raw_indices_or_null), _stream(stream, scores.device)))


def topk_transform_launches(batch: int, max_seq_len: int, k: int) -> int:
    """Kernels one topk_transform call with these arguments enqueues (1 or 2)."""
    n = _lib.topk_transform_launches(batch, max_seq_len, k)
    if n < 0:
        raise TopkError("topk_transform_launches", n)
    return int(n)


def topk_page_transform(raw_indices: torch.Tensor, batch: int, k: int, page_table: torch.Tensor,
                        page_table_stride: int, page_size: int, out_indices: torch.Tensor, stream=None) -> None:
    _check("topk_page_transform", _lib.topk_page_transform(
        _ptr(raw_indices), batch, k, _ptr(page_table), page_table_stride, page_size, _ptr(out_indices),
        _stream(stream, raw_indices.device)))


def topk_key_map(x: torch.Tensor, n: int, keys: torch.Tensor, stream=None) -> None:
    _check("topk_key_map", _lib.topk_key_map(_ptr(x), n, _ptr(keys), _stream(stream, x.device)))


def topk_read_flags(workspace: torch.Tensor, clear: bool = False, stream=None) -> int:
    flags = ctypes.c_uint32(0)
    _check("topk_read_flags", _lib.topk_read_flags(_ptr(workspace), ctypes.byref(flags), int(clear),
                                                   _stream(stream, workspace.device)))
    return int(flags.value)


def topk_get_tuning() -> topk_tuning_t:
    t = topk_tuning_t()
    _check("topk_get_tuning", _lib.topk_get_tuning(ctypes.byref(t)))
    return t


def topk_set_tuning(t: topk_tuning_t) -> None:
    _check("topk_set_tuning", _lib.topk_set_tuning(ctypes.byref(t)))
