"""Tensor-level conveniences over the C ABI (allocation and marshalling only)."""
from __future__ import annotations

import torch

from . import _lib


def plan(seq_lens: torch.Tensor, max_seq_len: int, workspace: torch.Tensor | None = None,
         stream=None) -> torch.Tensor:
    """Runs ``topk_plan`` and returns the (possibly newly allocated) workspace."""
    batch = seq_lens.shape[0]
    need = _lib.topk_plan_workspace_bytes(batch)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=seq_lens.device)
    _lib.topk_plan(seq_lens, batch, max_seq_len, workspace, stream)
    return workspace


def topk_transform(scores: torch.Tensor, seq_lens: torch.Tensor, page_table: torch.Tensor, page_size: int,
                   k: int, max_seq_len: int | None = None, want_raw: bool = False,
                   workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                   raw_out: torch.Tensor | None = None, stream=None):
    """Plans (unless a planned ``workspace`` is given) and runs the transform.

    ``scores``: float32 cuda [batch, row_stride] (row-contiguous); ``seq_lens``:
    int32 cuda [batch]; ``page_table``: int32 cuda [batch, pages].  Returns
    ``(out, raw_or_None, workspace)``.
    """
    batch, row_stride = scores.shape
    if max_seq_len is None:
        max_seq_len = row_stride
    if scores.stride(1) != 1 or page_table.stride(1) != 1:
        raise ValueError("scores and page_table rows must be contiguous")
    if workspace is None:
        workspace = plan(seq_lens, max_seq_len, stream=stream)
    if out is None:
        out = torch.empty((batch, k), dtype=torch.int32, device=scores.device)
    if want_raw and raw_out is None:
        raw_out = torch.empty((batch, k), dtype=torch.int32, device=scores.device)
    _lib.topk_transform(scores, scores.stride(0), seq_lens, batch, max_seq_len, page_table, page_table.stride(0),
                        page_size, k, out, raw_out if want_raw else None, workspace, stream)
    return out, (raw_out if want_raw else None), workspace
