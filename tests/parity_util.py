"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and compare it with the CPU oracle row by row (as sorted index sets)."""
from __future__ import annotations

import contextlib
import os

import numpy as np

import oracle

NTHREADS = max(1, min(16, os.cpu_count() or 1))


def to_device(wl):
    import torch

    dev = torch.device("cuda", 0)
    return (torch.from_numpy(wl.scores).to(dev), torch.from_numpy(wl.seq_lens).to(dev),
            torch.from_numpy(wl.page_table).to(dev))


def run_gpu(wl, want_raw=True):
    """Plan + transform on cuda:0; returns host (out, raw, flags)."""
    import torch

    from sparse_attention_indexer_uint32_gb300 import _lib, api

    scores, seq_lens, table = to_device(wl)
    out, raw, ws = api.topk_transform(scores, seq_lens, table, wl.page_size, wl.k, max_seq_len=wl.max_seq_len,
                                      want_raw=want_raw)
    torch.cuda.synchronize()
    flags = _lib.topk_read_flags(ws)
    return out.cpu().numpy(), (raw.cpu().numpy() if raw is not None else None), flags


def compare(wl, out, raw, rows=None, check_raw=True):
    """Asserts that the GPU rows equal the oracle's as sorted sets, that the
    padding is -1, and that out is the page transform of raw slot by slot."""
    rows = np.arange(wl.batch) if rows is None else np.asarray(rows)
    o_out, o_raw, _ = oracle.topk_transform(wl.scores[rows], wl.seq_lens[rows], wl.page_table[rows], wl.page_size,
                                            wl.k, max_seq_len=wl.max_seq_len, want_raw=True, nthreads=NTHREADS)
    eff = np.clip(wl.seq_lens[rows].astype(np.int64), 0, wl.max_seq_len)
    n = np.minimum(eff, wl.k)
    slot = np.arange(wl.k)[None, :]
    valid = slot < n[:, None]
    g_out = out[rows]
    assert (g_out[~valid] == -1).all(), "out padding is not -1"
    big = np.iinfo(np.int64).max
    srt = lambda a: np.sort(np.where(valid, a.astype(np.int64), big), axis=1)  # noqa: E731
    bad = np.nonzero((srt(g_out) != srt(o_out)).any(axis=1))[0]
    if check_raw and raw is not None:
        g_raw = raw[rows]
        assert (g_raw[~valid] == -1).all(), "raw padding is not -1"
        bad_raw = np.nonzero((srt(g_raw) != srt(o_raw)).any(axis=1))[0]
        assert len(bad_raw) == 0, f"raw set differs from the oracle in rows {rows[bad_raw][:10].tolist()}"
        again = oracle.page_transform(g_raw, wl.page_table[rows], wl.page_size)
        assert (again == g_out).all(), "out is not the page transform of raw slot by slot"
    assert len(bad) == 0, f"out set differs from the oracle in rows {rows[bad][:10].tolist()}"


@contextlib.contextmanager
def tuning(**overrides):
    """Temporarily overrides dispatch knobs of the CUDA library."""
    from sparse_attention_indexer_uint32_gb300 import _lib

    old = _lib.topk_get_tuning()
    new = _lib.topk_tuning_t(**old.as_dict())
    if "long_threshold" in overrides and "long_threshold_large_batch" not in overrides:
        # one threshold for every batch above the small-batch tier
        overrides = {**overrides, "long_threshold_large_batch": overrides["long_threshold"]}
    for k, v in overrides.items():
        setattr(new, k, v)
    _lib.topk_set_tuning(new)
    try:
        yield
    finally:
        _lib.topk_set_tuning(old)


def check_properties_all_rows(wl, raw):
    """Checks every row of a full-size run against properties that fix the
    answer without running the oracle on all rows: min(k, L) distinct
    in-range positions; every selected score >= every unselected one
    (IEEE comparison, so -0 == +0); and where the k-th score is tied, the
    selected copies are the smallest positions of that score.  Vectorised
    over rows; for workloads whose rows have no NaN."""
    B, S = wl.scores.shape
    eff = np.clip(wl.seq_lens.astype(np.int64), 0, wl.max_seq_len)
    n = np.minimum(eff, wl.k)
    slot = np.arange(wl.k)[None, :]
    valid = slot < n[:, None]
    assert (raw[~valid] == -1).all(), "raw padding is not -1"
    r = raw.astype(np.int64)
    assert ((r >= 0) & (r < eff[:, None]))[valid].all(), "a selected position is outside its row"
    mask = np.zeros((B, S), dtype=bool)
    bi = np.broadcast_to(np.arange(B)[:, None], r.shape)[valid]
    mask[bi, r[valid]] = True
    assert (mask.sum(axis=1) == n).all(), "selected positions repeat within a row"
    in_row = np.arange(S)[None, :] < eff[:, None]
    x = wl.scores
    sel_min = np.where(mask, x, np.inf).min(axis=1)
    uns = in_row & ~mask
    uns_max = np.where(uns, x, -np.inf).max(axis=1)
    has_uns = uns.any(axis=1) & (n > 0)
    assert (sel_min[has_uns] >= uns_max[has_uns]).all(), "an unselected score beats a selected one"
    tie = has_uns & (sel_min == uns_max)
    if tie.any():
        pos = np.arange(S)[None, :]
        t = sel_min[tie][:, None]
        xt = x[tie]
        last_sel = np.where(mask[tie] & (xt == t), pos, -1).max(axis=1)
        first_uns = np.where(uns[tie] & (xt == t), pos, S).min(axis=1)
        assert (last_sel < first_uns).all(), "tied copies of the k-th score not taken smallest position first"
