"""The allocation-free entry point, topk_transform_noalloc, called through the C ABI.

It serves callers that cannot allocate device memory (a plugin or an
allocator-managed runtime that only receives its inputs and outputs): the
plan's work lists live in a fixed device array owned by the library.  This
test checks it against the workspace-based topk_plan + topk_transform on two
calls in a row with different inputs (the second call must not see the first
call's lists), bit-exact as sorted index sets, checks both calls against the
CPU oracle as well, and checks that a batch above the array's limit is
refused.  The file name makes pytest collect it last.
"""
from __future__ import annotations

import numpy as np
import pytest

from sparse_attention_indexer_uint32_gb300 import workloads

pytestmark = pytest.mark.gpu


def _sorted_valid(a: np.ndarray, n: np.ndarray) -> np.ndarray:
    slot = np.arange(a.shape[1])[None, :]
    return np.sort(np.where(slot < n[:, None], a.astype(np.int64), np.iinfo(np.int64).max), axis=1)


def _run_both(wl):
    import torch

    from sparse_attention_indexer_uint32_gb300 import _lib, api

    dev = torch.device("cuda", 0)
    scores = torch.from_numpy(wl.scores).to(dev)
    seq = torch.from_numpy(wl.seq_lens).to(dev)
    table = torch.from_numpy(wl.page_table).to(dev)
    ref_out, ref_raw, _ = api.topk_transform(scores, seq, table, wl.page_size, wl.k, max_seq_len=wl.max_seq_len,
                                             want_raw=True)
    out = torch.full((wl.batch, wl.k), -7, dtype=torch.int32, device=dev)
    raw = torch.full((wl.batch, wl.k), -7, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    status = _lib.library().topk_transform_noalloc(
        scores.data_ptr(), wl.row_stride, seq.data_ptr(), wl.batch, wl.max_seq_len, table.data_ptr(),
        wl.page_table.shape[1], wl.page_size, wl.k, out.data_ptr(), raw.data_ptr(), stream)
    assert status == _lib.TOPK_OK, _lib.topk_status_string(status)
    torch.cuda.synchronize()
    return ref_out.cpu().numpy(), ref_raw.cpu().numpy(), out.cpu().numpy(), raw.cpu().numpy()


def test_no_alloc_matches_workspace_entry_point_on_two_calls():
    cases = [
        # mixes long rows (cluster path) and short ones, ties and a ragged tail
        workloads.random_case(seed=71, batch=40, min_len=0, max_len=90001, k=700, page_size=64, dist="bf16"),
        # a different batch and k: the second call must not reuse the first call's lists
        workloads.random_case(seed=72, batch=9, min_len=100, max_len=40000, k=2048, page_size=16, dist="normal"),
    ]
    from tests.parity_util import compare

    for wl in cases:
        ref_out, ref_raw, out, raw = _run_both(wl)
        n = np.minimum(np.clip(wl.seq_lens, 0, wl.max_seq_len), wl.k)
        valid = np.arange(wl.k)[None, :] < n[:, None]
        assert (out[~valid] == -1).all() and (raw[~valid] == -1).all()
        assert (_sorted_valid(raw, n) == _sorted_valid(ref_raw, n)).all()
        assert (_sorted_valid(out, n) == _sorted_valid(ref_out, n)).all()
        compare(wl, out, raw)  # and against the CPU oracle, row by row


def test_no_alloc_on_the_segment_split_path():
    """With the segment-split path asked for, the library's own array also
    holds that path's row states and candidate buffers: a skewed batch and a
    second, different one in a row, both against the oracle."""
    from tests.parity_util import compare, tuning

    cases = [
        workloads.random_case(seed=73, batch=30, min_len=0, max_len=300000, k=1024, page_size=64, dist="bf16"),
        workloads.random_case(seed=74, batch=128, min_len=1, max_len=20000, k=2048, page_size=16, dist="int"),
    ]
    with tuning(split_rows=1):
        for wl in cases:
            _, _, out, raw = _run_both(wl)
            compare(wl, out, raw)


def test_no_alloc_refuses_a_batch_above_its_limit():
    import torch

    from sparse_attention_indexer_uint32_gb300 import _lib

    batch = _lib.TOPK_NOALLOC_MAX_BATCH + 1
    dev = torch.device("cuda", 0)
    scores = torch.zeros((batch, 4), dtype=torch.float32, device=dev)
    seq = torch.full((batch,), 4, dtype=torch.int32, device=dev)
    table = torch.zeros((batch, 1), dtype=torch.int32, device=dev)
    out = torch.full((batch, 1), -7, dtype=torch.int32, device=dev)
    status = _lib.library().topk_transform_noalloc(
        scores.data_ptr(), 4, seq.data_ptr(), batch, 4, table.data_ptr(), 1, 64, 1, out.data_ptr(), None, None)
    assert status == _lib.TOPK_ENOSPACE
    torch.cuda.synchronize()
    assert (out.cpu().numpy() == -7).all()
