"""GPU checks of the single steps exposed at the C ABI: the key map, the
stand-alone page transform and the plan, plus argument errors."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from sparse_attention_indexer_uint32_gb300 import workloads

pytestmark = pytest.mark.gpu


def _lib():
    from sparse_attention_indexer_uint32_gb300 import _lib

    return _lib


def test_key_map_orders_every_float():
    """Walk every non-NaN fp32 in increasing IEEE order: the keys must increase
    strictly, except that -0.0 and +0.0 share a key; NaNs sit outside."""
    import torch

    lib = _lib()
    dev = torch.device("cuda", 0)
    chunk = 1 << 26
    # increasing order: -inf (0xFF800000) down the bit patterns to -0.0
    # (0x80000000), then +0.0 (0x00000000) up to +inf (0x7F800000)
    segments = [(0xFF800000, 0x80000000, -1), (0x00000000, 0x7F800000, +1)]
    last_key = None
    for seg, (start, stop, step) in enumerate(segments):
        count = abs(stop - start) + 1
        for off in range(0, count, chunk):
            n = min(chunk, count - off)
            bits = start + step * (off + torch.arange(n, device=dev, dtype=torch.int64))
            b32 = torch.where(bits >= 2 ** 31, bits - 2 ** 32, bits).to(torch.int32)
            keys = torch.empty(n, dtype=torch.int32, device=dev)
            lib.topk_key_map(b32.view(torch.float32), n, keys)
            k64 = keys.to(torch.int64).bitwise_and(0xFFFFFFFF)
            assert bool((k64[1:] > k64[:-1]).all()), f"keys not increasing near bits {start + step * off:#x}"
            first = int(k64[0])
            if last_key is not None:
                if seg == 1 and off == 0:
                    assert first == last_key, "-0.0 and +0.0 must share a key"
                else:
                    assert first > last_key
            last_key = int(k64[-1])
    nan_bits = np.array([0x7FC00000, 0x7F800001, 0xFFC00000, 0xFF800001], dtype=np.uint32)
    x = torch.from_numpy(nan_bits.view(np.float32)).to(dev)
    inf = torch.tensor([np.inf, -np.inf], dtype=torch.float32, device=dev)
    k_nan = torch.empty(4, dtype=torch.int32, device=dev)
    k_inf = torch.empty(2, dtype=torch.int32, device=dev)
    lib.topk_key_map(x, 4, k_nan)
    lib.topk_key_map(inf, 2, k_inf)
    kn = k_nan.cpu().numpy().view(np.uint32).astype(np.int64)
    ki = k_inf.cpu().numpy().view(np.uint32).astype(np.int64)
    assert kn[0] > ki[0] and kn[1] > ki[0] and kn[0] > kn[1]  # +NaN above +inf, larger payload higher
    assert kn[2] < ki[1] and kn[3] < ki[1] and kn[2] < kn[3]  # -NaN below -inf, larger payload lower


def test_page_transform_standalone_matches_oracle():
    import torch

    lib = _lib()
    rng = np.random.default_rng(0)
    for P in (1, 64, 128):
        B, k, NP = 33, 517, 300
        table = rng.permutation(B * NP).astype(np.int32).reshape(B, NP)
        raw = rng.integers(-1, NP * P, size=(B, k)).astype(np.int32)
        raw[:, -5:] = -1
        expect = oracle.page_transform(raw, table, P)
        dev = torch.device("cuda", 0)
        raw_d = torch.from_numpy(raw).to(dev)
        table_d = torch.from_numpy(table).to(dev)
        out = torch.empty_like(raw_d)
        lib.topk_page_transform(raw_d, B, k, table_d, NP, P, out)
        assert (out.cpu().numpy() == expect).all()


def test_plan_lists_match_oracle_classification():
    import torch

    lib = _lib()
    rng = np.random.default_rng(1)
    cases = [(5, 1 << 20, None), (200, 300000, None), (3000, 70000, None), (8192, 8192, None),
             # every row in one (class, bucket): the plan writes no lists and sets the identity flag
             (8192, 8192, 8192), (3, 1 << 20, 1 << 20), (16384, 70000, 65000), (16385, 8192, 8192)]
    for batch, max_len, same in cases:
        lens = rng.integers(-5, max_len + 1000, size=batch).astype(np.int32)
        if same is not None:
            lens[:] = same
        dev = torch.device("cuda", 0)
        seq = torch.from_numpy(lens).to(dev)
        nbytes = lib.topk_plan_workspace_bytes(batch)
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        lib.topk_plan(seq, batch, max_len, ws)
        torch.cuda.synchronize()
        host = ws.cpu().numpy()
        hdr = host[:64].view(np.int32)
        t = lib.topk_get_tuning()
        thr = (t.long_threshold_small_batch if batch <= t.small_batch_max
               else t.long_threshold if batch <= t.large_batch_min else t.long_threshold_large_batch)
        eff, is_long, flags = oracle.plan_classify(lens, max_len, thr)
        n_long, n_short = int(hdr[4]), int(hdr[5])
        lists = host[64:64 + 8 * batch].view(np.int32)
        long_rows, short_rows = lists[:n_long], lists[batch:batch + n_short]
        # identity: one sweep (batch <= 16384) with a single (class, bucket)
        assert int(hdr[7]) == int(same is not None and batch <= 16384)
        if int(hdr[7]):
            assert (lists == 0).all()  # nothing written
            long_rows, short_rows = np.arange(n_long), np.arange(n_short)
        assert sorted(long_rows.tolist()) == np.nonzero(is_long)[0].tolist()
        assert sorted(short_rows.tolist()) == np.nonzero(~is_long)[0].tolist()
        assert int(hdr[6]) == flags
        # longest first (by half-octave bucket)
        for rows in (long_rows, short_rows):
            L = eff[rows].astype(np.int64)
            bl = np.where(L > 0, np.floor(np.log2(np.maximum(L, 1))).astype(np.int64) + 1, 0)
            bucket = np.where(bl >= 2, 2 * bl + ((L >> np.maximum(bl - 2, 0)) & 1), 2 * bl)
            assert (np.diff(bucket) <= 0).all()


def test_argument_errors_raise():
    import torch

    lib = _lib()
    dev = torch.device("cuda", 0)
    scores = torch.zeros((2, 64), dtype=torch.float32, device=dev)
    seq = torch.full((2,), 64, dtype=torch.int32, device=dev)
    table = torch.zeros((2, 1), dtype=torch.int32, device=dev)
    out = torch.empty((2, 8), dtype=torch.int32, device=dev)
    ws = torch.zeros(lib.topk_plan_workspace_bytes(2), dtype=torch.uint8, device=dev)
    lib.topk_plan(seq, 2, 64, ws)
    cases = [
        dict(k=0), dict(k=2049), dict(page_size=3), dict(row_stride=62), dict(page_table_stride=0),
        dict(max_seq_len=128),
    ]
    for over in cases:
        args = dict(scores=scores, row_stride=64, seq_lens=seq, batch=2, max_seq_len=64, page_table=table,
                    page_table_stride=1, page_size=64, k=8, out_indices=out, out_raw_indices_or_null=None,
                    workspace=ws)
        args.update(over)
        with pytest.raises(lib.TopkError) as e:
            lib.topk_transform(**args)
        assert e.value.status in (lib.TOPK_EINVAL, lib.TOPK_EALIGN)
    with pytest.raises(lib.TopkError):
        lib.topk_transform(scores.view(-1)[1:], 64, seq, 2, 60, table, 1, 64, 8, out, None, ws)  # misaligned


def test_plan_mismatch_is_flagged_and_nothing_written():
    import torch

    lib = _lib()
    dev = torch.device("cuda", 0)
    wl = workloads.random_case(seed=1, batch=4, min_len=100, max_len=1000, k=16, page_size=4)
    scores = torch.from_numpy(wl.scores).to(dev)
    seq = torch.from_numpy(wl.seq_lens).to(dev)
    table = torch.from_numpy(wl.page_table).to(dev)
    ws = torch.zeros(lib.topk_plan_workspace_bytes(4), dtype=torch.uint8, device=dev)
    lib.topk_plan(seq, 4, wl.max_seq_len - 4, ws)  # planned for another max_seq_len
    out = torch.full((4, 16), -7, dtype=torch.int32, device=dev)
    lib.topk_transform(scores, wl.row_stride, seq, 4, wl.max_seq_len, table, wl.page_table.shape[1], 4, 16, out,
                       None, ws)
    torch.cuda.synchronize()
    assert lib.topk_read_flags(ws) & lib.TOPK_FLAG_PLAN_MISMATCH
    assert (out.cpu().numpy() == -7).all()


def test_launch_count_query_matches_the_dispatch():
    lib = _lib()
    t = lib.topk_get_tuning()
    assert t.cluster_size == 0  # automatic
    # short rows only: one single-block launch
    assert lib.topk_transform_launches(8192, 8192, 512) == 1
    assert lib.topk_transform_launches(2048, 65536, 512) == 1
    # long rows of a small batch: the cluster kernel takes every row
    assert lib.topk_transform_launches(1, 1 << 20, 2048) == 1
    assert lib.topk_transform_launches(32, 1 << 20, 2048) == 1
    assert lib.topk_transform_launches(128, 262144, 1024) == 1
    # a large batch with long rows: single-block kernel for short rows, then the cluster kernel
    assert lib.topk_transform_launches(4096, 262144, 512) == 2


@pytest.mark.parametrize("path", ["single_block", "stream", "cluster"])
def test_bounded_wait_gives_up_and_the_next_call_is_correct(path):
    """A wait limit of 1 us is shorter than a bulk copy of scores takes, so the
    select blocks give up waiting: the call must return, the flag word must
    carry TOPK_FLAG_TIMEOUT, and a following call with the default limit (on
    the same buffers, the same stream) must give the exact answer again.  The
    expiry is the kernel's own bounded wait running out; nothing faults."""
    import torch

    from tests.parity_util import compare, run_gpu, tuning

    lib = _lib()
    if path == "cluster":
        wl = workloads.random_case(seed=801, batch=160, min_len=150000, max_len=262144, k=512, page_size=64,
                                   dist="normal")
        thr, extra = 0, dict(cluster_size=4)
    else:
        wl = workloads.random_case(seed=800, batch=1200, min_len=40000, max_len=65536, k=512, page_size=64,
                                   dist="normal")
        thr, extra = 1 << 30, dict(single_block_kernel=2 if path == "stream" else 1)
    # A wait runs out only when a copy takes longer than the limit after the
    # first probe, which a memory-bound launch of this size shows many times;
    # a few attempts keep the test independent of one launch's timing.
    seen = 0
    for _ in range(4):
        with tuning(wait_limit_us=1, long_threshold=thr, long_threshold_small_batch=thr, **extra):
            _, _, flags = run_gpu(wl)
        seen |= flags
        if flags & lib.TOPK_FLAG_TIMEOUT:
            break
    assert seen & lib.TOPK_FLAG_TIMEOUT, f"no wait gave up (flags {seen:#x})"
    torch.cuda.synchronize()
    with tuning(long_threshold=thr, long_threshold_small_batch=thr, **extra):
        out, raw, flags = run_gpu(wl)
    assert flags == 0
    compare(wl, out, raw)


def test_dependent_consumer_chained_after_the_transform():
    """plan -> transform -> a consumer kernel on one stream with no host sync:
    the consumer (the stand-alone page transform, launched with programmatic
    stream serialization) may be placed as soon as every select block has
    written its output and triggered, and waits for the select grid before it
    reads raw_out.  raw_out is poisoned with -7 before every step, so a
    consumer that read early would map -7 to -1 and fail the comparison."""
    import torch

    from sparse_attention_indexer_uint32_gb300 import api
    from tests.parity_util import compare

    lib = _lib()
    dev = torch.device("cuda", 0)
    rng = np.random.default_rng(5)
    for dist, k in (("normal", 512), ("bf16", 2048)):
        wl = workloads.random_case(seed=810 + k, batch=300, min_len=0, max_len=70001, k=k, page_size=64, dist=dist)
        scores = torch.from_numpy(wl.scores).to(dev)
        seq = torch.from_numpy(wl.seq_lens).to(dev)
        table = torch.from_numpy(wl.page_table).to(dev)
        pages = wl.page_table.shape[1]
        table2_h = rng.permutation(wl.batch * pages).astype(np.int32).reshape(wl.batch, pages)
        table2 = torch.from_numpy(table2_h).to(dev)
        out = torch.empty((wl.batch, wl.k), dtype=torch.int32, device=dev)
        raw = torch.empty_like(out)
        out2 = torch.empty_like(out)
        ws = torch.zeros(lib.topk_plan_workspace_bytes(wl.batch), dtype=torch.uint8, device=dev)
        for _ in range(3):
            raw.fill_(-7)
            out2.fill_(-9)
            api.plan(seq, wl.max_seq_len, ws)
            lib.topk_transform(scores, wl.row_stride, seq, wl.batch, wl.max_seq_len, table, pages, wl.page_size,
                               wl.k, out, raw, ws)
            lib.topk_page_transform(raw, wl.batch, wl.k, table2, pages, wl.page_size, out2)
            torch.cuda.synchronize()
            g_raw, g_out2 = raw.cpu().numpy(), out2.cpu().numpy()
            compare(wl, out.cpu().numpy(), g_raw)  # the select's own output against the oracle
            assert (g_out2 == oracle.page_transform(g_raw, table2_h, wl.page_size)).all()
            o_out2, _, _ = oracle.topk_transform(wl.scores, wl.seq_lens, table2_h, wl.page_size, wl.k)
            valid = np.arange(wl.k)[None, :] < np.minimum(np.clip(wl.seq_lens, 0, wl.max_seq_len), wl.k)[:, None]
            big = np.iinfo(np.int64).max
            srt = lambda a: np.sort(np.where(valid, a.astype(np.int64), big), axis=1)  # noqa: E731
            assert (srt(g_out2) == srt(o_out2)).all() and (g_out2[~valid] == -1).all()
