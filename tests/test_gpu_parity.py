"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bit-exact comparison of the selected index sets (raw and transformed), the -1
padding and slot alignment, on seeded inputs: the five benchmark workloads at
their full sizes and small ragged cases that span several tiles, every
dispatch path and the degenerate inputs.  Every row of every case is
compared.
"""
from __future__ import annotations

import numpy as np
import pytest

from sparse_attention_indexer_uint32_gb300 import workloads
from tests.parity_util import check_properties_all_rows, compare, run_gpu, tuning

pytestmark = pytest.mark.gpu


# ----------------------------------------------------------- the five workloads
# Every row of every workload is compared with the oracle (raw and
# transformed, as sorted sets, with the -1 padding and the slot alignment);
# the property check runs on every row as a second, oracle-free check.
def test_tiny_workload():
    wl = workloads.tiny()
    out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


def test_decode_workload_all_rows():
    wl = workloads.decode()
    out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    check_properties_all_rows(wl, raw)
    assert flags == 0


def test_throughput_workload_all_rows():
    wl = workloads.throughput()
    out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    check_properties_all_rows(wl, raw)
    assert flags == 0


@pytest.mark.parametrize("batch", [1, 8, 32])
def test_long_context_workload_all_rows(batch):
    wl = workloads.long_context(batch)
    out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    check_properties_all_rows(wl, raw)
    assert flags == 0


def test_ragged_workload_all_rows():
    wl = workloads.ragged()
    out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


def test_golden_cases_on_the_gpu():
    """The hand-worked cases (tests/golden/hand_worked.txt: ties, signed
    zeros, -inf, NaN payload order, short and empty rows, clamped and negative
    seq_lens, the 32-bit wrap of the transform) through the CUDA path, checked
    against their hand-worked answers, not against the oracle."""
    from tests.golden_cases import load_cases

    for case in load_cases():
        L = len(case.scores)
        stride = max(4, -(-L // 4) * 4)
        scores = np.full((1, stride), np.inf, np.float32)
        scores[0, :L] = case.scores
        wl = workloads.Workload(case.name, scores, np.array([case.seq_len], np.int32), case.table[None, :].copy(),
                                case.page_size, case.k, case.max_seq_len, True)
        out, raw, _ = run_gpu(wl)
        n = case.k - case.pad
        assert sorted(raw[0, :n].tolist()) == case.raw, case.name
        assert sorted(out[0, :n].tolist()) == sorted(case.out), case.name
        assert (raw[0, n:] == -1).all() and (out[0, n:] == -1).all(), case.name


# ------------------------------------------------------------ small ragged cases
DISTS = ["normal", "bf16", "int", "flat", "neginf"]


@pytest.mark.parametrize("dist", DISTS)
@pytest.mark.parametrize("k", [1, 37, 512, 2048])
def test_random_ragged_single_block(dist, k):
    wl = workloads.random_case(seed=DISTS.index(dist) * 10000 + k, batch=40, min_len=0, max_len=20011, k=k,
                               page_size=64, dist=dist)
    out, raw, _ = run_gpu(wl)
    compare(wl, out, raw)


@pytest.mark.parametrize("batch", [3, 40])  # few rows: 512-thread blocks, 32 KB copies; many: 256, 16 KB
@pytest.mark.parametrize("cluster", [2, 3, 4, 8, 16])
@pytest.mark.parametrize("dist", ["normal", "bf16", "flat", "neginf"])
def test_cluster_path_forced(cluster, dist, batch):
    wl = workloads.random_case(seed=100 + cluster + batch, batch=batch, min_len=1, max_len=70001, k=700,
                               page_size=16, dist=dist)
    with tuning(long_threshold=0, long_threshold_small_batch=0, cluster_size=cluster, split_rows=2):
        out, raw, _ = run_gpu(wl)
    compare(wl, out, raw)


@pytest.mark.parametrize("cluster", [1, 8])
@pytest.mark.parametrize("dist", ["normal", "int", "flat"])
def test_two_pass_streaming_forced(cluster, dist):
    wl = workloads.random_case(seed=200 + cluster, batch=10, min_len=3000, max_len=90000, k=300, page_size=32,
                               dist=dist)
    thr = 0 if cluster > 1 else 1 << 30
    with tuning(force_two_pass=1, long_threshold=thr, long_threshold_small_batch=thr, split_rows=2):
        out, raw, _ = run_gpu(wl)
    compare(wl, out, raw)


@pytest.mark.parametrize("cluster", [1, 8])
@pytest.mark.parametrize("dist", ["normal", "bf16"])
def test_ungated_first_pass(cluster, dist):
    wl = workloads.random_case(seed=300 + cluster, batch=9, min_len=1000, max_len=60000, k=1024, page_size=8,
                               dist=dist)
    thr = 0 if cluster > 1 else 1 << 30
    with tuning(disable_gate=1, long_threshold=thr, long_threshold_small_batch=thr, split_rows=2):
        out, raw, _ = run_gpu(wl)
    compare(wl, out, raw)


@pytest.mark.parametrize("samples", [32, 64])
def test_few_samples_gate_misses(samples):
    """With very few samples the gate is often too tight or too loose; the
    fallbacks must still give the exact answer."""
    wl = workloads.random_case(seed=400 + samples, batch=16, min_len=5000, max_len=40000, k=2048, page_size=64,
                               dist="normal")
    for split_rows in (2, 1):  # the cluster kernel, then the segment-split path
        with tuning(samples=samples, split_rows=split_rows):
            out, raw, flags = run_gpu(wl)
        compare(wl, out, raw)
        assert flags == 0


@pytest.mark.parametrize("fill", [1, 100])
@pytest.mark.parametrize("cluster", [1, 8])
def test_gate_fill_extremes(fill, cluster):
    """fill = 1: the gate sits at its sampling bound, so some rows pass fewer
    than k elements and are recounted; fill = 100: the gate aims at the whole
    candidate buffer, so many rows overflow it and re-read their scores."""
    wl = workloads.random_case(seed=450 + fill + cluster, batch=24, min_len=3000, max_len=200000, k=512,
                               page_size=64, dist="bf16")
    thr = 0 if cluster > 1 else 1 << 30
    with tuning(gate_fill_percent=fill, long_threshold=thr, long_threshold_small_batch=thr, split_rows=2):
        out, raw, _ = run_gpu(wl)
    compare(wl, out, raw)


@pytest.mark.parametrize("dist", ["normal", "bf16"])
def test_single_block_512_threads(dist):
    """The 512-thread single-block kernel on rows over 16K (ragged tail,
    short rows and ties included)."""
    wl = workloads.random_case(seed=470, batch=40, min_len=0, max_len=150001, k=1000, page_size=32, dist=dist)
    with tuning(single_block_threads=512, long_threshold=1 << 30, long_threshold_small_batch=1 << 30):
        out, raw, _ = run_gpu(wl)
    compare(wl, out, raw)


@pytest.mark.parametrize("copy_bytes,stages", [(8192, 2), (8192, 5), (16384, 4), (24576, 3)])
def test_single_block_copy_shapes(copy_bytes, stages):
    """Other bulk-copy sizes and ring depths of the single-block kernel (the
    8 KB copy is the 2-float4-per-thread tile loop): rows shorter and longer
    than one ring, a ragged tail, ties."""
    wl = workloads.random_case(seed=490 + copy_bytes // 4096 + stages, batch=30, min_len=0, max_len=70001, k=512,
                               page_size=64, dist="bf16")
    with tuning(single_block_copy_bytes=copy_bytes, single_block_stages=stages, long_threshold=1 << 30,
                long_threshold_small_batch=1 << 30):
        out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


@pytest.mark.parametrize("refresh", [1, 2, 5])
@pytest.mark.parametrize("dist", ["normal", "bf16", "int", "flat", "neginf"])
def test_gate_refresh(refresh, dist):
    """The monotone gate refresh of the single-block kernel: the gate rises
    during a row from its own counts; no top-k element may be lost (ragged
    rows over several copies, ties, -inf rows, flat rows)."""
    wl = workloads.random_case(seed=520 + refresh * 10 + DISTS.index(dist), batch=24, min_len=0, max_len=140001,
                               k=700, page_size=16, dist=dist)
    with tuning(gate_refresh_tiles=refresh, long_threshold=1 << 30, long_threshold_small_batch=1 << 30):
        out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


@pytest.mark.parametrize("mode", ["ungated", "two_pass", "small_copies"])
def test_gate_refresh_modes(mode):
    """The refresh from an open gate (every element counted until the counts
    allow a gate: an online gate with no samples), with the histogram-only
    first pass, and with 8 KB copies (many refreshes per row)."""
    extra = {"ungated": dict(disable_gate=1), "two_pass": dict(force_two_pass=1),
             "small_copies": dict(single_block_copy_bytes=8192)}[mode]
    wl = workloads.random_case(seed=540 + len(mode), batch=16, min_len=2000, max_len=100001, k=512, page_size=64,
                               dist="normal")
    with tuning(gate_refresh_tiles=2, long_threshold=1 << 30, long_threshold_small_batch=1 << 30, **extra):
        out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


def test_trend_rows_cluster():
    """Rows with a positional trend (the gate's sample must not alias)."""
    wl = workloads.long_context(batch=2, seq_len=300000)
    for split_rows in (2, 1):  # the cluster kernel, then the segment-split path
        with tuning(long_threshold=0, long_threshold_small_batch=0, split_rows=split_rows):
            out, raw, _ = run_gpu(wl)
        compare(wl, out, raw)


# ------------------------------------------------------------------ edge cases
def _make(scores, lens, k, page_size=1, max_seq_len=None, table=None):
    scores = np.ascontiguousarray(scores, np.float32)
    B, S = scores.shape
    max_seq_len = S if max_seq_len is None else max_seq_len
    pages = workloads.pages_for(S, page_size)
    if table is None:
        table = workloads.identity_table(B, pages)
    return workloads.Workload("edge", scores, np.asarray(lens, np.int32), table, page_size, k, max_seq_len, True)


def test_empty_and_tiny_rows():
    rng = np.random.default_rng(1)
    S = 64
    scores = rng.standard_normal((8, S)).astype(np.float32)
    wl = _make(scores, [0, 1, 2, 3, 4, 5, 63, 64], k=4)
    out, raw, _ = run_gpu(wl)
    compare(wl, out, raw)


@pytest.mark.parametrize("k", [1, 2, 511, 512, 513, 2047, 2048])
def test_k_boundaries(k):
    rng = np.random.default_rng(k)
    S = 4100
    lens = [k - 1, k, k + 1, 4097, 4100, 2 * k + 3]
    scores = rng.standard_normal((len(lens), S)).astype(np.float32)
    wl = _make(scores, np.minimum(lens, S), k=k, page_size=4)
    out, raw, _ = run_gpu(wl)
    compare(wl, out, raw)


def test_seq_len_flags():
    from sparse_attention_indexer_uint32_gb300 import _lib  # noqa: F401

    rng = np.random.default_rng(2)
    S = 4096
    scores = rng.standard_normal((4, S)).astype(np.float32)
    wl = _make(scores, [-7, 5000, 3000, 100], k=64, max_seq_len=4000)
    out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags & 0x1 and flags & 0x2


def test_special_values():
    S = 9000
    rng = np.random.default_rng(3)
    base = rng.standard_normal(S).astype(np.float32)
    rows = []
    r = base.copy()
    r[::3] = np.inf
    rows.append(r)
    r = base.copy()
    r[::5] = -np.inf
    r[1::5] = -0.0
    r[2::5] = 0.0
    rows.append(r)
    r = np.where(np.arange(S) % 2 == 0, np.float32(-0.0), np.float32(0.0)).astype(np.float32)
    rows.append(r)
    r = np.full(S, -np.inf, np.float32)
    rows.append(r)
    r = base.copy()
    r[::7] = np.float32(np.nan)
    r.view(np.uint32)[3::11] = 0xFFC00001  # negative NaNs
    r.view(np.uint32)[4::13] = 0x7F800001  # positive NaN with another payload
    rows.append(r)
    r = np.float32(1e-45) * (np.arange(S) % 17).astype(np.float32)  # denormals
    rows.append(r)
    scores = np.stack(rows)
    wl = _make(scores, [S] * len(rows), k=1000, page_size=2)
    out, raw, _ = run_gpu(wl)
    compare(wl, out, raw)


def test_row_stride_larger_than_length_and_unaligned_tail():
    rng = np.random.default_rng(4)
    S = 12004
    lens = [12001, 11999, 7, 5003, 12004, 4097]
    scores = rng.standard_normal((len(lens), S)).astype(np.float32)
    for b, L in enumerate(lens):
        scores[b, L:] = np.inf  # would win if a read past seq_len leaked in
    wl = _make(scores, lens, k=512, page_size=64)
    out, raw, _ = run_gpu(wl)
    compare(wl, out, raw)


@pytest.mark.parametrize("page_size", [1, 2, 128, 1 << 16])
def test_page_sizes_permuted(page_size):
    wl = workloads.random_case(seed=500 + page_size, batch=6, min_len=100, max_len=30000, k=256,
                               page_size=page_size, dist="normal", permuted=True)
    out, raw, _ = run_gpu(wl)
    compare(wl, out, raw)


def test_repeat_runs_identical_sets():
    wl = workloads.random_case(seed=9, batch=24, min_len=0, max_len=80000, k=512, page_size=64, dist="bf16")
    ref_out, ref_raw, _ = run_gpu(wl)
    for _ in range(10):
        out, raw, _ = run_gpu(wl)
        assert (np.sort(out, axis=1) == np.sort(ref_out, axis=1)).all()
        assert (np.sort(raw, axis=1) == np.sort(ref_raw, axis=1)).all()
    compare(wl, ref_out, ref_raw)


def test_many_rows_several_windows_and_plan_sweeps():
    """A batch past one plan sweep (16384 rows) and past one window of work
    items per block (256 rows per block): short rows with ties and a ragged
    tail, every row checked."""
    wl = workloads.random_case(seed=480, batch=130001, min_len=0, max_len=97, k=9, page_size=4, dist="int")
    out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


def test_mixed_batch_with_long_and_short_launches():
    """A batch large enough that the single-block kernel runs first on the short
    rows and the cluster kernel second on the long ones."""
    from sparse_attention_indexer_uint32_gb300 import _lib

    wl = workloads.random_case(seed=481, batch=400, min_len=100, max_len=140000, k=256, page_size=64,
                               dist="bf16")
    assert _lib.topk_transform_launches(wl.batch, wl.max_seq_len, wl.k) == 2
    out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    check_properties_all_rows(wl, raw)
    assert flags == 0


@pytest.mark.parametrize("path", ["auto", "single_block", "split"])
def test_rows_far_past_one_million(path):
    """A 16M-token row, two rows of about 6M and a short one (k = 2048, a
    permuted table): the slice, tile and position arithmetic of the cluster
    kernel (automatic: 16 blocks per row, with the larger per-block buffer
    such rows need) and of one block streaming a whole 64 MB row; for the
    segment-split path, which takes rows of up to about 2M tokens at this k,
    a 2M row, one of 1.5M and a short one."""
    rng = np.random.default_rng(2100)
    S = 1 << 24 if path != "split" else 1 << 21
    lens = [S, 6_000_001, 6_000_000 - 3, 777] if path != "split" else [S, 1_500_001, 777]
    scores = np.full((len(lens), S), np.inf, np.float32)
    for b, L in enumerate(lens):
        scores[b, :L] = rng.standard_normal(L).astype(np.float32)
    table = workloads.permuted_table(rng, len(lens), workloads.pages_for(S, 64))
    wl = _make(scores, lens, k=2048, page_size=64, table=table)
    extra = {"auto": {}, "single_block": dict(long_threshold=1 << 30, long_threshold_small_batch=1 << 30),
             "split": dict(split_rows=1)}[path]
    with tuning(**extra):
        out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


def test_five_to_ten_very_long_rows():
    """Five to ten rows of about 600K tokens through the automatic dispatch
    (the cluster sizes it picks around one wave of 16-block clusters), with
    ragged tails, bf16-rounded scores and a permuted table."""
    import torch

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(2300)
    for batch in (5, sms // 16, sms // 16 + 1):
        S = 600_000
        lens = [S - int(x) for x in rng.integers(0, 80_000, batch)]
        scores = np.full((batch, S), np.inf, np.float32)
        for b, L in enumerate(lens):
            scores[b, :L] = workloads._round_bf16(rng.standard_normal(L).astype(np.float32))
        table = workloads.permuted_table(rng, batch, workloads.pages_for(S, 64))
        wl = workloads.Workload("few_long", scores, np.asarray(lens, np.int32), table, 64, 2048, S, True)
        out, raw, flags = run_gpu(wl)
        compare(wl, out, raw)
        assert flags == 0


def test_three_block_clusters_on_long_mixes():
    """3-block clusters (a cluster size that does not split rows in powers of
    two) on batches of long rows that give 4-block clusters two rows, through
    the automatic dispatch (which takes them for a ragged mix at k = 1024,
    and for 260 mixed rows at k = 512: three waves in one launch) and asked
    for (rows of 70K-300K with k = 2048, where the automatic dispatch keeps
    4 blocks: a 3-block buffer would not hold the gate's floor at 40 %)."""
    rng = np.random.default_rng(2400)
    for batch, lo, hi, k, dist in ((100, 1024, 262144, 1024, "normal"), (160, 70001, 300001, 2048, "bf16"),
                                   (260, 1024, 262144, 512, "bf16")):
        wl = workloads.random_case(seed=int(rng.integers(1 << 30)), batch=batch, min_len=lo, max_len=hi, k=k,
                                   page_size=64, dist=dist)
        out, raw, flags = run_gpu(wl)
        compare(wl, out, raw)
        assert flags == 0
        with tuning(cluster_size=3):
            out, raw, flags = run_gpu(wl)
        compare(wl, out, raw)
        assert flags == 0
