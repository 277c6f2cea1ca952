"""GPU parity of the warp-specialised single-block kernel (8 streaming warps,
4 or 8 resolving warps, two candidate-buffer / histogram sets; rows of up to
65536) against the CPU oracle: the kernel forced (`single_block_kernel = 2`) over the score
distributions, k boundaries, special values and ragged tails, every fallback
of the resolving warps (a gate too tight or too loose, no gate, the
histogram-only first pass, buffer overflow), batches whose rows span several
work windows, and the mixed launch with the cluster kernel."""
from __future__ import annotations

import numpy as np
import pytest

from sparse_attention_indexer_uint32_gb300 import workloads
from tests.parity_util import compare, run_gpu, tuning

pytestmark = pytest.mark.gpu

DISTS = ["normal", "bf16", "int", "flat", "neginf"]
SHAPES = [2, 3]  # 4 resolving warps, two blocks per SM; 8 resolving warps, one block per SM


def single(shape):
    return dict(single_block_kernel=shape, long_threshold=1 << 30, long_threshold_small_batch=1 << 30)


def _make(scores, lens, k, page_size=1):
    scores = np.ascontiguousarray(scores, np.float32)
    B, S = scores.shape
    table = workloads.identity_table(B, workloads.pages_for(S, page_size))
    return workloads.Workload("edge", scores, np.asarray(lens, np.int32), table, page_size, k, S, True)


@pytest.mark.parametrize("dist", DISTS)
@pytest.mark.parametrize("k", [1, 37, 512, 640, 2048])
@pytest.mark.parametrize("shape", SHAPES)
def test_stream_random_ragged(dist, k, shape):
    wl = workloads.random_case(seed=900 + DISTS.index(dist) * 1000 + k, batch=40, min_len=0, max_len=65536, k=k,
                               page_size=64, dist=dist)
    with tuning(**single(shape)):
        out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


@pytest.mark.parametrize("mode", ["two_pass", "ungated", "few_samples", "fill1", "fill100", "small_cap"])
@pytest.mark.parametrize("shape", SHAPES)
def test_stream_fallbacks(mode, shape):
    """two_pass: every row resolved from re-reads; ungated: every element
    counted, the buffer overflows on long rows; few_samples / fill1: gates
    tighter than the k-th key (recounts); fill100 / small_cap: buffers that
    overflow (collect passes)."""
    extra = {"two_pass": dict(force_two_pass=1), "ungated": dict(disable_gate=1), "few_samples": dict(samples=32),
             "fill1": dict(gate_fill_percent=1), "fill100": dict(gate_fill_percent=100),
             "small_cap": dict(candidate_capacity=2048)}[mode]
    for dist in ("normal", "bf16", "flat", "neginf"):
        wl = workloads.random_case(seed=950 + len(mode) * 7 + DISTS.index(dist), batch=24, min_len=0,
                                   max_len=65536, k=512, page_size=32, dist=dist)
        with tuning(**single(shape), **extra):
            out, raw, flags = run_gpu(wl)
        compare(wl, out, raw)
        assert flags == 0


@pytest.mark.parametrize("shape", SHAPES)
def test_stream_special_values(shape):
    S = 40000
    rng = np.random.default_rng(960)
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
    rows.append(np.where(np.arange(S) % 2 == 0, np.float32(-0.0), np.float32(0.0)).astype(np.float32))
    rows.append(np.full(S, -np.inf, np.float32))
    r = base.copy()
    r[::7] = np.float32(np.nan)
    r.view(np.uint32)[3::11] = 0xFFC00001
    r.view(np.uint32)[4::13] = 0x7F800001
    rows.append(r)
    rows.append(np.float32(1e-45) * (np.arange(S) % 17).astype(np.float32))
    rows.append(np.arange(S, dtype=np.float32))
    rows.append(-np.arange(S, dtype=np.float32))
    wl = _make(np.stack(rows), [S] * len(rows), k=1000, page_size=2)
    for extra in ({}, {"disable_gate": 1}, {"force_two_pass": 1}):
        with tuning(**single(shape), **extra):
            out, raw, flags = run_gpu(wl)
        compare(wl, out, raw)


@pytest.mark.parametrize("shape", SHAPES)
def test_stream_ties_across_the_threshold(shape):
    """Many copies of the k-th value: the smallest positions among them, from
    the buffer (position rounds) and from re-reads (the ordered final pass)."""
    rng = np.random.default_rng(970)
    S = 65536
    rows = []
    for frac in (0.002, 0.02, 0.2, 0.6):
        r = rng.standard_normal(S).astype(np.float32)
        r[rng.random(S) < frac] = np.float32(1.75)
        rows.append(r)
    wl = _make(np.stack(rows), [S, S - 3, S - 100, 40000], k=512, page_size=16)
    for extra in ({}, {"force_two_pass": 1}, {"candidate_capacity": 2048}):
        with tuning(**single(shape), **extra):
            out, raw, flags = run_gpu(wl)
        compare(wl, out, raw)
        assert flags == 0


@pytest.mark.parametrize("shape", SHAPES)
def test_stream_unaligned_tails_and_stride(shape):
    rng = np.random.default_rng(980)
    S = 60004
    lens = [60001, 59999, 7, 24577, 60004, 16385, 513, 514, 515, 6145, 6143]
    scores = rng.standard_normal((len(lens), S)).astype(np.float32)
    for b, L in enumerate(lens):
        scores[b, L:] = np.inf  # would win if a read past seq_len leaked in
    wl = _make(scores, lens, k=512, page_size=64)
    with tuning(**single(shape)):
        out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


@pytest.mark.parametrize("shape", SHAPES)
def test_stream_many_rows_several_windows(shape):
    """More rows per block than one window of work items (256): the
    hand-over phases and the ring carry across windows; short and trivial
    rows (L <= k) mixed in."""
    wl = workloads.random_case(seed=990, batch=120001, min_len=0, max_len=700, k=33, page_size=4, dist="int")
    with tuning(**single(shape)):
        out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


@pytest.mark.parametrize("shape", SHAPES)
def test_stream_k_boundaries(shape):
    rng = np.random.default_rng(995)
    S = 20004
    for k in (511, 512, 513, 640, 2047, 2048):
        lens = [k - 1, k, k + 1, 20001, 20004, 2 * k + 3, 6144, 6145]
        scores = rng.standard_normal((len(lens), S)).astype(np.float32)
        wl = _make(scores, np.minimum(lens, S), k=k, page_size=4)
        with tuning(**single(shape)):
            out, raw, flags = run_gpu(wl)
        compare(wl, out, raw)
        assert flags == 0


@pytest.mark.parametrize("shape", SHAPES)
def test_stream_with_cluster_launch(shape):
    """A large mixed batch: the warp-specialised kernel takes the short list,
    the cluster kernel the long one."""
    from sparse_attention_indexer_uint32_gb300 import _lib

    wl = workloads.random_case(seed=996, batch=600, min_len=100, max_len=300000, k=512, page_size=64, dist="bf16")
    with tuning(single_block_kernel=shape, long_threshold_large_batch=65536):
        assert _lib.topk_transform_launches(wl.batch, wl.max_seq_len, wl.k) == 2
        out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


@pytest.mark.parametrize("shape", SHAPES)
def test_stream_and_single_role_kernels_agree_on_the_throughput_shape(shape):
    """Rows of the 64K throughput shape through both single-block kernels."""
    wl = workloads.random_case(seed=997, batch=300, min_len=30000, max_len=65536, k=512, page_size=64,
                               dist="normal")
    with tuning(single_block_kernel=shape):
        out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    with tuning(single_block_kernel=1):
        out1, raw1, _ = run_gpu(wl)
    compare(wl, out1, raw1)
