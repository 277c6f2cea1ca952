"""GPU parity of the warp-per-row kernel (short rows, k <= 512) against the
CPU oracle: the kernel forced on small batches (`warp_rows = 1`), over the
score distributions, k boundaries, special values, ragged tails and every
fallback (a gate too tight or too loose, no gate, the histogram-only pass),
on batches with several rows per warp, and on the full decode workload."""
from __future__ import annotations

import numpy as np
import pytest

from sparse_attention_indexer_uint32_gb300 import workloads
from tests.parity_util import compare, run_gpu, tuning

pytestmark = pytest.mark.gpu

DISTS = ["normal", "bf16", "int", "flat", "neginf"]


def _make(scores, lens, k, page_size=1):
    scores = np.ascontiguousarray(scores, np.float32)
    B, S = scores.shape
    table = workloads.identity_table(B, workloads.pages_for(S, page_size))
    return workloads.Workload("edge", scores, np.asarray(lens, np.int32), table, page_size, k, S, True)


@pytest.mark.parametrize("dist", DISTS)
@pytest.mark.parametrize("k", [1, 37, 512])
def test_warp_random_ragged(dist, k):
    wl = workloads.random_case(seed=600 + DISTS.index(dist) * 1000 + k, batch=48, min_len=0, max_len=16384, k=k,
                               page_size=16, dist=dist, permuted=True)
    with tuning(warp_rows=1):
        out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


@pytest.mark.parametrize("mode", ["two_pass", "ungated", "fill1", "fill100"])
def test_warp_fallbacks(mode):
    """two_pass: radix rounds over re-reads and a collect pass; ungated: the
    buffer overflows on long rows and the row is re-read; fill1 / fill100:
    the gate at its sampling bound or aimed at the whole buffer."""
    extra = {"two_pass": dict(force_two_pass=1), "ungated": dict(disable_gate=1),
             "fill1": dict(gate_fill_percent=1), "fill100": dict(gate_fill_percent=100)}[mode]
    for dist in ("normal", "bf16", "flat"):
        wl = workloads.random_case(seed=650 + len(mode) + DISTS.index(dist), batch=24, min_len=0, max_len=16384,
                                   k=300, page_size=64, dist=dist)
        with tuning(warp_rows=1, **extra):
            out, raw, flags = run_gpu(wl)
        compare(wl, out, raw)
        assert flags == 0


@pytest.mark.parametrize("k", [1, 2, 511, 512])
def test_warp_k_boundaries(k):
    rng = np.random.default_rng(700 + k)
    S = 4100
    lens = [k - 1, k, k + 1, 4097, 4100, 2 * k + 3, 1025, 1023]
    scores = rng.standard_normal((len(lens), S)).astype(np.float32)
    wl = _make(scores, np.clip(lens, 0, S), k=k, page_size=4)
    with tuning(warp_rows=1):
        out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


def test_warp_special_values():
    S = 9000
    rng = np.random.default_rng(710)
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
    r.view(np.uint32)[3::11] = 0xFFC00001  # negative NaNs
    r.view(np.uint32)[4::13] = 0x7F800001  # positive NaN with another payload
    rows.append(r)
    r = np.full(S, np.float32(1.0))
    r.view(np.uint32)[::2] = 0xFFFFFFFF  # the lowest key of all, tied
    rows.append(r)
    rows.append(np.float32(1e-45) * (np.arange(S) % 17).astype(np.float32))  # denormals
    rows.append(np.arange(S, dtype=np.float32))  # increasing: the top k at the end
    rows.append(-np.arange(S, dtype=np.float32))  # decreasing: the top k at the start
    wl = _make(np.stack(rows), [S] * len(rows), k=500, page_size=2)
    for extra in ({}, {"disable_gate": 1}, {"force_two_pass": 1}):
        with tuning(warp_rows=1, **extra):
            out, raw, flags = run_gpu(wl)
        compare(wl, out, raw)
        assert flags == 0


def test_warp_unaligned_tails_and_stride():
    rng = np.random.default_rng(720)
    S = 12004
    lens = [12001, 11999, 7, 5003, 12004, 4097, 513, 514, 515]
    scores = rng.standard_normal((len(lens), S)).astype(np.float32)
    for b, L in enumerate(lens):
        scores[b, L:] = np.inf  # would win if a read past seq_len leaked in
    wl = _make(scores, lens, k=512, page_size=64)
    with tuning(warp_rows=1):
        out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


def test_warp_ties_across_the_threshold():
    """Many copies of the k-th value spread over the row: the smallest
    positions among them are taken (the position bitmap), from the buffer and
    from the re-read path."""
    rng = np.random.default_rng(730)
    S = 16384
    rows = []
    for frac in (0.01, 0.1, 0.5):
        r = rng.standard_normal(S).astype(np.float32)
        tie = rng.random(S) < frac
        r[tie] = np.float32(1.5)
        rows.append(r)
    wl = _make(np.stack(rows), [S, S - 5, S - 100], k=512, page_size=8)
    for extra in ({}, {"force_two_pass": 1}):
        with tuning(warp_rows=1, **extra):
            out, raw, flags = run_gpu(wl)
        compare(wl, out, raw)
        assert flags == 0


@pytest.mark.parametrize("dist", ["bf16", "int"])
def test_warp_many_rows_per_warp(dist):
    """More rows than warps in flight (the grid is capped at the resident
    blocks): each warp resolves several rows in turn, so every per-warp
    structure must be clean again after each row."""
    wl = workloads.random_case(seed=740 + DISTS.index(dist), batch=6000, min_len=0, max_len=3000, k=100,
                               page_size=32, dist=dist)
    with tuning(warp_rows=1):
        out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


def test_warp_decode_workload():
    """The 8192 x 8192 decode workload through the warp kernel: every row
    against the oracle, and every row against the selection properties."""
    from tests.parity_util import check_properties_all_rows

    wl = workloads.decode()
    with tuning(warp_rows=1):
        out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    check_properties_all_rows(wl, raw)
    assert flags == 0
