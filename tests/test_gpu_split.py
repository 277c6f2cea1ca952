"""GPU parity of the segment-split path (the rows of a batch of up to 128 cut
into segments that every SM streams; the block that finishes a row's last
segment resolves the row) against the CPU oracle: the path forced
(`split_rows = 1`) over the score distributions, k boundaries, segment sizes,
special values and ragged tails; each of its three resolves (k or more
candidates above the gate; the candidates plus the smallest positions tied at
the gate key; the full-row path, forced and through an ungated overflow);
batches of 1 to 128 rows; a reused plan; and the automatic dispatch."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest

from sparse_attention_indexer_uint32_gb300 import workloads
from tests.parity_util import compare, run_gpu, tuning

pytestmark = pytest.mark.gpu

DISTS = ["normal", "bf16", "int", "flat", "neginf"]


def split(**extra):
    return dict(split_rows=1, **extra)


def _make(scores, lens, k, page_size=1):
    scores = np.ascontiguousarray(scores, np.float32)
    B, S = scores.shape
    table = workloads.identity_table(B, workloads.pages_for(S, page_size))
    return workloads.Workload("edge", scores, np.asarray(lens, np.int32), table, page_size, k, S, True)


@pytest.mark.parametrize("dist", DISTS)
@pytest.mark.parametrize("k", [1, 37, 512, 1024, 2048])
def test_split_random_ragged(dist, k):
    wl = workloads.random_case(seed=1200 + DISTS.index(dist) * 1000 + k, batch=48, min_len=0, max_len=150000,
                               k=k, page_size=64, dist=dist)
    with tuning(**split()):
        out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


@pytest.mark.parametrize("seg", [4096, 8192, 65536])
@pytest.mark.parametrize("dist", ["bf16", "flat", "int"])
def test_split_segment_sizes(seg, dist):
    """Small segments put a row's ties and candidates in many segments; a
    large one puts whole rows in one segment."""
    wl = workloads.random_case(seed=1300 + seg // 4096 + len(dist), batch=20, min_len=1000, max_len=300000,
                               k=1024, page_size=128, dist=dist)
    with tuning(**split(split_segment=seg)):
        out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


@pytest.mark.parametrize("mode", ["full", "ungated"])
@pytest.mark.parametrize("dist", ["normal", "int", "flat", "neginf"])
def test_split_full_row_path(mode, dist):
    """full: every row resolved by radix rounds over the whole row read from
    memory; ungated: every element is a candidate, so rows longer than the
    candidate buffer overflow into that path and shorter ones resolve from
    the buffer."""
    extra = {"full": dict(split_full_resolve=1), "ungated": dict(disable_gate=1)}[mode]
    wl = workloads.random_case(seed=1400 + DISTS.index(dist) + len(mode), batch=12, min_len=0, max_len=60000,
                               k=512, page_size=32, dist=dist)
    with tuning(**split(**extra)):
        out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


def test_split_special_values():
    S = 40000
    rng = np.random.default_rng(1500)
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
    for extra in ({}, {"disable_gate": 1}, {"split_full_resolve": 1}, {"split_segment": 4096}):
        with tuning(**split(**extra)):
            out, raw, flags = run_gpu(wl)
        compare(wl, out, raw)
        assert flags == 0


def test_split_ties_across_the_threshold():
    """Many copies of the k-th value, at the gate key or above it: the
    smallest positions among them, from the candidates (distinct composites)
    and from the ordered re-read of the tied segments."""
    rng = np.random.default_rng(1600)
    S = 200000
    rows = []
    for frac in (0.002, 0.02, 0.2, 0.6, 1.0):
        r = rng.standard_normal(S).astype(np.float32)
        r[rng.random(S) < frac] = np.float32(1.75)
        rows.append(r)
    r = np.full(S, -np.inf, np.float32)  # a few finite values among -inf
    r[rng.integers(0, S, 300)] = rng.standard_normal(300).astype(np.float32)
    rows.append(r)
    wl = _make(np.stack(rows), [S, S - 3, S - 100, 40000, S - 1, S], k=512, page_size=16)
    for extra in ({}, {"split_segment": 4096}, {"split_full_resolve": 1}):
        with tuning(**split(**extra)):
            out, raw, flags = run_gpu(wl)
        compare(wl, out, raw)
        assert flags == 0


def test_split_unaligned_tails():
    rng = np.random.default_rng(1700)
    S = 140004
    lens = [140001, 139999, 7, 24577, 140004, 16385, 513, 514, 515, 6145, 6143, 0, 1, 65537, 4097]
    scores = rng.standard_normal((len(lens), S)).astype(np.float32)
    for b, L in enumerate(lens):
        scores[b, L:] = np.inf  # would win if a read past seq_len leaked in
    wl = _make(scores, lens, k=512, page_size=64)
    for seg in (0, 4096):
        with tuning(**split(split_segment=seg)):
            out, raw, flags = run_gpu(wl)
        compare(wl, out, raw)
        assert flags == 0


def test_split_k_boundaries():
    rng = np.random.default_rng(1800)
    S = 40004
    for k in (1, 511, 512, 513, 1023, 1024, 2047, 2048):
        lens = [k - 1, k, k + 1, 40001, 40004, 2 * k + 3, 8191, 8193, 12289]
        scores = rng.standard_normal((len(lens), S)).astype(np.float32)
        wl = _make(scores, np.minimum(lens, S), k=k, page_size=4)
        with tuning(**split(split_segment=4096)):
            out, raw, flags = run_gpu(wl)
        compare(wl, out, raw)
        assert flags == 0


@pytest.mark.parametrize("batch", [1, 2, 127, 128])
def test_split_batch_sizes(batch):
    max_len = 1 << 20 if batch <= 2 else 40000
    wl = workloads.random_case(seed=1900 + batch, batch=batch, min_len=max_len // 2, max_len=max_len, k=2048,
                               page_size=64, dist="bf16")
    with tuning(**split()):
        out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


def test_split_plan_reused_by_two_transforms():
    """The gate kernel rewrites every counter of the split state, so one plan
    serves consecutive transforms on different scores."""
    import torch

    from sparse_attention_indexer_uint32_gb300 import _lib, api

    dev = torch.device("cuda", 0)
    a = workloads.random_case(seed=2000, batch=30, min_len=0, max_len=200000, k=1024, page_size=64, dist="bf16")
    # the same lengths and table (one plan), other scores: a's negated
    b = dataclasses.replace(a, scores=np.ascontiguousarray(-a.scores))
    seq = torch.from_numpy(a.seq_lens).to(dev)
    table = torch.from_numpy(a.page_table).to(dev)
    ws = torch.zeros(_lib.topk_plan_workspace_bytes(a.batch), dtype=torch.uint8, device=dev)
    with tuning(**split()):
        api.plan(seq, a.max_seq_len, ws)
        for wl in (a, b, a):
            scores = torch.from_numpy(wl.scores).to(dev)
            out = torch.empty((wl.batch, wl.k), dtype=torch.int32, device=dev)
            raw = torch.empty_like(out)
            _lib.topk_transform(scores, wl.row_stride, seq, wl.batch, wl.max_seq_len, table,
                                wl.page_table.shape[1], wl.page_size, wl.k, out, raw, ws)
            torch.cuda.synchronize()
            compare(wl, out.cpu().numpy(), raw.cpu().numpy())
    assert _lib.topk_read_flags(ws) == 0


def test_split_flat_and_neginf_rows_in_the_ragged_mix():
    """The ragged workload's shape at a smaller width: flat rows and half -inf
    rows resolve through the tie path, short rows are written by the gate."""
    wl = workloads.ragged(batch=128, max_len=65536, min_len=1024)
    with tuning(**split()):
        out, raw, flags = run_gpu(wl)
    compare(wl, out, raw)
    assert flags == 0


@pytest.mark.parametrize("path", ["auto", "split"])
def test_skewed_batches(path):
    """A few very long rows among many short ones: the shapes where the split
    path is faster, and where the cluster size floor (buffers at most 80 %
    full at the gate's sampling floor) keeps the cluster path off its
    overflow path."""
    rng = np.random.default_rng(2200)
    for lens, k in (([1 << 20] * 2 + [4096] * 62, 2048), ([1 << 21] + [16384] * 15, 2048),
                    ([1 << 20] * 4 + [8192] * 124, 1024)):
        S = max(lens)
        scores = np.full((len(lens), S), np.inf, np.float32)
        for b, L in enumerate(lens):
            scores[b, :L] = workloads._round_bf16(rng.standard_normal(L).astype(np.float32))
        table = workloads.permuted_table(rng, len(lens), workloads.pages_for(S, 64))
        wl = workloads.Workload("skew", scores, np.asarray(lens, np.int32), table, 64, k, S, True)
        with tuning(**({} if path == "auto" else split())):
            out, raw, flags = run_gpu(wl)
        compare(wl, out, raw)
        assert flags == 0
