"""Seeded synthetic inputs for the indexer top-k + page-table transform.

This module only draws inputs.  It holds none of the selection or transform
arithmetic, so the CUDA path and the CPU oracle can both be fed from it
without sharing any of the method.

The five workloads follow the shapes the pages benchmark (SGLang PR #26788,
"Performance" and its commit log: decode at batch 8192 x seq 8192, throughput
at batch >= 2048 x seq 64K with k=512 and page size 64; the DistRadixTopK
README's latency table for one row of up to 1M tokens with top-2048; the
LiteTopk PR #32094 "Validation" list for short rows, ties and flat-score
rows):

====  ==========================================================  =========
name  scores                                                      table
====  ==========================================================  =========
tiny  4 x 8192, N(0,1), k=512, page 64, raw output requested      identity
decode 8192 x 8192, N(0,1), k=512, page 64                        permuted
throughput 2048 x 65536, q_b . k_j with q, k ~ N(0,1)^128 fp32    permuted
long  {1,8,32} x 1,048,576, N(0,1) + 0.5 sin(2 pi j / 4096), k=2048 identity
ragged 128 rows, seq_len ~ U[1024, 262144] with short / flat / half--inf
      rows, bf16-representable values, k=1024, page 128           permuted
====  ==========================================================  =========

Every array is produced by numpy's PCG64 generator from a fixed seed, in
float64, and rounded once to float32 (round to nearest even).  The ragged
workload then rounds to the nearest bf16 value (round to nearest even on the
fp32 bit pattern).  Row padding past ``seq_len`` is filled with ``+inf`` so a
read past the end of a row would change the result.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

BASE_SEED = 20261202


@dataclasses.dataclass
class Workload:
    name: str
    scores: np.ndarray  # float32 [batch, row_stride]
    seq_lens: np.ndarray  # int32 [batch]
    page_table: np.ndarray  # int32 [batch, pages_per_row]
    page_size: int
    k: int
    max_seq_len: int
    want_raw: bool = False

    @property
    def batch(self) -> int:
        return int(self.scores.shape[0])

    @property
    def row_stride(self) -> int:
        return int(self.scores.shape[1])

    def algorithmic_bytes(self) -> int:
        """Scores read + seq_lens read + indices written (page table excluded).

        This is the footprint SGLang PR #26788 reports (commit "Pass scores +
        seq_lens + page_table as input_args ...": only about k page-table
        entries are touched per row, so the table is not counted).
        """
        eff = np.clip(self.seq_lens.astype(np.int64), 0, self.max_seq_len)
        outputs = 2 if self.want_raw else 1
        return int(4 * eff.sum() + 4 * self.batch + 4 * self.batch * self.k * outputs)


# Seed offset between shards: shard r of a workload (one per process when
# several GPUs each run their own batch) draws from tag + SHARD_STRIDE * r.
SHARD_STRIDE = 7919


def _rng(tag: int, shard: int = 0) -> np.random.Generator:
    return np.random.default_rng(BASE_SEED + tag + SHARD_STRIDE * shard)


def _normal_f32(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float64).astype(np.float32)


def _round_bf16(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 value (ties to even), kept in float32 storage."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    finite = np.isfinite(x)
    r = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    r = np.where(finite, r, u & 0xFFFF0000).astype(np.uint32)
    return r.view(np.float32)


def identity_table(batch: int, pages: int) -> np.ndarray:
    return np.broadcast_to(np.arange(pages, dtype=np.int32), (batch, pages)).copy()


def permuted_table(rng: np.random.Generator, batch: int, pages: int) -> np.ndarray:
    return rng.permutation(batch * pages).astype(np.int32).reshape(batch, pages)


def pages_for(max_seq_len: int, page_size: int) -> int:
    return max(1, -(-max_seq_len // page_size))


def tiny() -> Workload:
    rng = _rng(1)
    B, L = 4, 8192
    return Workload("tiny_4x8192_k512", _normal_f32(rng, (B, L)), np.full(B, L, np.int32),
                    identity_table(B, pages_for(L, 64)), 64, 512, L, want_raw=True)


def decode(batch: int = 8192, seq_len: int = 8192, shard: int = 0) -> Workload:
    rng = _rng(2, shard)
    scores = _normal_f32(rng, (batch, seq_len))
    table = permuted_table(rng, batch, pages_for(seq_len, 64))
    return Workload(f"decode_{batch}x{seq_len}_k512", scores, np.full(batch, seq_len, np.int32),
                    table, 64, 512, seq_len)


def throughput(batch: int = 2048, seq_len: int = 65536, dim: int = 128, chunk: int = 256,
               shard: int = 0) -> Workload:
    rng = _rng(3, shard)
    q = _normal_f32(rng, (batch, dim)).astype(np.float64)
    kmat = _normal_f32(rng, (seq_len, dim)).astype(np.float64)
    scores = np.empty((batch, seq_len), dtype=np.float32)
    kt = kmat.T.copy()
    for b0 in range(0, batch, chunk):
        scores[b0:b0 + chunk] = (q[b0:b0 + chunk] @ kt).astype(np.float32)
    table = permuted_table(rng, batch, pages_for(seq_len, 64))
    return Workload(f"throughput_{batch}x{seq_len}_k512", scores, np.full(batch, seq_len, np.int32),
                    table, 64, 512, seq_len)


def long_context(batch: int = 1, seq_len: int = 1 << 20, shard: int = 0) -> Workload:
    rng = _rng(4, shard)
    trend = 0.5 * np.sin(2.0 * math.pi * np.arange(seq_len, dtype=np.float64) / 4096.0)
    scores = np.empty((batch, seq_len), dtype=np.float32)
    for b in range(batch):
        scores[b] = (rng.standard_normal(seq_len, dtype=np.float64) + trend).astype(np.float32)
    return Workload(f"long_{batch}x{seq_len}_k2048", scores, np.full(batch, seq_len, np.int32),
                    identity_table(batch, pages_for(seq_len, 64)), 64, 2048, seq_len)


RAGGED_SHORT = {3: 1, 40: 7, 77: 513, 114: 1023}
RAGGED_FLAT = (10, 50, 90, 127)
RAGGED_SIGNED_ZERO = 90
RAGGED_HALF_NEG_INF = (20, 60, 100, 121)
RAGGED_FORCED = {20: 1500}


def ragged(batch: int = 128, max_len: int = 262144, min_len: int = 1024, shard: int = 0) -> Workload:
    rng = _rng(5, shard)
    lens = rng.integers(min_len, max_len, size=batch, endpoint=True).astype(np.int32)
    for b, L in {**RAGGED_SHORT, **RAGGED_FORCED}.items():
        if b < batch:
            lens[b] = L
    scores = np.full((batch, max_len), np.inf, dtype=np.float32)
    for b in range(batch):
        L = int(lens[b])
        row = _round_bf16(_normal_f32(rng, L))
        if b in RAGGED_FLAT:
            row = np.ones(L, dtype=np.float32)
            if b == RAGGED_SIGNED_ZERO:
                row = np.where(np.arange(L) % 2 == 0, np.float32(-0.0), np.float32(0.0)).astype(np.float32)
        if b in RAGGED_HALF_NEG_INF:
            row = np.where(rng.random(L) < 0.5, np.float32(-np.inf), row).astype(np.float32)
        scores[b, :L] = row
    table = permuted_table(rng, batch, pages_for(max_len, 128))
    return Workload(f"ragged_{batch}_k1024", scores, lens, table, 128, 1024, max_len)


def random_case(seed: int, batch: int, min_len: int, max_len: int, k: int, page_size: int,
                dist: str = "normal", row_stride: int | None = None, want_raw: bool = True,
                permuted: bool = True) -> Workload:
    """Small seeded cases for parity tests (several tiles and a ragged tail).

    ``dist``: "normal" (N(0,1) fp32), "bf16" (N(0,1) rounded to bf16),
    "int" (small integers, heavy ties), "flat" (all 1.0), "neginf" (half -inf).
    """
    rng = np.random.default_rng(BASE_SEED + 1000 + seed)
    lens = rng.integers(min_len, max_len, size=batch, endpoint=True).astype(np.int32)
    if row_stride is None:
        row_stride = max(4, -(-int(lens.max()) // 4) * 4)
    scores = np.full((batch, row_stride), np.inf, dtype=np.float32)
    for b in range(batch):
        L = int(lens[b])
        if dist == "normal":
            row = _normal_f32(rng, L)
        elif dist == "bf16":
            row = _round_bf16(_normal_f32(rng, L))
        elif dist == "int":
            row = rng.integers(-8, 8, size=L).astype(np.float32)
        elif dist == "flat":
            row = np.ones(L, dtype=np.float32)
        elif dist == "neginf":
            row = np.where(rng.random(L) < 0.5, np.float32(-np.inf), _normal_f32(rng, L)).astype(np.float32)
        else:
            raise ValueError(dist)
        scores[b, :L] = row
    pages = pages_for(row_stride, page_size)
    table = permuted_table(rng, batch, pages) if permuted else identity_table(batch, pages)
    return Workload(f"random_{dist}_{seed}", scores, lens, table, page_size, k, row_stride, want_raw)
