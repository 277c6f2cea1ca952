"""Pins of the CPU oracle to facts that do not come from the oracle itself.

* hand-worked examples (``tests/golden/hand_worked.txt``, each with its source);
* brute force over every subset of tiny rows drawn from a tie-heavy alphabet;
* invariants on random rows (count, -1 padding, selected >= unselected,
  tie order, no duplicates);
* closed forms (flat, increasing, decreasing rows);
* a library cross-check on tie-free rows (numpy's stable argsort);
* page-transform facts (identity table, inverse of a permutation, brute force
  over page sizes);
* planted mistakes: each mutant build of the oracle must fail at least one pin.
"""
from __future__ import annotations

import itertools
import math
import os

import numpy as np
import pytest

import oracle
from oracle import oracle as oracle_mod
from tests.golden_cases import load_cases

CASES = load_cases()
ALPHABET = [-math.inf, -1.0, -0.0, 0.0, 1.0, math.inf]


def _run_case(case, lib_path=oracle_mod.LIBRARY):
    scores = case.scores[None, :]
    table = case.table[None, :]
    out, raw, flags = oracle.topk_transform(
        scores, np.array([case.seq_len], np.int32), table, case.page_size, case.k,
        max_seq_len=case.max_seq_len, lib_path=lib_path)
    return out[0], raw[0], flags


def check_golden(lib_path=oracle_mod.LIBRARY):
    for case in CASES:
        out, raw, flags = _run_case(case, lib_path)
        n = case.k - case.pad
        assert sorted(raw[:n].tolist()) == case.raw, case.name
        assert (raw[n:] == -1).all(), case.name
        assert sorted(out[:n].tolist()) == sorted(case.out), case.name
        assert (out[n:] == -1).all(), case.name
        if case.seq_len < 0:
            assert flags & oracle.FLAG_SEQ_NEGATIVE, case.name
        if case.seq_len > case.max_seq_len:
            assert flags & oracle.FLAG_SEQ_CLAMPED, case.name


@pytest.mark.parametrize("case", CASES, ids=[c.name for c in CASES])
def test_golden_case(case):
    out, raw, flags = _run_case(case)
    n = case.k - case.pad
    assert sorted(raw[:n].tolist()) == case.raw
    assert (raw[n:] == -1).all()
    assert sorted(out[:n].tolist()) == sorted(case.out)
    assert (out[n:] == -1).all()
    # slot alignment: out[j] is the transform of raw[j], in 32-bit wrap-around
    for j in range(n):
        r = int(raw[j])
        v = (int(case.table[r // case.page_size]) * case.page_size + r % case.page_size) % (1 << 32)
        assert int(out[j]) == (v - (1 << 32) if v >= (1 << 31) else v)
    if case.seq_len < 0:
        assert flags & oracle.FLAG_SEQ_NEGATIVE
    if case.seq_len > case.max_seq_len:
        assert flags & oracle.FLAG_SEQ_CLAMPED


def brute_force_set(row: list[float], k: int) -> list[int]:
    """The unique size-min(k, L) subset S with (i) every selected score >=
    every unselected score and (ii) among equal scores across the boundary,
    every selected position < every unselected one.  Found by enumeration."""
    L = len(row)
    n = min(k, L)
    found = []
    for subset in itertools.combinations(range(L), n):
        s = set(subset)
        ok = True
        for a in s:
            for u in range(L):
                if u in s:
                    continue
                if row[a] < row[u]:
                    ok = False
                elif row[a] == row[u] and a > u:
                    ok = False
                if not ok:
                    break
            if not ok:
                break
        if ok:
            found.append(sorted(subset))
    assert len(found) == 1, (row, k, found)
    return found[0]


def _tiny_rows(rng, count, max_len):
    rows = []
    for L in range(0, 4):
        rows.extend(list(r) for r in itertools.product(ALPHABET, repeat=L))
    for _ in range(count):
        L = int(rng.integers(4, max_len + 1))
        rows.append([ALPHABET[i] for i in rng.integers(0, len(ALPHABET), L)])
    return rows


def check_brute_force(lib_path=oracle_mod.LIBRARY, count=400, max_len=7):
    rng = np.random.default_rng(7)
    for row in _tiny_rows(rng, count, max_len):
        L = len(row)
        stride = max(L, 1)
        scores = np.zeros((1, stride), np.float32)
        scores[0, :L] = row
        for k in range(1, L + 3):
            _, raw, _ = oracle.topk_transform(scores, np.array([L], np.int32),
                                              np.arange(stride, dtype=np.int32)[None, :], 1, k,
                                              lib_path=lib_path)
            n = min(k, L)
            assert sorted(raw[0, :n].tolist()) == brute_force_set(row, k), (row, k)
            assert (raw[0, n:] == -1).all()


def test_brute_force_tiny_rows():
    check_brute_force()


def _check_invariants(scores, lens, k, raw):
    for b in range(scores.shape[0]):
        L = int(min(max(lens[b], 0), scores.shape[1]))
        n = min(k, L)
        sel = raw[b, :n]
        assert (raw[b, n:] == -1).all()
        assert len(set(sel.tolist())) == n
        assert ((sel >= 0) & (sel < L)).all()
        row = scores[b, :L].astype(np.float64)
        mask = np.zeros(L, bool)
        mask[sel] = True
        if n == 0 or n == L:
            continue
        vmin = row[mask].min()
        vmax_un = row[~mask].max()
        assert vmin >= vmax_un
        # tie order at the boundary: unselected equal values come after selected ones
        eq_sel = np.nonzero(mask & (row == vmin))[0]
        eq_un = np.nonzero(~mask & (row == vmin))[0]
        if len(eq_un):
            assert eq_sel.max() < eq_un.min()


@pytest.mark.parametrize("dist", ["normal", "int", "bf16"])
def test_invariants_random(dist):
    rng = np.random.default_rng(11)
    B, S = 24, 700
    lens = rng.integers(0, S + 1, B).astype(np.int32)
    if dist == "normal":
        scores = rng.standard_normal((B, S)).astype(np.float32)
    elif dist == "int":
        scores = rng.integers(-3, 4, (B, S)).astype(np.float32)
    else:
        scores = (rng.standard_normal((B, S)) * 4).round().astype(np.float32) / 4
    for k in (1, 5, 64, 699, 1000):
        _, raw, _ = oracle.topk_transform(scores, lens, np.zeros((B, S), np.int32), 1, k)
        _check_invariants(scores, lens, k, raw)


def test_closed_forms():
    L, k = 300, 37
    inc = np.arange(L, dtype=np.float32)[None, :]
    _, raw, _ = oracle.topk_transform(inc, np.array([L], np.int32), np.zeros((1, L), np.int32), 1, k)
    assert sorted(raw[0].tolist()) == list(range(L - k, L))
    dec = inc[:, ::-1].copy()
    _, raw, _ = oracle.topk_transform(dec, np.array([L], np.int32), np.zeros((1, L), np.int32), 1, k)
    assert sorted(raw[0].tolist()) == list(range(k))
    flat = np.full((1, L), -2.5, np.float32)
    _, raw, _ = oracle.topk_transform(flat, np.array([L], np.int32), np.zeros((1, L), np.int32), 1, k)
    assert raw[0].tolist() == list(range(k))
    neg = np.full((1, L), -np.inf, np.float32)
    _, raw, _ = oracle.topk_transform(neg, np.array([L], np.int32), np.zeros((1, L), np.int32), 1, k)
    assert sorted(raw[0].tolist()) == list(range(k))


def test_library_cross_check_tie_free():
    rng = np.random.default_rng(3)
    B, S, k = 16, 5000, 300
    scores = rng.permutation(B * S).reshape(B, S).astype(np.float32) - B * S / 2  # distinct values
    lens = rng.integers(0, S + 1, B).astype(np.int32)
    _, raw, _ = oracle.topk_transform(scores, lens, np.zeros((B, S), np.int32), 1, k)
    for b in range(B):
        L = int(lens[b])
        expect = np.argsort(-scores[b, :L].astype(np.float64), kind="stable")[:min(k, L)]
        assert sorted(raw[b, :min(k, L)].tolist()) == sorted(expect.tolist())


def check_page_transform(lib_path=oracle_mod.LIBRARY):
    rng = np.random.default_rng(5)
    for P in (1, 2, 64, 128):
        B, L, k = 6, 3 * P + 5, 7
        NP = -(-L // P)
        scores = rng.standard_normal((B, L)).astype(np.float32)
        lens = np.full(B, L, np.int32)
        perm = rng.permutation(B * NP).astype(np.int32).reshape(B, NP)
        out, raw, _ = oracle.topk_transform(scores, lens, perm, P, k, lib_path=lib_path)
        for b in range(B):
            for j in range(k):
                r = int(raw[b, j])
                assert out[b, j] == perm[b, r // P] * P + r % P
                page, off = divmod(int(out[b, j]), P)
                b2, p2 = np.argwhere(perm == page)[0]
                assert b2 == b and p2 * P + off == r  # the permutation's inverse recovers raw
        ident = np.broadcast_to(np.arange(NP, dtype=np.int32), (B, NP)).copy()
        out, raw, _ = oracle.topk_transform(scores, lens, ident, P, k, lib_path=lib_path)
        assert (out == raw).all()
        pt = oracle.page_transform(raw, perm, P, lib_path=lib_path)
        assert (pt == np.where(raw < 0, -1, perm[np.arange(B)[:, None], np.maximum(raw, 0) // P] * P
                               + np.maximum(raw, 0) % P)).all()


def test_page_transform_pins():
    check_page_transform()


def test_seq_len_flags_and_padding():
    scores = np.arange(40, dtype=np.float32).reshape(4, 10)
    lens = np.array([-3, 0, 4, 25], np.int32)
    out, raw, flags = oracle.topk_transform(scores, lens, np.zeros((4, 10), np.int32), 1, 6, max_seq_len=8)
    assert flags == oracle.FLAG_SEQ_CLAMPED | oracle.FLAG_SEQ_NEGATIVE
    assert (raw[0] == -1).all() and (raw[1] == -1).all()
    assert sorted(raw[2, :4].tolist()) == [0, 1, 2, 3] and (raw[2, 4:] == -1).all()
    assert sorted(raw[3].tolist()) == [2, 3, 4, 5, 6, 7]  # clamped to 8 positions


def test_plan_classify():
    lens = np.array([-1, 0, 10, 11, 50, 1000], np.int32)
    eff, is_long, flags = oracle.plan_classify(lens, 100, 10)
    assert eff.tolist() == [0, 0, 10, 11, 50, 100]
    assert is_long.tolist() == [False, False, False, True, True, True]
    assert flags == oracle.FLAG_SEQ_CLAMPED | oracle.FLAG_SEQ_NEGATIVE


def test_multithreaded_matches_single_thread():
    rng = np.random.default_rng(9)
    B, S = 33, 900
    scores = (rng.standard_normal((B, S)) * 3).round().astype(np.float32)
    lens = rng.integers(0, S + 1, B).astype(np.int32)
    table = rng.permutation(B * S).astype(np.int32).reshape(B, S)
    a = oracle.topk_transform(scores, lens, table, 1, 50, nthreads=1)
    b = oracle.topk_transform(scores, lens, table, 1, 50, nthreads=8)
    assert (a[0] == b[0]).all() and (a[1] == b[1]).all() and a[2] == b[2]


MUTANTS = [
    "ORACLE_MUTATION_TIE_LARGER_INDEX",
    "ORACLE_MUTATION_ASCENDING",
    "ORACLE_MUTATION_SIGNED_ZERO",
    "ORACLE_MUTATION_PAGE_OFFSET",
    "ORACLE_MUTATION_NO_CLAMP_COUNT",
    "ORACLE_MUTATION_NAN_PAYLOAD",
]


@pytest.mark.parametrize("mutant", MUTANTS)
def test_planted_mistakes_are_caught(mutant, tmp_path):
    """Each planted mistake in the oracle must make at least one pin fail."""
    path = oracle_mod.build(os.path.join(str(tmp_path), f"lib_{mutant}.so"), (mutant,))
    oracle_mod.load(path)
    failures = 0
    for check in (check_golden, check_brute_force, check_page_transform):
        try:
            if check is check_brute_force:
                check(path, count=60)
            else:
                check(path)
        except (AssertionError, IndexError, ValueError):
            failures += 1
    assert failures >= 1, f"{mutant} survived every pin"
