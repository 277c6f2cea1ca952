"""The all-rows property check used on full-size GPU runs, pinned on the CPU:
it accepts the oracle's answer and rejects planted mistakes (a lower score
swapped in, a tie broken toward the larger position, a repeated position, a
position past the row)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from sparse_attention_indexer_uint32_gb300 import workloads
from tests.parity_util import check_properties_all_rows


def _case(dist):
    return workloads.random_case(seed=9100 + len(dist), batch=12, min_len=0, max_len=3000, k=100, page_size=16,
                                 dist=dist)


@pytest.mark.parametrize("dist", ["normal", "bf16", "int", "flat"])
def test_accepts_the_oracle(dist):
    wl = _case(dist)
    _, raw, _ = oracle.topk_transform(wl.scores, wl.seq_lens, wl.page_table, wl.page_size, wl.k,
                                      max_seq_len=wl.max_seq_len, want_raw=True)
    check_properties_all_rows(wl, raw)


def _oracle_raw(wl):
    return oracle.topk_transform(wl.scores, wl.seq_lens, wl.page_table, wl.page_size, wl.k,
                                 max_seq_len=wl.max_seq_len, want_raw=True)[1].copy()


def _long_row(wl):
    eff = np.clip(wl.seq_lens, 0, wl.max_seq_len)
    return int(np.argmax(eff > wl.k + 10))


def test_rejects_a_lower_score_swapped_in():
    wl = _case("normal")
    raw = _oracle_raw(wl)
    b = _long_row(wl)
    L = int(min(wl.seq_lens[b], wl.max_seq_len))
    chosen = set(raw[b, :wl.k].tolist())
    worst = min((i for i in range(L) if i not in chosen), key=lambda i: wl.scores[b, i])
    raw[b, 0] = worst
    with pytest.raises(AssertionError):
        check_properties_all_rows(wl, raw)


def test_rejects_a_tie_broken_toward_the_larger_position():
    wl = _case("int")  # small integers: many ties at the k-th value
    raw = _oracle_raw(wl)
    eff = np.clip(wl.seq_lens, 0, wl.max_seq_len)
    for b in range(wl.batch):
        L = int(eff[b])
        if L <= wl.k:
            continue
        sel = raw[b, :wl.k]
        t = wl.scores[b, sel].min()
        later = [i for i in range(L) if wl.scores[b, i] == t and i not in set(sel.tolist())]
        if later:
            j = int(np.nonzero(wl.scores[b, sel] == t)[0][0])
            raw[b, j] = later[-1]
            break
    else:
        pytest.skip("no tie at the k-th value")
    with pytest.raises(AssertionError):
        check_properties_all_rows(wl, raw)


def test_rejects_a_repeated_position_and_one_past_the_row():
    wl = _case("normal")
    b = _long_row(wl)
    raw = _oracle_raw(wl)
    raw[b, 1] = raw[b, 0]
    with pytest.raises(AssertionError):
        check_properties_all_rows(wl, raw)
    raw = _oracle_raw(wl)
    raw[b, 0] = int(min(wl.seq_lens[b], wl.max_seq_len))
    with pytest.raises(AssertionError):
        check_properties_all_rows(wl, raw)


def test_bench_timed_output_check_accepts_the_oracle_and_rejects_a_swap():
    import bench

    for dist in ("normal", "int"):
        wl = workloads.random_case(seed=9300 + len(dist), batch=20, min_len=0, max_len=4000, k=200, page_size=16,
                                   dist=dist)
        out, raw, _ = oracle.topk_transform(wl.scores, wl.seq_lens, wl.page_table, wl.page_size, wl.k,
                                            max_seq_len=wl.max_seq_len, want_raw=True)
        assert bench.check_timed_rows(wl, out, count=20)["result"] == "ok"
    b = _long_row(wl)
    L = int(min(wl.seq_lens[b], wl.max_seq_len))
    chosen = set(raw[b, :wl.k].tolist())
    worst = min((i for i in range(L) if i not in chosen), key=lambda i: wl.scores[b, i])
    bad_raw = raw.copy()
    bad_raw[b, 0] = worst
    bad_out = oracle.page_transform(bad_raw, wl.page_table, wl.page_size)
    with pytest.raises(AssertionError):
        bench.check_timed_rows(wl, bad_out, count=20)
