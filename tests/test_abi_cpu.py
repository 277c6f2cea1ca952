"""Host-only checks of the C ABI (no GPU needed, no compute calls): the library
loads, exports every function the header declares, and rejects bad arguments
on the host before any CUDA call."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from sparse_attention_indexer_uint32_gb300 import build as build_mod

HEADER = os.path.join(build_mod.ROOT, "include", "topkidx.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    from sparse_attention_indexer_uint32_gb300 import _lib

    return _lib


def declared_functions() -> list[str]:
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:[A-Za-z_][\w\s\*]*?)\b(topk_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_documented_entry_points():
    names = declared_functions()
    for required in ("topk_plan", "topk_transform", "topk_plan_workspace_bytes", "topk_page_transform",
                     "topk_key_map", "topk_read_flags", "topk_status_string", "topk_get_tuning",
                     "topk_set_tuning", "topk_last_error_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    cdll = lib.library()
    for name in declared_functions():
        assert hasattr(cdll, name), f"{name} declared in topkidx.h but not exported"
    assert set(declared_functions()) == set(lib.EXPORTED)


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert isinstance(lib.topk_status_string(code), str) and lib.topk_status_string(code)
    assert lib.topk_status_string(0) == "ok"
    assert lib.topk_status_string(99) == "unknown status"
    assert lib.topk_last_error_string() == ""  # no CUDA call has failed on this thread


def test_workspace_bytes(lib):
    assert lib.topk_plan_workspace_bytes(0) == 0
    assert lib.topk_plan_workspace_bytes(-3) == 0
    for b in (1, 7, 128, 8192):
        n = lib.topk_plan_workspace_bytes(b)
        assert n >= 64 + 8 * b and n % 256 == 0


def test_tuning_roundtrip_and_validation(lib):
    old = lib.topk_get_tuning()
    try:
        t = lib.topk_tuning_t(**old.as_dict())
        t.cluster_size = 4
        lib.topk_set_tuning(t)
        assert lib.topk_get_tuning().cluster_size == 4
        assert old.wait_limit_us == 0  # default: 2 s
        t.wait_limit_us = 1
        lib.topk_set_tuning(t)
        assert lib.topk_get_tuning().wait_limit_us == 1
        for field, bad in (("cluster_size", 5), ("candidate_capacity", 100), ("samples", 33),
                           ("long_threshold", -1), ("gate_fill_percent", 101), ("gate_fill_percent", -1),
                           ("single_block_threads", 128), ("single_block_copy_bytes", 4096), ("single_block_stages", 1),
                           ("single_block_stages", 9), ("gate_refresh_tiles", -1), ("gate_refresh_tiles", 65),
                           ("warp_rows", 3), ("warp_rows", -1), ("long_threshold_large_batch", -1),
                           ("large_batch_min", -1), ("warp_batch_min", -1), ("stream_batch_min", -1), ("wait_limit_us", -1),
                           ("wait_limit_us", 60000001), ("single_block_kernel", -1), ("single_block_kernel", 4),
                           ("split_rows", 3), ("split_segment", 2048), ("split_segment", 12288),
                           ("split_full_resolve", 2)):
            t2 = lib.topk_tuning_t(**old.as_dict())
            setattr(t2, field, bad)
            with pytest.raises(lib.TopkError) as e:
                lib.topk_set_tuning(t2)
            assert e.value.status == lib.TOPK_EINVAL
    finally:
        lib.topk_set_tuning(old)
    assert lib.topk_get_tuning().as_dict() == old.as_dict()


def test_host_side_argument_checks_return_before_any_launch(lib):
    """Fake (never dereferenced) pointers: the checks run before any CUDA call."""
    c = lib.library()
    fake = 1 << 20  # 16-byte aligned, never touched
    ok = dict(scores=fake, row_stride=64, seq_lens=fake, batch=2, max_seq_len=64, page_table=fake, pt_stride=1,
              page_size=64, k=8, out=fake, raw=None, ws=fake, stream=None)

    def call(**over):
        a = dict(ok)
        a.update(over)
        return c.topk_transform(a["scores"], a["row_stride"], a["seq_lens"], a["batch"], a["max_seq_len"],
                                a["page_table"], a["pt_stride"], a["page_size"], a["k"], a["out"], a["raw"],
                                a["ws"], a["stream"])

    assert call(k=0) == lib.TOPK_EINVAL
    assert call(k=2049) == lib.TOPK_EINVAL
    assert call(page_size=48) == lib.TOPK_EINVAL
    assert call(page_size=0) == lib.TOPK_EINVAL
    assert call(batch=0) == lib.TOPK_EINVAL
    assert call(max_seq_len=-1) == lib.TOPK_EINVAL
    assert call(row_stride=60, max_seq_len=64) == lib.TOPK_EINVAL
    assert call(pt_stride=0) == lib.TOPK_EINVAL
    assert call(scores=None) == lib.TOPK_EINVAL
    assert call(ws=None) == lib.TOPK_EINVAL
    assert call(scores=fake + 4) == lib.TOPK_EALIGN
    assert call(row_stride=66, max_seq_len=64) == lib.TOPK_EALIGN
    assert call(ws=fake + 8) == lib.TOPK_EALIGN
    assert call(out=fake + 2) == lib.TOPK_EALIGN
    # plan
    assert c.topk_plan(fake, 0, 10, fake, 4096, None) == lib.TOPK_EINVAL
    assert c.topk_plan(fake, 4, -1, fake, 4096, None) == lib.TOPK_EINVAL
    assert c.topk_plan(fake, 1000, 10, fake, 64, None) == lib.TOPK_ENOSPACE
    assert c.topk_plan(fake, 4, 10, fake + 4, lib.topk_plan_workspace_bytes(4), None) == lib.TOPK_EALIGN
    # page transform / key map
    assert c.topk_page_transform(fake, 0, 4, fake, 1, 64, fake, None) == lib.TOPK_EINVAL
    assert c.topk_page_transform(fake, 2, 4, fake, 1, 63, fake, None) == lib.TOPK_EINVAL
    assert c.topk_key_map(fake, -1, fake, None) == lib.TOPK_EINVAL
    assert c.topk_key_map(fake + 2, 8, fake, None) == lib.TOPK_EALIGN
    # launch-count query
    assert c.topk_transform_launches(0, 64, 8) == lib.TOPK_EINVAL
    assert c.topk_transform_launches(4, -1, 8) == lib.TOPK_EINVAL
    assert c.topk_transform_launches(4, 64, 2049) == lib.TOPK_EINVAL
    flags = ctypes.c_uint32(0)
    assert c.topk_read_flags(None, ctypes.byref(flags), 0, None) == lib.TOPK_EINVAL
