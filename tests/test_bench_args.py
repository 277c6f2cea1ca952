"""bench.py's --tuning option (CPU): names are checked against the library's
tuning struct, values are integers."""
from __future__ import annotations

import pytest

import bench


def test_parse_tuning_accepts_struct_fields():
    assert bench.parse_tuning("") == {}
    assert bench.parse_tuning("warp_rows=1, cluster_size=8") == {"warp_rows": 1, "cluster_size": 8}


@pytest.mark.parametrize("spec", ["warp_rows", "no_such_knob=1", "=3"])
def test_parse_tuning_rejects_unknown_or_malformed(spec):
    with pytest.raises(ValueError):
        bench.parse_tuning(spec)


def test_parse_tuning_rejects_non_integer_values():
    with pytest.raises(ValueError):
        bench.parse_tuning("warp_rows=yes")
