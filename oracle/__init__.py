"""CPU oracle for the top-k + page-table transform (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg import this package.  The CUDA library and its Python binding never do.
"""
from .oracle import (  # noqa: F401
    FLAG_SEQ_CLAMPED,
    FLAG_SEQ_NEGATIVE,
    build,
    load,
    page_transform,
    plan_classify,
    topk_transform,
)
