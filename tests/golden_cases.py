"""Parser for the hand-worked fixtures in ``tests/golden/hand_worked.txt``."""
from __future__ import annotations

import dataclasses
import os
import struct

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_worked.txt")


@dataclasses.dataclass
class GoldenCase:
    name: str
    cite: str
    k: int
    page_size: int
    seq_len: int
    max_seq_len: int
    scores: np.ndarray
    table: np.ndarray
    raw: list[int]
    pad: int
    out: list[int]


def _parse_scores(text: str, n: int) -> np.ndarray:
    toks = text.split()
    if toks and toks[0].startswith("fill:"):
        row = np.full(n, float(toks[0][5:]), dtype=np.float32)
        for t in toks[1:]:
            pos, val = t[3:].split("=")
            row[int(pos)] = float(val)
        return row
    vals = []
    for t in toks:
        if t.startswith("bits:"):
            vals.append(struct.unpack("<f", struct.pack("<I", int(t[5:], 16)))[0])
        else:
            vals.append(float(t))
    out = np.empty(len(vals), dtype=np.float32)
    for i, t in enumerate(toks):  # keep NaN payloads bit-exact
        if t.startswith("bits:"):
            out.view(np.uint32)[i] = int(t[5:], 16)
        else:
            out[i] = np.float32(vals[i])
    return out


def load_cases() -> list[GoldenCase]:
    cases = []
    block: dict[str, str] = {}
    with open(GOLDEN) as f:
        lines = [ln.rstrip("\n") for ln in f] + [""]
    for ln in lines:
        if ln.startswith("#"):
            continue
        if not ln.strip():
            if block:
                cases.append(_make(block))
                block = {}
            continue
        key, _, val = ln.partition(":")
        block[key.strip()] = val.strip()
    return cases


def _make(b: dict[str, str]) -> GoldenCase:
    seq_len = int(b["seq_len"])
    scores_len = len(b["scores"].split()) if not b["scores"].startswith("fill:") else max(seq_len, 1)
    scores = _parse_scores(b["scores"], scores_len)
    ints = lambda s: [int(t) for t in s.split()]  # noqa: E731
    return GoldenCase(
        name=b["case"], cite=b["cite"], k=int(b["k"]), page_size=int(b["page_size"]), seq_len=seq_len,
        max_seq_len=int(b.get("max_seq_len", len(scores))), scores=scores,
        table=np.array(ints(b["table"]), dtype=np.int32), raw=ints(b.get("raw", "")), pad=int(b["pad"]),
        out=ints(b.get("out", "")),
    )
