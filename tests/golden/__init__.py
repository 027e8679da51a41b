"""Parser for the hand-worked fixtures in this folder."""

from __future__ import annotations

import dataclasses
import os
import struct

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def _value(tok: str) -> float:
    if tok.startswith("0x"):
        return struct.unpack("<f", struct.pack("<I", int(tok, 16)))[0]
    return float(tok)


@dataclasses.dataclass
class Case:
    name: str
    cites: str
    form: str
    k: int
    seq_lens: np.ndarray
    scores: np.ndarray
    expect: np.ndarray
    page_size: int = 64
    page_table: np.ndarray | None = None
    row_starts: np.ndarray | None = None
    expect_sorted: np.ndarray | None = None
    expect_values: np.ndarray | None = None


def load_cases(filename: str = "topk_cases.txt") -> list[Case]:
    with open(os.path.join(HERE, filename)) as f:
        lines = [ln.rstrip("\n") for ln in f]
    blocks, cur = [], []
    for ln in lines:
        if ln.startswith("#"):
            continue
        if not ln.strip():
            if cur:
                blocks.append(cur)
                cur = []
            continue
        cur.append(ln)
    if cur:
        blocks.append(cur)
    cases = []
    for blk in blocks:
        fields: dict[str, list[str]] = {}
        key = None
        for ln in blk:
            if ":" in ln and not ln[0].isdigit() and not ln[0] in "-.0123456789":
                key, _, rest = ln.partition(":")
                key = key.strip()
                fields[key] = [rest.strip()] if rest.strip() else []
            else:
                fields[key].append(ln.strip())
        rows = lambda k: [[t for t in r.split()] for r in fields[k]]
        form = fields["form"][0]
        scores_rows = [[_value(t) for t in r] for r in rows("scores")]
        if form == "ragged":
            scores = np.array(scores_rows[0], dtype=np.float32)
        else:
            scores = np.array(scores_rows, dtype=np.float32)
        case = Case(
            name=fields["case"][0],
            cites=fields.get("cites", [""])[0],
            form=form,
            k=int(fields["k"][0]),
            seq_lens=np.array([int(t) for t in fields["seq_lens"][0].split()], dtype=np.int32),
            scores=scores,
            expect=np.array([[int(t) for t in r] for r in rows("expect")], dtype=np.int32),
        )
        if "page_size" in fields:
            case.page_size = int(fields["page_size"][0])
        if "page_table" in fields:
            case.page_table = np.array([[int(t) for t in r] for r in rows("page_table")],
                                       dtype=np.int32)
        if "expect_sorted" in fields:
            case.expect_sorted = np.array([[int(t) for t in r] for r in rows("expect_sorted")],
                                          dtype=np.int32)
        if "expect_values" in fields:
            case.expect_values = np.array([[_value(t) for t in r] for r in rows("expect_values")],
                                          dtype=np.float32)
        if "row_starts" in fields:
            case.row_starts = np.array([int(t) for t in fields["row_starts"][0].split()],
                                       dtype=np.int32)
        cases.append(case)
    return cases
