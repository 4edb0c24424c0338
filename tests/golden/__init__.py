"""Readers for the cited text fixtures in this folder."""
from __future__ import annotations

from fractions import Fraction
from pathlib import Path

HERE = Path(__file__).resolve().parent


def read_fixture(name: str) -> dict:
    """Parse `key = v1 v2 ...` lines; repeated keys collect into lists of rows."""
    out: dict = {}
    for line in (HERE / name).read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, val = line.partition("=")
        key = key.strip()
        row = [Fraction(tok) for tok in val.split()]
        if key in out:
            if not isinstance(out[key][0], list):
                out[key] = [out[key]]
            out[key].append(row)
        else:
            out[key] = row
    return out
