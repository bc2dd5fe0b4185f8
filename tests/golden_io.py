"""Reader for the hand-expanded fixtures under tests/golden/.

A fixture is ``key = values`` lines; values are decimals, ``inf``/``-inf`` or
exact fractions such as ``18/5``.  Lines starting with ``#`` hold the citation
and the derivation.
"""

from __future__ import annotations

import glob
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

INT_KEYS = {"n", "d", "K", "T"}


def _num(tok: str) -> float:
    if tok in ("inf", "+inf"):
        return float("inf")
    if tok == "-inf":
        return float("-inf")
    return float(Fraction(tok))


def load(path: str) -> dict:
    out: dict = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition("=")
            key = key.strip()
            toks = rest.split()
            if key in INT_KEYS:
                out[key] = int(toks[0])
            else:
                out[key] = np.array([_num(t) for t in toks], dtype=np.float64)
    return out


def to_bf16_exact(values: np.ndarray) -> np.ndarray:
    """BF16 bits of values that BF16 holds exactly (asserted)."""
    f = np.asarray(values, np.float32)
    bits = f.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "fixture weight not exact in BF16"
    return (bits >> 16).astype(np.uint16)


def fixtures() -> list[str]:
    return sorted(glob.glob(os.path.join(GOLDEN, "hand_*.txt")))
