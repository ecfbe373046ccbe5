"""Reader of the hand-derived fixtures in tests/golden/: `key = value` lines, `#` comments,
space-separated numbers, `;` between matrix rows, `pi/n` for exact angles."""

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    d = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split("=", 1)
                d[k.strip()] = v.strip()
    return d


def num(v: str):
    """A scalar angle (pi/n), a vector, or a matrix (rows split by ';')."""
    if v.startswith("pi/"):
        return math.pi / float(v[3:])
    rows = [[float(x) for x in r.split()] for r in v.split(";")]
    return np.array(rows[0] if len(rows) == 1 else rows, dtype=np.float64)


def scalar(v: str) -> float:
    x = num(v)
    return float(x) if np.ndim(x) == 0 else float(np.asarray(x).reshape(-1)[0])


ANGLES = (("t_pi_6", 6), ("t_pi_4", 4), ("t_pi_3", 3))
