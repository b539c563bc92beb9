"""Reader for the hand-worked fixtures in this folder.

Format: ``name = v v v`` for vectors, ``name = v v ; v v`` for matrices
(rows separated by ``;``), ``#`` starts a comment line.
"""
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent


def load(name: str) -> dict:
    out = {}
    for line in (HERE / name).read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, val = (s.strip() for s in line.split("=", 1))
        if key == "act":
            out[key] = val
            continue
        rows = [r.split() for r in val.split(";")]
        arr = np.array([[float(v) for v in r] for r in rows], dtype=np.float64)
        out[key] = arr if len(rows) > 1 else arr[0]
    return out
