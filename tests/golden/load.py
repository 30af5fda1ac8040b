"""Reader for the text fixtures in this folder (each case cites its page and section)."""

import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def worked_examples(path: str = os.path.join(HERE, "worked_examples.txt")):
    """Returns a list of dicts with keys name, M, N, K, A, B, C (float32 arrays)."""
    cases = []
    cur = None
    with open(path, encoding="utf-8") as fh:
        for raw in fh:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0]}
            elif key == "dims":
                cur["M"], cur["N"], cur["K"] = (int(v) for v in vals)
            elif key in ("A", "B", "C"):
                cur[key] = np.array([float(v) for v in vals], dtype=np.float32)
            elif key == "end":
                cur["A"] = cur["A"].reshape(cur["M"], cur["N"])
                cur["B"] = cur["B"].reshape(cur["N"], cur["K"])
                cur["C"] = cur["C"].reshape(cur["M"], cur["K"])
                cases.append(cur)
                cur = None
            else:
                raise ValueError(f"bad fixture line: {raw!r}")
    return cases
