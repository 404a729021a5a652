"""Reader of the hand-derived text fixtures under tests/golden/.

Format: '#' starts a comment; every other non-empty line is
`name: v1 v2 ...`.  Values are returned as numpy arrays (float64, or int64
when every value is an integer literal); one-element arrays become scalars.
"""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, vals = line.split(":", 1)
            toks = vals.split()
            if all(t.lstrip("-").isdigit() for t in toks):
                arr = np.array([int(t) for t in toks], dtype=np.int64)
            else:
                arr = np.array([float(t) for t in toks], dtype=np.float64)
            out[key.strip()] = arr[0] if arr.size == 1 else arr
    return out
