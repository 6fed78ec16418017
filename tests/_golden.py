"""Reader for the small text fixtures under tests/golden/.

Format: '#' comment lines (the citation), then 'key: values' lines; a value
list is whitespace-separated numbers with ';' separating matrix rows.
"""

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            rows = [r.split() for r in val.split(";")]
            if len(rows) == 1:
                out[key.strip()] = rows[0]
            else:
                out[key.strip()] = rows
    return out


def matrix(rows):
    if rows and isinstance(rows[0], str):
        return np.array([float(v) for v in rows])
    return np.array([[float(v) for v in r] for r in rows])
