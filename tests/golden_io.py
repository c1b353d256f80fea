"""Reader for the small text fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _value(v):
    v = v.strip()
    if v == "-":
        return np.zeros(0, dtype=np.int64)
    parts = v.split()
    vals = [int(x) for x in parts]
    return vals[0] if len(vals) == 1 else np.array(vals, dtype=np.int64)


def read_sections(name):
    """{section: {key: int | int array}} from a [section] / key = values file."""
    out = {}
    cur = None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("[") and line.endswith("]"):
                cur = out.setdefault(line[1:-1], {})
                continue
            key, val = line.split("=", 1)
            tgt = out.setdefault("", {}) if cur is None else cur
            tgt[key.strip()] = _value(val)
    return out


def as_array(v):
    return np.atleast_1d(np.asarray(v, dtype=np.int64))
