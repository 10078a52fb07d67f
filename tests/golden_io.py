"""Readers for the hand-derived fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_fixture(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(":")
            out.setdefault(key.strip(), []).extend(rest.split())
    res = {}
    for key, toks in out.items():
        if key == "bytes":
            res[key] = np.array([int(t, 16) for t in toks], np.uint8)
        elif key == "values":
            res[key] = np.array([float(t) for t in toks], np.float64)
        else:
            res[key] = int(toks[0])
    return res


def same_values(a_bits, b_bits):
    """bf16 bit arrays hold the same values (+0 and -0 count as equal)."""
    a = np.asarray(a_bits, np.uint16).astype(np.uint32) << 16
    b = np.asarray(b_bits, np.uint16).astype(np.uint32) << 16
    return np.array_equal(a.view(np.float32), b.view(np.float32))
