"""Parser for the hand-worked block fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _pairs(field, conv):
    out = {}
    for tok in field.split():
        k, v = tok.split(":")
        out[int(k)] = conv(v)
    return out


def load_blocks(name):
    """Yield (case, values[32] float32, scale byte, {byte index: code}, {index: dequant})."""
    cases = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            case, vals, scale, codes, deq = [p.strip() for p in line.split("|")]
            x = np.zeros(32, np.float32)
            for i, v in _pairs(vals, float).items():
                x[i] = np.float32(v)
            cases.append((case, x, int(scale, 16), _pairs(codes, lambda s: int(s, 16)),
                          _pairs(deq, float)))
    return cases
