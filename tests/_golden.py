"""Reader for the hand-worked fixtures in tests/golden/ (``key: values`` lines, ``#`` comments)."""

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(":")
            toks = rest.split()
            if len(toks) == 1 and not toks[0].startswith("0x"):
                try:
                    out[key.strip()] = float(toks[0])
                except ValueError:
                    out[key.strip()] = toks[0]
                continue
            if toks and toks[0].startswith("0x"):
                out[key.strip()] = np.array([int(t, 16) for t in toks], dtype=np.uint8)
            else:
                out[key.strip()] = np.array([float(t) for t in toks], dtype=np.float64)
    return out
