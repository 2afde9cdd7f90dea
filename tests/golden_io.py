"""Reader for the small text fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(":")
            rows = [r.split() for r in rest.split("|")]
            arr = np.array([[float(v) for v in r] for r in rows])
            if arr.shape[0] == 1:
                arr = arr[0]
                if arr.shape[0] == 1:
                    arr = arr[0]
            vals[key.strip()] = arr
    return vals
