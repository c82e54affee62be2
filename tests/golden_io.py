"""Reader for the small text fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_fixture(name):
    meta, rows = {}, []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0].isalpha():
                vals = [float(x) if "." in x else int(x) for x in parts[1:]]
                meta[parts[0]] = vals[0] if len(vals) == 1 else vals
            else:
                rows.append([float(x) if "." in x else int(x) for x in parts])
    return meta, (np.asarray(rows) if rows else None)
