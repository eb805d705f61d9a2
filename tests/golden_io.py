"""Parser of the hand-written metadata fixtures in tests/golden/meta_cases.txt."""
import os

import numpy as np

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _expand(tokens):
    out = []
    for t in tokens:
        if "*" in t:
            v, n = t.split("*")
            out.extend([int(v)] * int(n))
        else:
            out.append(int(t))
    return out


def load_meta_cases(fname="meta_cases.txt"):
    cases = {}
    cur = None
    with open(os.path.join(HERE, fname)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("[case"):
                cur = line[len("[case"):].strip(" ]")
                cases[cur] = {}
                continue
            key, *vals = line.split()
            cases[cur][key] = np.array(_expand(vals), dtype=np.int64)
    return cases
