"""Reader for the small text fixtures under tests/golden/ (comments start with '#')."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read(name):
    """Returns {key: value}. ``key: a b c`` lines give 1-D arrays; ``key d0 d1 ...`` lines are
    followed by prod(d[:-1]) rows of d[-1] numbers and give an array of shape d."""
    with open(os.path.join(GOLDEN, name)) as f:
        lines = [ln.split("#", 1)[0].strip() for ln in f]
    lines = [ln for ln in lines if ln]
    out, i = {}, 0
    while i < len(lines):
        ln = lines[i]
        if ":" in ln:
            key, vals = ln.split(":", 1)
            toks = vals.split()
            try:
                out[key.strip()] = np.array([float(t) for t in toks])
            except ValueError:
                out[key.strip()] = toks
            i += 1
            continue
        toks = ln.split()
        try:
            shape = [int(t) for t in toks[1:]]
        except ValueError:
            shape = []
        if toks and shape:
            nrows = int(np.prod(shape[:-1])) if len(shape) > 1 else 1
            rows = [[float(t) for t in lines[i + 1 + r].split()] for r in range(nrows)]
            out[toks[0]] = np.array(rows).reshape(shape)
            i += 1 + nrows
            continue
        out.setdefault("_rows", []).append(toks)
        i += 1
    return out
