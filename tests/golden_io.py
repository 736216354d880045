"""Reader for the small text fixtures under tests/golden/ (the pages' printed values)."""
import math
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _num(tok):
    if tok == "ln3":
        return math.log(3.0)
    if tok in ("-inf", "inf"):
        return float(tok)
    return float(tok)


def load(name):
    """Return {key: [floats]} (or a list of lists for '|'-separated groups)."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(":")
            rest = rest.strip()
            if "|" in rest:
                out[key.strip()] = [[_num(t) for t in g.split()] for g in rest.split("|")]
            else:
                out[key.strip()] = [_num(t) for t in rest.split()]
    return out
