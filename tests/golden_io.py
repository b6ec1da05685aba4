"""Reader for the hand-worked fixtures under tests/golden/ ("key: values" lines, '#' comments)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            out[key.strip()] = val.split()
    return out


def floats(v):
    return [float(t) for t in v]


def hexbytes(v):
    return [int(t, 16) for t in v]
