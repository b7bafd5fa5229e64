"""Reader for the small text fixtures under tests/golden/ (key, then values per line)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read(name):
    """Return {key: [values...]} with repeated keys collected as lists of lists."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out.setdefault(key, []).append(vals)
    return out


def scalar(d, key, cast=int):
    return cast(d[key][0][0])
