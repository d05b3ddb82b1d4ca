"""Reader for the small text fixtures under tests/golden/ (key followed by values)."""
import os

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    out = {}
    with open(os.path.join(HERE, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = [float(v) if any(c in v for c in ".e") else int(v) for v in vals]
    return out
