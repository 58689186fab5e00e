"""Reads the fixtures under tests/golden/: '#' lines are the citation and
notes, every other line is `name value` (a number)."""
import os

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    vals = {}
    with open(os.path.join(GOLDEN_DIR, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split()
            vals[key] = float(val)
    return vals
