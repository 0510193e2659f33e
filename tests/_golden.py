"""Reader for the hand-written golden fixtures under tests/golden/."""
import os
from collections import defaultdict

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    """{section: {rank: [ints]}} from tests/golden/<name>."""
    out = defaultdict(dict)
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, vals = line.split(":", 1)
            section, rank = head.split()
            out[section][int(rank)] = [int(v) for v in vals.split()]
    return dict(out)
