"""Reader of the hand-worked IBP examples under tests/golden/."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    d = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            d[key] = vals
    out = {}
    for k, v in d.items():
        if k in ("R", "C", "bits", "raw", "num", "den"):
            out[k] = int(v[0])
        elif k == "p":
            out[k] = [int(x) for x in v]
        else:
            out[k] = [int(x, 16) for x in v]
    return out


def names(prefix=""):
    return sorted(f for f in os.listdir(GOLDEN) if f.endswith(".txt") and f.startswith(prefix)
                  and f != "README.txt")
