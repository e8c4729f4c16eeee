"""Readers for the small text fixtures under tests/golden/."""
import os

_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_kv(name):
    out = {}
    with open(os.path.join(_DIR, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = v.split()
    return out


def shapes(name, key):
    return [tuple(int(t) for t in s.split("x")) for s in read_kv(name)[key]]
