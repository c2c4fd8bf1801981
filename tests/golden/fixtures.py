"""Reader for the small text fixtures in this folder (each file cites its page)."""
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def read_kv(name):
    out = {}
    with open(os.path.join(HERE, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            out[k] = v
    return out


def shape(s):
    return tuple(int(x) for x in s.split(","))
