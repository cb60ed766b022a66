"""Golden values printed by the pages (each file cites its source)."""
import os

_DIR = os.path.dirname(os.path.abspath(__file__))


def load_kv(name: str) -> dict:
    out = {}
    with open(os.path.join(_DIR, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split("=", 1)
            out[k.strip()] = v.strip()
    return out


def load_rows(name: str) -> list:
    rows = []
    with open(os.path.join(_DIR, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows
