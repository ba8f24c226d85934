"""Reader for the hand-derived fixtures under tests/golden/ (``key: value`` lines)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = v.strip()
    return out


def hex_bytes(s: str) -> list:
    """'00 3C E4*3' -> [0x00, 0x3C, 0xE4, 0xE4, 0xE4]."""
    out = []
    for tok in s.split():
        if "*" in tok:
            v, n = tok.split("*")
            out += [int(v, 16)] * int(n)
        else:
            out.append(int(tok, 16))
    return out


def ints(s: str) -> list:
    return [int(t) for t in s.split()]


def floats(s: str) -> list:
    return [float(t) for t in s.split()]


def kv(s: str) -> dict:
    """'code=8 d=1400' -> {'code': '8', 'd': '1400'}"""
    return dict(t.split("=") for t in s.split())
