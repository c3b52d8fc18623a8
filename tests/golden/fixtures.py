"""Readers for the hand-written golden fixtures in this folder."""

import os

HERE = os.path.dirname(os.path.abspath(__file__))


def _expand(tokens, conv):
    out = []
    for t in tokens:
        if "*" in t:
            v, n = t.rsplit("*", 1)
            out.extend([conv(v)] * int(n))
        else:
            out.append(conv(t))
    return out


def _num(t):
    t = t.strip()
    if t.lstrip("-").startswith("0x"):
        return float.fromhex(t)
    return float(t)


def load_blocks():
    """List of dicts: name, fmt, x (32 floats), scale (int), codes (32 ints)."""
    cases, cur = [], None
    with open(os.path.join(HERE, "mx_blocks.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"name": rest}
                cases.append(cur)
            elif key == "fmt":
                cur["fmt"] = rest
            elif key == "x":
                cur["x"] = _expand(rest.split(), _num)
            elif key == "scale":
                cur["scale"] = int(rest)
            elif key == "codes":
                cur["codes"] = _expand(rest.split(), lambda t: int(t, 16))
    for c in cases:
        assert len(c["x"]) == 32 and len(c["codes"]) == 32, c["name"]
    return cases


def load_e2m1_values():
    vals = {}
    with open(os.path.join(HERE, "e2m1_values.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            c, v = line.split()
            vals[int(c)] = float(v)
    return vals


def load_e2m1_packed():
    """List of dicts: name, x (32 floats), scale (int), packed (16 ints) --
    hand-derived E2M1 blocks with their packed code bytes."""
    cases, cur = [], None
    with open(os.path.join(HERE, "e2m1_packed.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"name": rest}
                cases.append(cur)
            elif key == "x":
                cur["x"] = _expand(rest.split(), _num)
            elif key == "scale":
                cur["scale"] = int(rest)
            elif key == "packed":
                cur["packed"] = _expand(rest.split(), lambda t: int(t, 16))
    for c in cases:
        assert len(c["x"]) == 32 and len(c["packed"]) == 16, c["name"]
    return cases
