"""Readers for the hand-derived fixtures in tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _expand(field: str, conv):
    out = []
    for tok in field.split(","):
        tok = tok.strip()
        if "*" in tok:
            v, k = tok.split("*")
            out += [conv(v)] * int(k)
        else:
            out.append(conv(tok))
    return out


def q8_0_blocks():
    """[(name, x fp32[32], codes int8[32], scale_bits)]"""
    res = []
    with open(os.path.join(GOLDEN, "q8_0_closed_form.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, xs, qs, sc = [p.strip() for p in line.split("|")]
            x = np.array(_expand(xs, float), dtype=np.float32)
            q = np.array(_expand(qs, int), dtype=np.int8)
            assert x.size == 32 and q.size == 32, name
            res.append((name, x, q, int(sc, 16)))
    return res


def q4_0_blocks():
    """[(name, x fp32[32], codes u8[32], packed u8[16], scale_bits)]"""
    res = []
    with open(os.path.join(GOLDEN, "q4_0_closed_form.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, xs, qs, bs, sc = [p.strip() for p in line.split("|")]
            x = np.array(_expand(xs, float), dtype=np.float32)
            q = np.array(_expand(qs, int), dtype=np.uint8)
            b = np.array([int(t, 16) for t in bs.split()], dtype=np.uint8)
            assert x.size == 32 and q.size == 32 and b.size == 16, name
            res.append((name, x, q, b, int(sc, 16)))
    return res


def hexfile(name: str) -> bytes:
    out = bytearray()
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                out += bytes(int(t, 16) for t in line.split())
    return bytes(out)
