"""Reader for the hand-derived worked examples under tests/golden/."""
from fractions import Fraction
import os

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_case(name):
    """Returns a dict: T, heads, kv_heads, c, q, k, vT (binary16) and the expected
    entries o[(h, i, e)] = Fraction, lse_arg[(h, i)] = Fraction (LSE = log2 of it)."""
    T = heads = kv = None
    c = None
    entries = {"q": [], "k": [], "v": []}
    o, lse = {}, {}
    with open(os.path.join(GOLDEN_DIR, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "shape":
                T, heads, kv = map(int, tok[1:4])
            elif tok[0] == "c":
                c = float(tok[1])
            elif tok[0] in entries:
                a, b, e = map(int, tok[1:4])
                entries[tok[0]].append((a, b, e, float(tok[4])))
            elif tok[0] == "o":
                h, i, e = map(int, tok[1:4])
                o[(h, i, e)] = Fraction(tok[4])
            elif tok[0] == "lse":
                h, i = map(int, tok[1:3])
                lse[(h, i)] = Fraction(tok[3])
            else:
                raise ValueError(f"unknown golden line: {line}")
    q = np.zeros((heads, T, 64), np.float16)
    k = np.zeros((kv, T, 64), np.float16)
    v = np.zeros((kv, T, 64), np.float16)
    for a, b, e, x in entries["q"]:
        q[a, b, e] = x
    for a, b, e, x in entries["k"]:
        k[a, b, e] = x
    for a, b, e, x in entries["v"]:
        v[a, b, e] = x
    vT = np.ascontiguousarray(v.transpose(0, 2, 1))
    return dict(T=T, heads=heads, kv_heads=kv, c=c, q=q, k=k, vT=vT, o=o, lse=lse)


def load_constants(name="scale_constant.txt"):
    out = {}
    with open(os.path.join(GOLDEN_DIR, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, val = line.split()
                out[key] = int(val, 0)
    return out
