"""Reader for the hand-worked fixtures under tests/golden/ (text, no arithmetic)."""
from __future__ import annotations

import os

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _tokens(text: str):
    out = []
    for tok in text.split():
        if "*" in tok:
            v, n = tok.split("*")
            out.extend([v] * int(n))
        else:
            out.append(tok)
    return out


def _num(tok: str) -> float:
    t = tok.lower()
    if t.startswith("0x") or t.startswith("-0x"):
        return float.fromhex(t)
    return float(t)


def _rows(text: str, conv):
    return [[conv(t) for t in _tokens(r)] for r in text.split(";")]


def load(name: str) -> dict:
    """{case name: case dict} of one fixture file."""
    cases, cur = {}, None
    with open(os.path.join(GOLDEN_DIR, name)) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("["):
                cur = line.strip("[]")
                cases[cur] = {}
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            cases[cur][key] = val
    out = {}
    for cname, c in cases.items():
        bits, N, K = int(c["codec"]), int(c["N"]), int(c["K"])
        rb = (K * bits + 7) // 8
        packed = np.array([int(t, 16) for t in _tokens(c["bytes"])], np.uint8).reshape(N, rb)
        G = (K + 63) // 64
        scales = np.array([int(t, 16) for t in _tokens(c["scales"])], np.uint16).reshape(N, G)
        x = np.array(_rows(c["x"], lambda t: int(t, 16)), np.uint16)
        y = np.array(_rows(c["y"], _num), np.float64)
        a = np.array(_rows(c["a"], _num), np.float64)
        T = x.shape[0]
        assert x.shape == (T, K) and y.shape == (T, N) and a.shape == (T, N), cname
        out[cname] = dict(bits=bits, N=N, K=K, packed=packed, scales=scales, x=x, y=y, a=a)
    return out
