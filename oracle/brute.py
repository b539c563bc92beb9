"""Pure-Python brute force of the same path, for tiny layers only.

Test infrastructure.  Plain nested loops over Python floats (binary64), no
numpy: an independent restatement used to check ``oracle.ffn`` itself.
Method: "PowerInfer" (egguo-blog reading report), section 2.3, core modules 3
(predictor) and 4 (neuron-aware operators).
"""
from __future__ import annotations

import math


def _rows(a):
    if hasattr(a, "tolist"):
        a = a.tolist()
    return [[float(v) for v in r] for r in a]


def _vec(a):
    if hasattr(a, "tolist"):
        a = a.tolist()
    return [float(v) for v in a]


def forward(layer: dict, x) -> dict:
    """layer: dict with act, W_up, W_gate, b, W_down, W_p1, W_p2, c_p (lists
    or arrays); x: [B][d].  Returns mask, S (union, ascending) and y."""
    X = _rows(x)
    W1, W2 = _rows(layer["W_p1"]), _rows(layer["W_p2"])
    Wu, Wd = _rows(layer["W_up"]), _rows(layer["W_down"])
    Wg = _rows(layer["W_gate"]) if layer.get("W_gate") is not None else None
    b = _vec(layer["b"])
    ffn, r, d = len(Wu), len(W1), len(Wu[0])
    c = _vec(layer["c_p"]) if layer.get("c_p") is not None else [0.0] * ffn

    masks = []
    for xb in X:
        h = []
        for k in range(r):
            s = 0.0
            for j in range(d):
                s += W1[k][j] * xb[j]
            h.append(s if s > 0.0 else 0.0)
        m = []
        for i in range(ffn):
            s = c[i]
            for k in range(r):
                s += W2[i][k] * h[k]
            m.append(s > 0.0)
        masks.append(m)

    S = [i for i in range(ffn) if any(m[i] for m in masks)]

    ys = []
    for xb in X:
        y = [0.0] * d
        for i in S:
            z = b[i]
            if layer["act"] == "relu":
                for j in range(d):
                    z += Wu[i][j] * xb[j]
                a = z if z > 0.0 else 0.0
            else:
                for j in range(d):
                    z += Wg[i][j] * xb[j]
                u = 0.0
                for j in range(d):
                    u += Wu[i][j] * xb[j]
                if layer["act"] == "reglu":
                    g = z if z > 0.0 else 0.0
                elif z >= 0.0:                      # SiLU z / (1 + e^-z), written per sign
                    g = z / (1.0 + math.exp(-z))
                else:
                    e = math.exp(z)
                    g = z * e / (1.0 + e)
                a = g * u
            for j in range(d):
                y[j] += a * Wd[j][i]
        ys.append(y)
    return dict(mask=masks, S=S, y=ys)
