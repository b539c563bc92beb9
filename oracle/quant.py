"""Float64 reference of the FP8 (E4M3) row format of the gathered weights.

Test infrastructure: only tests, the smoke check and the benchmark use this
module.  It shares no code with the CUDA library.

The pages report results with quantised weights ("PowerInfer: Fast Large
Language Model Serving with a Consumer-grade GPU", egguo-blog reading report,
section 3.1, Finding 2: INT4 runs) without fixing a format; the library's
format is its own choice, defined here from first principles:

* E4M3 ("fn" variant: no infinities, one NaN pattern per sign): bit 7 sign,
  bits 6..3 exponent field E (bias 7), bits 2..0 mantissa M.  E = 0 encodes
  the subnormals M * 2^-9; E = 1..15 encodes (1 + M/8) * 2^(E-7), except
  E = 15, M = 7, which is NaN.  The largest finite magnitude is 448.
* Each stored row w (d values, fp16) gets a binary32 scale
  s = max_j |w_j| / 448 (s = 1 for an all-zero row) and codes
  q_j = E4M3(w_j / s): the binary32 quotient rounded to the nearest E4M3
  value, ties to the even mantissa, magnitudes above 448 saturated to 448.
* The row then stands for the values s * value(q_j).

Where binary32 arithmetic decides a code (the scale and the quotient), this
module performs the same binary32 operations, so its codes are the exact
expected bytes.
"""
from __future__ import annotations

from dataclasses import replace

import numpy as np

from oracle.ffn import OracleLayer

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """float64 value of each E4M3 code (NaN for the two NaN patterns)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = (c >> 7) & 1
    ef = (c >> 3) & 0xF
    mf = c & 7
    mag = np.where(ef == 0, mf * 2.0 ** -9, (1.0 + mf / 8.0) * np.ldexp(1.0, ef - 7))
    mag = np.where((ef == 15) & (mf == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def e4m3_encode(v) -> np.ndarray:
    """E4M3 code of each binary32 value v: round to nearest, ties to even,
    saturating to +-448.  (No NaN inputs are expected.)"""
    v = np.asarray(v, dtype=np.float32)
    sign = np.signbit(v)
    a = np.minimum(np.abs(v).astype(np.float64), E4M3_MAX)
    # the quantum of the binade holding a: 2^(e-3) with 2^e <= a < 2^(e+1);
    # below the smallest normal (2^-6) the quantum stays 2^-9 (subnormals)
    _, E = np.frexp(np.where(a > 0, a, 1.0))
    e = np.maximum(E - 1, -6)
    quantum = np.ldexp(1.0, e - 3)
    val = np.round(a / quantum) * quantum            # numpy rounds halves to even
    # encode the rounded magnitude (it may have moved up one binade)
    code = np.zeros(v.shape, dtype=np.int64)
    sub = val < 2.0 ** -6
    code = np.where(sub, np.round(val / 2.0 ** -9).astype(np.int64), code)
    _, Ev = np.frexp(np.where(val > 0, val, 1.0))
    ev = Ev - 1
    mant = np.round((val / np.ldexp(1.0, ev) - 1.0) * 8.0).astype(np.int64)
    code = np.where(sub, code, ((ev + 7) << 3) | mant)
    return (code | (sign.astype(np.int64) << 7)).astype(np.uint8)


def quantize_rows(W16) -> tuple:
    """(codes uint8 [n, d], scales float32 [n]) of the rows of W16 [n, d] fp16."""
    W = np.asarray(W16).astype(np.float32)
    amax = np.abs(W).max(axis=1)
    s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    q = (W / s[:, None]).astype(np.float32)           # binary32 quotient, correctly rounded
    return e4m3_encode(q), s


def dequantize_rows(codes, scales) -> np.ndarray:
    """float64 [n, d]: row i is scales[i] * value(codes[i])."""
    return np.asarray(scales, dtype=np.float64)[:, None] * e4m3_decode(codes)


def fp8_rows(L: OracleLayer) -> dict:
    """Codes and scales of the three gathered matrices of L, row by row as
    the library stores them: W_up, W_gate (ReGLU) and W_down^T."""
    out = {"up": quantize_rows(L.W_up), "down": quantize_rows(np.asarray(L.W_down).T)}
    if L.W_gate is not None:
        out["gate"] = quantize_rows(L.W_gate)
    return out


def fp8_layer(L: OracleLayer) -> OracleLayer:
    """The layer whose up / gate / down weights are the FP8 rows' values
    (predictor, biases unchanged): the FFN an FP8 layer computes."""
    q = fp8_rows(L)
    return replace(
        L,
        W_up=dequantize_rows(*q["up"]),
        W_gate=None if L.W_gate is None else dequantize_rows(*q["gate"]),
        W_down=dequantize_rows(*q["down"]).T.copy(),
    )
