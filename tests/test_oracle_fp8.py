"""Pins of the oracle's FP8 (E4M3) row format against the format's definition,
hand-worked values, exhaustive round trips and an independent library cast."""
import numpy as np
import pytest
import torch

from oracle import ffn as O
from oracle import quant as Q
from workload import LayerSpec, make_layer, make_tokens


def test_decode_known_codes():
    # values fixed by the format: subnormal unit 2^-9, smallest normal 2^-6,
    # 1.0 at exponent field 7, largest finite 448 = 1.75 * 2^8
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x38: 1.0, 0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0,
             0x81: -(2.0 ** -9), 0xB8: -1.0, 0xFE: -448.0}
    got = Q.e4m3_decode(np.array(list(table), dtype=np.uint8))
    assert np.array_equal(got, np.array(list(table.values())))
    assert np.isnan(Q.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()
    neg0 = Q.e4m3_decode(np.array([0x80], dtype=np.uint8))[0]
    assert neg0 == 0.0 and np.signbit(neg0)


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = Q.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(Q.e4m3_encode(vals), codes)
    # 254 finite values, strictly increasing magnitude within each sign
    pos = Q.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0) and pos.max() == 448.0


def test_rounding_ties_go_to_even_and_saturate():
    cases = {1.0625: 0x38,        # halfway 1.0 / 1.125 -> even mantissa (1.0)
             1.1875: 0x3A,        # halfway 1.125 / 1.25 -> 1.25
             2.0 ** -10: 0x00,    # half the smallest subnormal -> 0
             3 * 2.0 ** -10: 0x02,
             15 * 2.0 ** -10: 0x08,   # halfway 7 * 2^-9 / 2^-6 -> 2^-6 (even)
             464.0: 0x7E,         # halfway 448 / (480, not a finite code) saturates
             1000.0: 0x7E, -1000.0: 0xFE, -0.0: 0x80}
    v = np.array(list(cases), dtype=np.float32)
    assert np.array_equal(Q.e4m3_encode(v), np.array(list(cases.values()), dtype=np.uint8))


def test_encode_matches_an_independent_cast():
    fp8 = getattr(torch, "float8_e4m3fn", None)
    if fp8 is None:
        pytest.skip("this torch has no float8_e4m3fn")
    g = np.random.default_rng(7)
    v = np.concatenate([g.uniform(-448, 448, 20000), g.normal(0, 1, 20000),
                        g.normal(0, 2.0 ** -7, 20000)]).astype(np.float32)
    ref = torch.from_numpy(v).to(fp8).view(torch.uint8).numpy()
    assert np.array_equal(Q.e4m3_encode(v), ref)


def test_quantize_rows_scale_rule_and_error():
    g = np.random.default_rng(3)
    W = (g.normal(0, 0.02, (64, 256))).astype(np.float16)
    W[5] = 0                                        # all-zero row: scale 1, codes 0
    codes, s = Q.quantize_rows(W)
    assert s.dtype == np.float32 and s[5] == 1.0 and not codes[5].any()
    amax = np.abs(W.astype(np.float32)).max(axis=1)
    nz = amax > 0
    assert np.array_equal(s[nz], (amax[nz] / np.float32(448)).astype(np.float32))
    # the largest element of each row lands on +-448 exactly
    rows = np.flatnonzero(nz)
    j = np.abs(W[rows].astype(np.float32)).argmax(axis=1)
    assert np.all((codes[rows, j] & 0x7F) == 0x7E)
    # rounding error: half a quantum, i.e. <= 2^-4 relative for normals and
    # <= 2^-10 * s below the smallest normal
    deq = Q.dequantize_rows(codes, s)
    w = W.astype(np.float64)
    err = np.abs(deq - w)
    bound = np.maximum(np.abs(w) * 2.0 ** -4, s.astype(np.float64)[:, None] * 2.0 ** -10)
    assert np.all(err <= bound * (1 + 1e-12))


def test_fp8_layer_is_the_ffn_of_the_dequantised_rows():
    spec = LayerSpec(d=64, ffn=96, rank=8, act="reglu", mean_f=0.3)
    t = make_layer(spec, 11, 0)
    L = O.OracleLayer.from_tensors(t)
    L8 = Q.fp8_layer(L)
    q = Q.fp8_rows(L)
    assert np.array_equal(L8.W_up, Q.dequantize_rows(*q["up"]))
    assert np.array_equal(L8.W_down.T, Q.dequantize_rows(*q["down"]))
    # predictor untouched; the FFN of the FP8 layer is within the rows'
    # rounding of the fp16 one
    assert L8.W_p1 is L.W_p1 and L8.W_p2 is L.W_p2
    x = make_tokens(64, 2, seed=4).numpy()
    y16 = O.dense_ffn(L, x)
    y8 = O.dense_ffn(L8, x)
    assert np.linalg.norm(y8 - y16) <= 0.1 * np.linalg.norm(y16)
    # quantising commutes with the storage permutation (row by row)
    perm = np.random.default_rng(1).permutation(96)
    Lp8 = Q.fp8_layer(O.permute_layer(L, perm))
    assert np.array_equal(Lp8.W_up, L8.W_up[perm])
    assert np.array_equal(Lp8.W_down, L8.W_down[:, perm])
