"""Pins of the FP8 (E4M3) KV-cache oracle (oracle/kvquant.py): hand values of
the OCP E4M3 format, its value grid (monotone codes, 8 values per binade at a
spacing of 2^-3 of the binade, subnormals m 2^-9, largest 448, NaN only at
S.1111.111), the per-(head, 128-row block) power-of-two scales against a
plain loop, and a round trip through the independent encoder of synth/."""
import math

import numpy as np

import oracle
import synth


def test_hand_values():
    v = oracle.e4m3_value
    assert v(0x00) == 0.0 and math.copysign(1.0, v(0x80)) == -1.0
    assert v(0x38) == 1.0 and v(0x40) == 2.0 and v(0x3C) == 1.5 and v(0xB8) == -1.0
    assert v(0x7E) == 448.0 and v(0xFE) == -448.0
    assert v(0x01) == 2.0 ** -9 and v(0x07) == 7 * 2.0 ** -9 and v(0x08) == 2.0 ** -6
    assert math.isnan(v(0x7F)) and math.isnan(v(0xFF))
    assert v(0x78) == 256.0 and v(0x77) == 240.0


def test_value_grid():
    pos = [oracle.e4m3_value(b) for b in range(0x7F)]
    assert all(a < b for a, b in zip(pos, pos[1:]))                          # codes are monotone
    assert all(oracle.e4m3_value(b | 0x80) == -oracle.e4m3_value(b) for b in range(1, 0x7F))
    for k in range(-6, 9):                                                    # binades [2^k, 2^(k+1))
        vals = [x for x in pos if 2.0 ** k <= x < 2.0 ** (k + 1)]
        assert len(vals) == (8 if k < 8 else 7)                                # the top binade ends at 448
        assert all(abs((b - a) - 2.0 ** (k - 3)) < 1e-18 for a, b in zip(vals, vals[1:]))
    sub = [x for x in pos if 0 < x < 2.0 ** -6]
    assert sub == [m * 2.0 ** -9 for m in range(1, 8)]


def test_dequantize_block_scales_by_loop():
    g = synth.rng(5, 1)
    q = g.integers(0, 256, size=(2, 300, 8)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x12                                              # no NaN codes
    e = g.integers(-8, 4, size=(2, 3)).astype(np.int8)
    got = oracle.dequantize_kv(q, e)
    for h in range(2):
        for s in range(300):
            for d in range(8):
                assert got[h, s, d] == oracle.e4m3_value(q[h, s, d]) * 2.0 ** int(e[h, s // 128])


def test_round_trip_through_the_encoder():
    """synth's encoder (nearest value, ties to the even mantissa) and the
    oracle's decoder are written apart; x -> bytes -> value is within half a
    grid step of x, the block's largest |x| maps to at most 448, and exactly
    representable values come back unchanged."""
    x = synth.rng(5, 2).standard_normal((2, 260, 16)) * 3.0
    q, e = synth.quantize_kv_e4m3(x)
    d = oracle.dequantize_kv(q, e)
    for h in range(2):
        for b in range(3):
            blk = slice(128 * b, 128 * (b + 1))
            s = 2.0 ** int(e[h, b])
            assert np.abs(x[h, blk]).max() / s <= 448.0
            step = np.where(np.abs(x[h, blk]) / s < 2.0 ** -6, 2.0 ** -9,
                            2.0 ** (np.floor(np.log2(np.maximum(np.abs(x[h, blk]) / s, 2.0 ** -6))) - 3))
            assert (np.abs(d[h, blk] - x[h, blk]) <= 0.5 * step * s * (1 + 1e-12)).all()
    exact = np.array([[[1.0, -1.5, 448.0, 2.0 ** -9, 0.0, -240.0, 3.25, 0.875]]])
    q, e = synth.quantize_kv_e4m3(exact)
    assert int(e[0, 0]) == 0 and np.array_equal(oracle.dequantize_kv(q, e), exact)
