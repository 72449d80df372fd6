"""Pins for the oracle's E4M3 codec: the format definition, hand-worked points,
exhaustive round trip, and torch's own float8_e4m3fn cast as an independent
library routine."""
import math

import numpy as np
import pytest
import torch

from conftest import read_golden
from oracle import e4m3


def test_decode_table_structure():
    t = e4m3.DECODE_TABLE
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.isnan(t).sum() == 2
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0
    assert t[0x00] == 0.0 and t[0x80] == 0.0 and math.copysign(1, t[0x80]) == -1
    assert t[0x01] == 2.0 ** -9 and t[0x08] == 2.0 ** -6 and t[0x38] == 1.0
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)          # codes ordered by magnitude
    assert np.array_equal(t[0x80:0xFF], -pos)


def test_roundtrip_all_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = e4m3.decode(codes).astype(np.float32)
    assert np.array_equal(e4m3.encode(vals), codes)


def test_golden_points():
    g = read_golden("e4m3_points.txt")
    for expr, code, *_ in g["point"]:
        v = eval(expr, {"__builtins__": {}})
        assert int(e4m3.encode(np.float32(v))) == int(code, 16), expr


def test_midpoints_tie_to_even():
    pos = e4m3.DECODE_TABLE[:0x7F]
    for c in range(0x7E):
        mid = np.float32((pos[c] + pos[c + 1]) / 2)
        if float(mid) != (pos[c] + pos[c + 1]) / 2:
            continue
        want = c if c % 2 == 0 else c + 1
        assert int(e4m3.encode(mid)) == want
        assert int(e4m3.encode(-mid)) == want | 0x80


def test_matches_torch_cast_in_range():
    rng = np.random.default_rng(0)
    v = np.concatenate([
        rng.standard_normal(200_000).astype(np.float32) * 60,
        rng.uniform(-448, 448, 100_000).astype(np.float32),
        (rng.standard_normal(100_000) * 1e-3).astype(np.float32),
        np.ldexp(rng.uniform(-1, 1, 50_000), rng.integers(-14, -5, 50_000)).astype(np.float32),
    ])
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3.encode(v), ref)


def test_saturates_instead_of_nan():
    v = np.array([448.0, 464.0, 480.0, 1e30, np.inf, -np.inf], dtype=np.float32)
    assert list(e4m3.encode(v)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE]


def test_two_encoders_agree():
    rng = np.random.default_rng(9)
    v = np.concatenate([rng.standard_normal(300_000).astype(np.float32) * 100,
                        np.ldexp(rng.uniform(-1, 1, 100_000), rng.integers(-16, 10, 100_000)).astype(np.float32),
                        e4m3.DECODE_TABLE[:0x7F].astype(np.float32),
                        ((e4m3.DECODE_TABLE[:0x7E] + e4m3.DECODE_TABLE[1:0x7F]) / 2).astype(np.float32)])
    assert np.array_equal(e4m3.encode(v), e4m3.encode_by_search(v))
