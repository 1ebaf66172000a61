"""Pins for the oracle's OCP FP8 E4M3 codec (CPU only).

The codec is written from the OCP 8-bit floating point definition of E4M3
(bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN, max 448).  It is
pinned by: an exhaustive round trip over every code, the midpoint rule between
every pair of neighbours, the spec's landmark values, saturation, and a
comparison with torch's own float8_e4m3fn conversion (a library routine,
called) over a wide sample of in-range f32 values.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _non_nan_codes():
    return [c for c in range(256) if (c & 0x7F) != 0x7F]


def test_landmark_values():
    # values fixed by the E4M3 definition
    assert oracle.e4m3_decode(0x00) == 0.0
    assert math.copysign(1.0, oracle.e4m3_decode(0x80)) == -1.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9          # smallest subnormal
    assert oracle.e4m3_decode(0x07) == 7 * 2.0 ** -9       # largest subnormal
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6           # smallest normal
    assert oracle.e4m3_decode(0x38) == 1.0                 # exponent field 7 = bias
    assert oracle.e4m3_decode(0x7E) == 448.0               # largest finite
    assert oracle.e4m3_decode(0xFE) == -448.0
    assert math.isnan(oracle.e4m3_decode(0x7F))
    assert math.isnan(oracle.e4m3_decode(0xFF))


def test_decode_matches_torch_bitcast():
    # torch's float8_e4m3fn bit cast is an independent decoder
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = oracle.e4m3_decode_table()
    both_nan = np.isnan(ref) & np.isnan(mine)
    assert np.all(both_nan | (ref == mine))


def test_round_trip_all_codes():
    for c in _non_nan_codes():
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c, hex(c)


def test_midpoints_round_to_even_code():
    tab = oracle.e4m3_decode_table()
    for c in range(0, 126):
        lo, hi = tab[c], tab[c + 1]
        mid = (lo + hi) / 2  # exactly representable in f32 (4 mantissa bits)
        assert np.float32(mid) == mid
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == want, (c, mid)
        assert oracle.e4m3_encode(-mid) == 0x80 | want
        # just off the midpoint goes to the nearer neighbour
        below = float(np.nextafter(np.float32(mid), np.float32(0)))
        above = float(np.nextafter(np.float32(mid), np.float32(1000)))
        assert oracle.e4m3_encode(below) == c
        assert oracle.e4m3_encode(above) == c + 1


def test_saturation_and_nan():
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(463.9) == 0x7E
    assert oracle.e4m3_encode(464.0) == 0x7E   # satfinite: never the NaN code
    assert oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(-1e30) == 0xFE
    assert oracle.e4m3_encode(float("inf")) == 0x7E
    assert oracle.e4m3_encode(float("nan")) == 0x7F
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(1e-30) == 0x00
    assert oracle.e4m3_encode(-1e-30) == 0x80


@pytest.mark.parametrize("seed", [0, 1])
def test_encode_matches_torch_cast(seed):
    rng = np.random.default_rng(seed)
    # log-uniform magnitudes from deep subnormal to the top of the range
    mag = np.exp(rng.uniform(math.log(2.0 ** -14), math.log(463.0), 20000))
    x = (mag * rng.choice([-1.0, 1.0], mag.size)).astype(np.float32)
    x = np.concatenate([x, rng.standard_normal(5000).astype(np.float32)])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = oracle.e4m3_encode_array(x)
    bad = np.nonzero(ref != mine)[0]
    assert bad.size == 0, (x[bad[:5]], ref[bad[:5]], mine[bad[:5]])
