"""Pins for the oracle's number formats: e4m3 and bf16.

The oracle's e4m3 encoder/decoder is written from the OCP 8-bit floating point
definition (E4M3: bias 7, 3 mantissa bits, max 448, no infinities).  These
tests hold it against torch's float8_e4m3fn conversion (a library routine) for
every code and for values in range, and against the definition for
saturation, ties and signed zero.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def test_decode_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c], (c, got, ref[c])
            assert math.copysign(1.0, got) == math.copysign(1.0, ref[c]), c


def test_encode_roundtrips_every_finite_code():
    for c in range(256):
        x = oracle.e4m3_decode(c)
        if math.isnan(x):
            continue
        assert oracle.e4m3_encode(np.float32(x)) == c, c


def test_encode_matches_torch_on_values_in_range():
    rng = np.random.default_rng(123)
    # random magnitudes over the whole exponent range, plus every midpoint
    # between neighbouring codes (ties) and their float32 neighbours
    xs = [rng.standard_normal(20000).astype(np.float32) * np.float32(s)
          for s in (1e-3, 1e-1, 1.0, 10.0, 100.0)]
    finite = sorted({oracle.e4m3_decode(c) for c in range(0, 0x7F)})
    mids = [(a + b) / 2 for a, b in zip(finite[:-1], finite[1:])]
    mids = np.array(mids + [-m for m in mids], np.float32)
    xs.append(mids)
    xs.append(np.nextafter(mids, np.float32(np.inf)))
    xs.append(np.nextafter(mids, np.float32(-np.inf)))
    x = np.concatenate(xs)
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(v) for v in x], np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(x[i]), int(got[i]), int(ref[i])) for i in bad[:10]]


def test_encode_saturates_and_rounds_to_even_by_definition():
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(470.0) == 0x7E          # would round to 480: saturate
    assert oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(float("inf")) == 0x7E
    assert oracle.e4m3_encode(-1e30) == 0xFE
    # tie between 1.0 (mantissa 000) and 1.125 (001): even mantissa wins
    assert oracle.e4m3_encode(1.0625) == oracle.e4m3_encode(1.0)
    # tie between 1.125 (001) and 1.25 (010): 1.25
    assert oracle.e4m3_decode(oracle.e4m3_encode(1.1875)) == 1.25
    # smallest subnormal 2^-9; half of it ties to 0 (even)
    assert oracle.e4m3_encode(2.0 ** -9) == 0x01
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00
    assert oracle.e4m3_encode(1.5 * 2.0 ** -10) == 0x01
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(0.0) == 0x00


def test_bf16_rounding_of_inputs_is_round_to_nearest_even():
    from workloads import bf16_bits_to_f32, to_bf16_bits
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.1415926], np.float32)
    b = to_bf16_bits(x)
    back = bf16_bits_to_f32(b)
    assert back[0] == 1.0
    assert back[1] == 1.0                     # tie -> even mantissa
    assert back[2] == 1.0 + 4 * 2 ** -8       # tie -> even (up)
    assert back[3] == -2.5
    assert abs(back[4] - 3.1415926) < 2 ** -7 * 4
