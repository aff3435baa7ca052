"""Oracle pins: scalar decoders and encoders against hand-worked codes,
library decoders and brute force over the formats' definitions."""
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                yield line.split()


def test_hand_worked_decodes():
    fns = {"int4": O.int4_value, "int8": O.int8_value, "fp16": O.fp16_to_double,
           "e2m1": O.e2m1_to_double, "e4m3": O.e4m3_to_double}
    n = 0
    for fmt, code, value in _rows("format_decode.txt"):
        assert fns[fmt](int(code, 16)) == float(value), (fmt, code)
        n += 1
    assert n >= 25


def test_fp16_matches_numpy_everywhere():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    for b in range(0, 65536, 7):
        if not np.isfinite(ref[b]):
            with pytest.raises(ValueError):
                O.fp16_to_double(b)
            continue
        assert O.fp16_to_double(b) == ref[b]


def test_e4m3_matches_torch_float8_everywhere():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    for b in range(256):
        if b in (0x7F, 0xFF):
            with pytest.raises(ValueError):
                O.e4m3_to_double(b)
            continue
        assert O.e4m3_to_double(b) == ref[b].item(), hex(b)


def test_bf16_decode_matches_torch():
    bits = torch.arange(0, 65536, 13, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64)
    for b, r in zip(bits.tolist(), ref.tolist()):
        if math.isnan(r):
            continue
        assert O.bf16_to_double(b & 0xFFFF) == r


def test_e2m1_value_set_from_the_pages():
    # magnitudes of the 8 non-negative codes are {0, .5, 1, 1.5, 2, 3, 4, 6}; bit 3 is the sign
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(16):
        v = O.e2m1_to_double(c)
        assert abs(v) == mags[c & 7]
        assert (math.copysign(1.0, v) < 0) == bool(c & 8)


def test_e2m1_rounding_table():
    for v, code in _rows("e2m1_rounding.txt"):
        assert O.e2m1_rn_satfinite(float(v)) == int(code, 16), v


def _e4m3_finite_values():
    vals = []
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            vals.append((m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7))
    return sorted(set(vals))


def _nearest_even(grid, codes_of, x):
    """Brute force: nearest grid value, ties to the even code, saturating."""
    a = abs(x)
    if a >= grid[-1]:
        return grid[-1]
    best = min(grid, key=lambda g: abs(g - a))
    ties = [g for g in grid if abs(g - a) == abs(best - a)]
    if len(ties) > 1:
        best = [g for g in ties if codes_of[g] % 2 == 0][0]
    return best


def test_e4m3_encoder_brute_force():
    grid = _e4m3_finite_values()
    codes = {O.e4m3_to_double(c): c for c in range(0x7F)}
    rng = np.random.default_rng(0)
    samples = list(rng.uniform(0, 500, 2000)) + list(2.0 ** rng.uniform(-12, 9, 2000))
    # every midpoint between neighbours (exact ties) and a few beyond the max
    samples += [(a + b) / 2 for a, b in zip(grid[:-1], grid[1:])] + [448.0, 460.0, 464.0, 1e9]
    for x in samples:
        x = float(np.float32(x))
        want = _nearest_even(grid, codes, x)
        got = O.e4m3_rn_satfinite(x)
        assert O.e4m3_to_double(got) == want, (x, hex(got), want)
    assert O.e4m3_rn_satfinite(-1.0) == 0xB8


def test_e2m1_encoder_brute_force():
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    codes = {v: i for i, v in enumerate(grid)}
    for x in np.linspace(-8, 8, 3201):
        x = float(np.float32(x))
        want = _nearest_even(grid, codes, x)
        got = O.e2m1_rn_satfinite(x)
        assert abs(O.e2m1_to_double(got)) == want, (x, hex(got))
        if x < 0:
            assert got & 8


def test_bf16_encoder_vs_exact_rounding():
    rng = np.random.default_rng(1)
    xs = list(rng.standard_normal(3000) * 10.0 ** rng.uniform(-30, 30, 3000))
    for x in xs:
        x = float(x)
        b = O.bf16_from_double(x)
        v = O.bf16_to_double(b)
        # neighbours of v in bf16 are v's bit pattern +-1: x must be no farther from v
        up = O.bf16_to_double((b + 1) & 0xFFFF)
        dn = O.bf16_to_double((b - 1) & 0xFFFF)
        assert abs(x - v) <= abs(x - up) and abs(x - v) <= abs(x - dn)
        if abs(x - v) == abs(x - up) or abs(x - v) == abs(x - dn):
            assert b % 2 == 0
