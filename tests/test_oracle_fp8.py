"""Pins for the FP8 E4M3 codec: format constants, torch's float8_e4m3fn, exhaustive round trip."""
import math

import numpy as np
import torch

from oracle import fp8


def test_format_constants():
    assert fp8.decode_code(0x00) == 0.0
    assert fp8.decode_code(0x01) == 2.0 ** -9          # smallest subnormal
    assert fp8.decode_code(0x07) == 7 * 2.0 ** -9      # largest subnormal
    assert fp8.decode_code(0x08) == 2.0 ** -6          # smallest normal
    assert fp8.decode_code(0x38) == 1.0                # exponent field 7 = bias
    assert fp8.decode_code(0x7E) == 448.0              # largest finite
    assert math.isnan(fp8.decode_code(0x7F)) and math.isnan(fp8.decode_code(0xFF))
    assert fp8.decode_code(0xFE) == -448.0
    assert math.copysign(1.0, fp8.decode_code(0x80)) == -1.0


def test_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    mine = fp8.decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert (np.isnan(mine) == nan).all()
    assert (mine[~nan] == ref[~nan]).all()


def test_roundtrip_every_code():
    for c in range(256):
        v = fp8.decode_code(c)
        if math.isnan(v):
            assert fp8.encode_value(v) == 0x7F
            continue
        assert fp8.encode_value(v) == c
    vals = fp8.decode(np.arange(256, dtype=np.uint8)).astype(np.float32)
    enc = fp8.encode_f32(vals)
    ok = ~np.isnan(vals)
    assert (enc[ok] == np.arange(256)[ok]).all()


def _halfway_points():
    vals = sorted(set(fp8.decode_code(c) for c in range(0x00, 0x7F)))
    mids = [(a + b) / 2 for a, b in zip(vals, vals[1:])]
    out = []
    for m in mids:
        m32 = np.float32(m)
        assert float(m32) == m                          # midpoints are exact in f32
        out += [m32, np.nextafter(m32, np.float32(0)), np.nextafter(m32, np.float32(1e9))]
    out = np.array(out, dtype=np.float32)
    return np.concatenate([out, -out])


def test_encode_ties_to_even_against_torch():
    x = _halfway_points()
    mine = fp8.encode_f32(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (mine == ref).all()
    scal = np.array([fp8.encode_value(float(t)) for t in x], dtype=np.uint8)
    assert (scal == mine).all()


def test_encode_random_against_torch_in_range():
    r = np.random.default_rng(3)
    x = (r.standard_normal(300000) * np.exp2(r.integers(-12, 9, 300000))).astype(np.float32)
    x = x[np.abs(x) < 448]
    mine = fp8.encode_f32(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (mine == ref).all()


def test_saturation_and_nan():
    x = np.array([448.0, 449.0, 464.0, 470.0, 1e30, np.inf, -500.0, -np.inf, np.nan],
                 dtype=np.float32)
    enc = fp8.encode_f32(x)
    assert enc.tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F]
    assert [fp8.encode_value(float(t)) for t in x] == enc.tolist()
