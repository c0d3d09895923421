"""Pins of the E4M3 oracle (oracle/fp8.py) against closed forms, the format's
invariants and torch's float8_e4m3fn conversion (a library routine)."""
import math

import numpy as np
import torch

import nc_synth
from oracle import fp8


def test_decode_closed_forms():
    cases = {0x00: 0.0, 0x80: -0.0, 0x38: 1.0, 0xB8: -1.0, 0x40: 2.0, 0x3C: 1.5,
             0x7E: 448.0, 0xFE: -448.0, 0x08: 2.0 ** -6, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9,
             0x30: 0.5, 0x39: 1.125, 0x77: 240.0}
    for code, val in cases.items():
        got = float(fp8.e4m3_decode(np.array([code], np.uint8))[0])
        assert got == val and math.copysign(1.0, got) == math.copysign(1.0, val), (hex(code), got)
    assert np.isnan(fp8.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()


def test_decode_matches_torch_float8_e4m3fn_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_decode_is_monotone_and_symmetric():
    pos = fp8.e4m3_decode(np.arange(0x00, 0x7F, dtype=np.uint8))   # 0 .. 448, NaN excluded
    assert np.all(np.diff(pos) > 0) and pos[-1] == fp8.E4M3_MAX
    neg = fp8.e4m3_decode(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.array_equal(neg, -pos)
    # consecutive normals in one binade differ by 2^(e - 7) / 8
    v = fp8.e4m3_decode(np.arange(0x38, 0x40, dtype=np.uint8))
    assert np.allclose(np.diff(v), 1.0 / 8.0, rtol=0, atol=0)


def test_gemm_brute_force_and_scale():
    a = nc_synth.make_e4m3_codes(5, 32, seed=1)
    b = nc_synth.make_e4m3_codes(3, 32, seed=2)
    got = fp8.gemm_e4m3(a, b, 0.25)
    da, db = fp8.e4m3_decode(a), fp8.e4m3_decode(b)
    for i in range(5):
        for j in range(3):
            s = 0.0
            for k in range(32):
                s += da[i, k] * db[j, k]
            assert got[i, j] == 0.25 * s
    # the generator never emits NaN codes and keeps the exponent field in range
    e = (nc_synth.make_e4m3_codes(64, 64, seed=3) >> 3) & 0xF
    assert e.min() >= 3 and e.max() <= 10
