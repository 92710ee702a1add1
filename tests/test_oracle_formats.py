"""Pins for the oracle's number formats (E2M1, E4M3, bf16) against closed forms
and library routines.  CPU only."""
import numpy as np
import pytest
import torch

import indep


def test_e2m1_table_matches_closed_form(orc):
    for c in range(16):
        assert orc.e2m1_value(c) == indep.e2m1_closed_form(c)
        # the sign bit is kept, zero included
        assert np.signbit(orc.e2m1_value(c)) == bool(c & 8)


def test_e4m3_decode_matches_torch_all_256(orc):
    ref = indep.e4m3_torch(np.arange(256))
    for b in range(256):
        v = orc.e4m3_value(b)
        if np.isnan(ref[b]):
            assert np.isnan(v), b
        else:
            assert v == ref[b], (b, v, ref[b])
    assert orc.e4m3_value(0x7E) == 448.0
    assert orc.e4m3_value(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_cast_and_rint(orc):
    rng = np.random.default_rng(0)
    # log-uniform magnitudes over the whole range, plus every midpoint between codes
    vals = np.exp2(rng.uniform(-12, 9.2, 4000)).astype(np.float32)
    grid = indep.e4m3_torch(np.arange(127))
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    vals = np.concatenate([vals, mids, grid.astype(np.float32), [0.0, 448.0, 463.9, 464.0]])
    vals = vals[vals < 464.0].astype(np.float32)
    torch_codes = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = np.array([orc.e4m3_encode(v) for v in vals], np.uint8)
    np.testing.assert_array_equal(mine, torch_codes)
    # independent rint route on the values
    dec = np.array([orc.e4m3_value(c) for c in mine])
    np.testing.assert_array_equal(dec, indep.e4m3_round(vals.astype(np.float64)))


def test_e4m3_encode_saturates(orc):
    for v in [464.0, 500.0, 1e6, 3.4e38]:
        assert orc.e4m3_encode(v) == 0x7E
        assert orc.e4m3_encode(-v) == 0xFE


def test_e2m1_encode_rint_route_and_ties(orc):
    rng = np.random.default_rng(1)
    mags = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    mids = (mags[:-1] + mags[1:]) / 2
    vals = np.concatenate([rng.uniform(-8, 8, 5000), mags, -mags, mids, -mids,
                           [6.5, 100.0, -1e9, 1e-30, -1e-30]]).astype(np.float32)
    for v in vals:
        c = orc.e2m1_encode(float(v))
        got = orc.e2m1_value(c)
        want = indep.e2m1_round(np.float64(v))
        assert got == want, (v, c, got, want)
        assert bool(c & 8) == bool(np.signbit(v))
    # the tie cases written out: ties go to the even mantissa bit
    for v, code in [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),
                    (-0.25, 8), (-5.0, 14), (7.0, 7), (-0.1, 8)]:
        assert orc.e2m1_encode(v) == code, (v, orc.e2m1_encode(v), code)


def test_bf16_round_trip_and_rne(orc):
    rng = np.random.default_rng(2)
    f = rng.standard_normal(3000).astype(np.float32) * np.exp2(rng.integers(-20, 20, 3000))
    # torch float32 -> bf16 is round-half-even; fp32 inputs avoid double rounding
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.bf16_from_double(float(v)) for v in f], np.uint16)
    np.testing.assert_array_equal(got, want)
    # exact ties between two bf16 values: 1 + 2^-8 lies between 1 and 1 + 2^-7
    assert orc.bf16_from_double(1.0 + 2.0 ** -8) == 0x3F80
    assert orc.bf16_from_double(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert orc.bf16_from_double(0.0) == 0 and orc.bf16_from_double(-0.0) == 0x8000
