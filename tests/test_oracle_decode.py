"""Pins for the oracle's format decoders (CPU only).

E4M3: every code against the float8_e4m3fn decode of a tensor library, plus closed-form spot
values from the OCP FP8 definition (tests/golden/e4m3_spot.txt).  f16: every code against
numpy.float16.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_spot.txt")


def _read_spots():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            code, val = line.split()
            rows.append((int(code, 16), val))
    return rows


def test_e4m3_spot_values(oracle):
    spots = _read_spots()
    assert len(spots) >= 12
    for code, val in spots:
        got = oracle.e4m3(code)
        if val == "nan":
            assert math.isnan(got), hex(code)
        elif val == "-0":
            assert got == 0.0 and math.copysign(1.0, got) < 0, hex(code)
        else:
            assert got == float(val), (hex(code), got, val)


def test_e4m3_all_codes_vs_library(oracle):
    tab = oracle.e4m3_table()
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan_o = np.isnan(tab)
    nan_l = np.isnan(lib)
    assert np.array_equal(nan_o, nan_l)
    assert set(np.nonzero(nan_o)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(tab[~nan_o], lib[~nan_l])
    # signs of zeros too
    assert np.array_equal(np.signbit(tab[~nan_o]), np.signbit(lib[~nan_l]))


def test_e4m3_structure(oracle):
    tab = oracle.e4m3_table()
    # sign bit negates exactly; magnitudes increase monotonically with the code
    for c in range(128):
        if c == 0x7F:
            continue
        assert tab[c | 0x80] == -tab[c]
    mags = tab[:0x7F]
    assert np.all(np.diff(mags) > 0)
    assert tab[0x7E] == 448.0 and tab[0x01] == 2.0 ** -9


def test_f16_all_codes_vs_numpy(oracle):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_decode(bits)
    ref = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))
    assert oracle.f16_decode(np.array([0x1400], np.uint16))[0] == 2.0 ** -10


@pytest.mark.parametrize("code,val", [(0x3C00, 1.0), (0x0001, 2.0 ** -24), (0x7BFF, 65504.0),
                                      (0xC000, -2.0), (0x0400, 2.0 ** -14)])
def test_f16_closed_forms(oracle, code, val):
    assert oracle.f16_decode(np.array([code], np.uint16))[0] == val
