"""Pins for the oracle's E4M3 decoder: hand-worked codes from the format's
definition, every code against torch's own float8_e4m3fn conversion (an
independent implementation), and the ordering of the codes. CPU only."""
import math

import numpy as np
import torch

from oracle import e4m3_decode


def test_hand_worked_codes():
    cases = {0x00: 0.0, 0x38: 1.0, 0x3C: 1.5, 0x40: 2.0, 0x7E: 448.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9,
             0x08: 2.0 ** -6, 0xB8: -1.0, 0xFE: -448.0, 0x30: 0.5, 0x4B: 2.0 ** 2 * 1.375}
    for code, val in cases.items():
        assert e4m3_decode(code) == val, hex(code)
    assert math.copysign(1.0, e4m3_decode(0x80)) == -1.0 and e4m3_decode(0x80) == 0.0
    assert np.isnan(e4m3_decode(0x7F)) and np.isnan(e4m3_decode(0xFF))


def test_every_code_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = e4m3_decode(np.arange(256))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_positive_codes_increase():
    v = e4m3_decode(np.arange(0x7F))
    assert np.all(np.diff(v) > 0)
    assert np.array_equal(e4m3_decode(np.arange(0x80, 0xFF)), -v)
