"""Pins of the oracle's E4M3 decoding (OCP 8-bit floating point, E4M3: bias 7, 3 mantissa
bits, subnormals, no infinities, S.1111.111 = NaN) used by the FP8 forward's parity tests."""
import math

import numpy as np
import torch

import oracle


def test_e4m3_landmark_codes():
    cases = {0x00: 0.0, 0x80: -0.0, 0x38: 1.0, 0xB8: -1.0, 0x40: 2.0, 0x3C: 1.5, 0x7E: 448.0, 0xFE: -448.0,
             0x08: 2.0 ** -6, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x30: 0.5, 0x77: 240.0}
    got = oracle.e4m3_to_f64(np.array(list(cases), dtype=np.uint8))
    for (code, want), g in zip(cases.items(), got):
        assert g == want and math.copysign(1, g) == math.copysign(1, want), (hex(code), g, want)
    nan = oracle.e4m3_to_f64(np.array([0x7F, 0xFF], dtype=np.uint8))
    assert np.all(np.isnan(nan))


def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.array_equal(ours[~both_nan], ref[~both_nan]) and np.array_equal(np.isnan(ours), np.isnan(ref))


def test_e4m3_forward_equals_f64_forward_of_decoded_values():
    g = torch.Generator().manual_seed(61)
    Q, K, V = (torch.randn(1, 2, 40, 16, generator=g).to(torch.float8_e4m3fn) for _ in range(3))
    O8, L8 = oracle.sdpa_forward_e4m3(Q, K, V, causal=True)
    O, L = oracle.sdpa_forward_f64(Q.to(torch.float64), K.to(torch.float64), V.to(torch.float64), causal=True)
    np.testing.assert_array_equal(O8, O)
    np.testing.assert_array_equal(L8, L)
