"""CPU check of the E1M2 rounding trick of the kernels.

The kernels round q (grid units, already clamped to |q| <= 3.5) to E1M2 by
the round-to-nearest-even E4M3 conversion of x = q * 2^-8: on [0, 15 * 2^-9]
E4M3 is a uniform grid of step 2^-9 (the subnormals, then the first normal
binade), so the E4M3 byte's low bits are m = rint(2 |q|) with ties to even
and its top bit is the sign.  This test restates the trick with torch's
float8_e4m3fn conversion and compares it with the oracle's E1M2 RTNE.
"""
import numpy as np
import pytest
import torch


def test_e1m2_from_e4m3_bits(oracle):
    rng = np.random.default_rng(21)
    q = np.concatenate([
        rng.uniform(-3.5, 3.5, 20000).astype(np.float32),
        np.arange(-7, 8, dtype=np.float32) * np.float32(0.5),          # grid points
        np.arange(-7, 7, dtype=np.float32) * np.float32(0.5) + np.float32(0.25),   # ties
        np.array([0.0, -0.0, 3.5, -3.5], np.float32),
    ])
    x = torch.from_numpy(q * np.float32(2.0 ** -8))
    b = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy().astype(np.int64)
    code = (b & 7) | ((b >> 4) & 8)
    assert ((b & 0x78) == 0).all()                       # never past index 7
    for qi, ci in zip(q, code):
        m = oracle.round_rtne(oracle.E1M2, abs(float(qi)))
        assert ci == ((8 if np.signbit(qi) else 0) | m), (float(qi), int(ci))


@pytest.mark.parametrize("q", [0.25, 0.75, 1.25, 1.75, 2.25, 2.75, 3.25])
def test_ties_go_to_even_index(oracle, q):
    b = int(torch.tensor([q * 2.0 ** -8]).to(torch.float8_e4m3fn).view(torch.uint8).item())
    assert (b & 7) % 2 == 0 and (b & 7) == oracle.round_rtne(oracle.E1M2, q)
