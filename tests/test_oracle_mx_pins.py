"""CPU pins of the oracle's MXFP4 quantization (a comparison format of the
pages; the OCP Microscaling definition is the reading: 32-element blocks, one
E8M0 scale 2^s with s = floor(log2(max|y|)) - 2, E2M1 elements by RTNE with
saturation at 6, or SR).

Each pin checks the oracle against something other than itself: the bit
pattern of fp32 exponents, closed-form blocks, brute-force nearest values,
power-of-two invariance, numpy statistics and the sample mean of SR.
"""
import math

import numpy as np
import pytest

from fp4_quantized_numerics_gb300 import inputs

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _val(codes):
    c = codes.astype(np.int64)
    return np.where(c & 8, -1.0, 1.0) * E2M1[c & 7]


def _block(vals):
    x = np.zeros((1, 32), np.float32)
    x[0, :len(vals)] = vals
    return x


def test_e8m0_decode_all_bytes(oracle):
    for b in range(255):
        assert oracle.e8m0_decode(b) == math.ldexp(1.0, b - 127)
    assert math.isnan(oracle.e8m0_decode(255))


def test_shared_exponent_from_fp32_bits(oracle):
    rng = np.random.default_rng(5)
    vals = np.concatenate([
        np.ldexp(1.0, np.arange(-126, 128)).astype(np.float32),                       # powers of two
        np.nextafter(np.ldexp(1.0, np.arange(-125, 128)).astype(np.float32), np.float32(0)),  # just below
        (rng.random(2000) * 10.0 ** rng.integers(-30, 30, 2000)).astype(np.float32),
    ])
    vals = vals[np.isfinite(vals) & (vals > 0)]
    for a in vals:
        bits = int(np.float32(a).view(np.uint32))
        ef = (bits >> 23) & 0xFF
        floor_log2 = ef - 127 if ef else (bits.bit_length() - 1) - 149
        assert oracle.mx_shared_exp(a) == max(min(floor_log2 - 2, 127), -127), a
    assert oracle.mx_shared_exp(0.0) == -127


@pytest.mark.parametrize("vals,scale_byte,codes", [
    ([6.0, 3.0, -1.5, 0.5, 0.0], 127, [7, 5, 8 | 3, 1, 0]),         # max 6: s = 0, all exact
    ([7.0, 5.0, -5.0, 1.25], 127, [7, 6, 8 | 6, 2]),                 # 7 saturates; 5 and 1.25 tie to even
    ([0.75, 0.375, -0.0625], 124, [7, 5, 8 | 1]),                    # max 0.75: s = -3, X = 1/8
    ([8.0, 1.0, 2.5], 128, [6, 1, 2]),                               # max 8: s = 1; 2.5/2 = 1.25 -> 1.0
    ([2.0 ** -130, -(2.0 ** -131)], 0, [0, 8]),                       # clamped to s = -127: flushes
])
def test_closed_form_blocks(oracle, vals, scale_byte, codes):
    r = oracle.quantize_mx(_block(vals))
    assert r["scales"][0, 0] == scale_byte
    np.testing.assert_array_equal(r["codes"][0, :len(codes)], codes)
    assert not r["codes"][0, len(vals):].any()


def test_zero_block(oracle):
    r = oracle.quantize_mx(np.zeros((3, 64), np.float32))
    assert not r["codes"].any() and not r["scales"].any()


@pytest.mark.parametrize("t", [-20, -3, 1, 7, 40])
def test_power_of_two_invariance(oracle, t):
    x = inputs.normal(7, (16, 128))
    a, b = oracle.quantize_mx(x), oracle.quantize_mx((x * np.float32(2.0 ** t)).astype(np.float32))
    np.testing.assert_array_equal(a["codes"], b["codes"])
    np.testing.assert_array_equal(b["scales"].astype(int), a["scales"].astype(int) + t)


def test_picks_nearest_representable(oracle):
    x = inputs.normal(8, (32, 256)) * np.float32(3.0)
    r = oracle.quantize_mx(x)
    X = np.ldexp(1.0, r["scales"].astype(np.int64) - 127).repeat(32, axis=1)
    q = x.astype(np.float64) / X
    a = np.minimum(np.abs(q), 6.0)
    err = np.abs(a[..., None] - E2M1[None, None, :])
    best = err.min(axis=-1)
    m = r["codes"] & 7
    np.testing.assert_array_equal(np.abs(a - E2M1[m]), best)          # nearest
    ties = (err == best[..., None]).sum(-1) > 1
    assert (m[ties] % 2 == 0).all()                                    # ties to the even index
    np.testing.assert_array_equal((r["codes"] >> 3).astype(bool), np.signbit(x))
    # the block max lands in (2, 6] after scaling (s = floor(log2 max) - 2); 6 saturates from [6, 8)
    amax = np.abs(x).reshape(32, 8, 32).max(-1)
    sc = amax / np.ldexp(1.0, r["scales"].astype(np.int64) - 127)
    assert ((sc >= 4.0) & (sc < 8.0)).all()


def test_colwise_is_rowwise_of_transpose(oracle):
    x = inputs.normal(9, (64, 96))
    a, b = oracle.quantize_mx(x, colwise=True), oracle.quantize_mx(np.ascontiguousarray(x.T))
    np.testing.assert_array_equal(a["codes"], b["codes"])
    np.testing.assert_array_equal(a["scales"], b["scales"])


def test_rht_rotates_each_half(oracle):
    x = inputs.normal(10, (8, 128))
    r = oracle.quantize_mx(x, rht=True, rht_seed=2)
    ref = oracle.quantize(x, oracle.E2M1, rht=True, rht_seed=2)["y"]     # 16-block rotation
    np.testing.assert_array_equal(r["y"], ref)


def test_dequantize_is_exact_product(oracle):
    x = inputs.normal(11, (16, 64))
    r = oracle.quantize_mx(x)
    d = oracle.dequantize_mx(r["codes"], r["scales"])
    np.testing.assert_array_equal(d, _val(r["codes"]) * np.ldexp(1.0, r["scales"].astype(np.int64) - 127).repeat(32, 1))
    inv = oracle.dequantize_mx(*(lambda q: (q["codes"], q["scales"]))(oracle.quantize_mx(x, rht=True, rht_seed=3)),
                               inverse_rht=True, rht_seed=3)
    assert np.abs(inv - x).max() <= 0.35 * np.abs(x).max()


def test_stats_match_numpy(oracle):
    x = inputs.normal(12, (32, 128))
    r = oracle.quantize_mx(x)
    s = oracle.stats_mx(r["y"], r["codes"], r["scales"])
    d = oracle.dequantize_mx(r["codes"], r["scales"])
    y = r["y"].astype(np.float64)
    assert s["alpha"] == pytest.approx((d * y).sum() / (y * y).sum(), rel=1e-12)
    assert s["sqnr_db"] == pytest.approx(10 * np.log10((y * y).sum() / ((y - d) ** 2).sum()), rel=1e-12)
    assert s["mean_bias"] < 0   # E2M1's asymmetric top bins pull toward zero


def test_sr_mean_is_unbiased_within_5_sigma(oracle):
    x = _block(np.linspace(-5.9, 5.9, 32).astype(np.float32))
    n = 600
    acc = np.zeros(32)
    for c in range(n):
        r = oracle.quantize_mx(x, round_mode=oracle.SR, sr_seed=17, sr_counter=c)
        acc += oracle.dequantize_mx(r["codes"], r["scales"])[0]
    mean = acc / n
    # per element the SR outcome is lo or hi (gap <= 2 X), so sigma <= gap / 2 / sqrt(n)
    assert (np.abs(mean - x[0]) <= 5 * (2.0 / 2) / math.sqrt(n)).all()
