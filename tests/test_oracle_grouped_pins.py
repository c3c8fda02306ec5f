"""Pins of the oracle's grouped (mixture-of-experts) quantization (CPU only).

oracle.quantize_grouped places every expert segment in one output tensor with
its own tensor scale: row-wise segments at 128-row offsets, column-wise
segments (the quantization of x_e^T, tokens zero-padded to a multiple of 16)
at 64-wide k offsets, stochastic rounding indexed by the element's place in
the whole output.  The checks below rebuild each code from scratch, one
element at a time, from the layout rules of include/ufp4.h and the oracle's
scalar primitives (E4M3 encode/decode, grid rounding, the SR word), with the
scale steps as single fp32 operations in numpy.  Nothing here calls
oracle.quantize, so a wrong segment offset, a shared tensor scale, padding
that is not zero or an SR word taken at the wrong index fails a test.
([HP] technical approach: the MoE 7.9B and 124B models; [ZC] Key points,
"Validation results".)
"""
import numpy as np
import pytest

from fp4_quantized_numerics_gb300 import inputs

F32 = np.float32


def _round_up(v, m):
    return (v + m - 1) // m * m


def _brute_segment(oracle, M, grid, rnd, sr_seed, sr_counter, index_of):
    """Codes [rows, k] and scales [rows, k/16] of the matrix M (blocks along
    its rows), element (r, j) drawing SR word index_of(r, j); returns
    (codes, scales, S_dec)."""
    qmax = F32(oracle.grid_qmax(grid))
    A_t = F32(np.abs(M).max()) if M.size else F32(0)
    if A_t > 0:
        S_enc = F32(F32(448) * qmax / A_t)
        S_dec = F32(A_t / (F32(448) * qmax))
    else:
        S_enc = S_dec = F32(1)
    rows, k = M.shape
    codes = np.zeros((rows, k), np.uint8)
    scales = np.zeros((rows, k // 16), np.uint8)
    for r in range(rows):
        for b in range(k // 16):
            blk = M[r, 16 * b:16 * b + 16]
            e = oracle.e4m3_encode(F32(F32(np.abs(blk).max()) / qmax) * S_enc)
            scales[r, b] = e
            if e == 0:
                continue
            kk = F32(S_enc / F32(oracle.e4m3_decode(e)))
            for j in range(16):
                q = F32(blk[j] * kk)
                a = min(abs(float(q)), float(qmax))
                if rnd == 1:
                    m = oracle.round_sr(grid, a, oracle.sr_bits(sr_seed, sr_counter, index_of(r, 16 * b + j)))
                else:
                    m = oracle.round_rtne(grid, a)
                codes[r, 16 * b + j] = (8 if np.signbit(q) else 0) | m
    return codes, scales, float(S_dec)


COUNTS = [37, 0, 130, 5, 1, 16]
COLS = 48


def _data(seed=3):
    g = np.random.default_rng(seed)
    x = inputs.to_bf16_f32(g.standard_normal((sum(COUNTS), COLS), dtype=np.float32))
    # segments of very different magnitude, so one shared scale would show
    starts = np.concatenate([[0], np.cumsum(COUNTS)])
    for e in range(len(COUNTS)):
        x[starts[e]:starts[e + 1]] *= np.float32(4.0 ** (e - 2))
    return x, starts


@pytest.mark.parametrize("grid", [0, 1])
@pytest.mark.parametrize("rnd", [0, 1])
def test_grouped_rowwise_element_by_element(oracle, grid, rnd):
    """Row-wise: segment e is its rows' quantization under its own tensor
    scale, placed at roff_e = sum of round_up(T, 128) of the earlier nonempty
    segments; SR word index (roff_e + r) * cols + c."""
    x, starts = _data()
    seed, ctr = 0x1234_5678_9ABC, 7
    got = oracle.quantize_grouped(x, COUNTS, grid, round_mode=rnd, sr_seed=seed, sr_counter=ctr)
    roff = 0
    for e, T in enumerate(COUNTS):
        if T == 0:
            assert got[e] is None
            continue
        seg = x[starts[e]:starts[e] + T]
        codes, scales, sdec = _brute_segment(oracle, seg, grid, rnd, seed, ctr,
                                             lambda r, c, o=roff: (o + r) * COLS + c)
        assert got[e]["off"] == roff
        np.testing.assert_array_equal(got[e]["scales"], scales)
        np.testing.assert_array_equal(got[e]["codes"], codes)
        assert got[e]["tensor_scale"] == sdec
        roff += _round_up(T, 128)


@pytest.mark.parametrize("grid", [0, 1])
@pytest.mark.parametrize("rnd", [0, 1])
def test_grouped_colwise_element_by_element(oracle, grid, rnd):
    """Column-wise: segment e is the quantization of x_e^T (cols x T16_e,
    tokens zero-padded to T16_e = round_up(T, 16)) at koff_e = sum of
    round_up(T, 64) of the earlier nonempty segments, in an output of row
    length Ktot = sum round_up(T, 64); SR word index c * Ktot + koff_e + t.
    The padded tokens carry code 0 (zero input, sign bit clear)."""
    x, starts = _data(4)
    seed, ctr = 99, 0xFFFF_FFFF_0000_0001
    ktot = sum(_round_up(T, 64) for T in COUNTS if T > 0)
    got = oracle.quantize_grouped(x, COUNTS, grid, round_mode=rnd, sr_seed=seed, sr_counter=ctr, colwise=True)
    koff = 0
    for e, T in enumerate(COUNTS):
        if T == 0:
            assert got[e] is None
            continue
        t16 = _round_up(T, 16)
        Mt = np.zeros((COLS, t16), np.float32)
        Mt[:, :T] = x[starts[e]:starts[e] + T].T
        codes, scales, sdec = _brute_segment(oracle, Mt, grid, rnd, seed, ctr,
                                             lambda c, t, o=koff: c * ktot + o + t)
        assert got[e]["off"] == koff
        assert got[e]["codes"].shape == (COLS, t16)
        np.testing.assert_array_equal(got[e]["scales"], scales)
        np.testing.assert_array_equal(got[e]["codes"], codes)
        assert not got[e]["codes"][:, T:].any()
        assert got[e]["tensor_scale"] == sdec
        koff += _round_up(T, 64)


def test_grouped_segments_are_independent(oracle):
    """Changing one segment's data leaves every other segment's codes, scales
    and tensor scale unchanged (each has its own amax), both layouts."""
    x, starts = _data(5)
    y = x.copy()
    y[starts[2]:starts[3]] *= np.float32(1000.0)
    for col in (False, True):
        a = oracle.quantize_grouped(x, COUNTS, 1, colwise=col)
        b = oracle.quantize_grouped(y, COUNTS, 1, colwise=col)
        for e in range(len(COUNTS)):
            if a[e] is None or e == 2:
                continue
            np.testing.assert_array_equal(a[e]["codes"], b[e]["codes"])
            assert a[e]["tensor_scale"] == b[e]["tensor_scale"]
        assert b[2]["tensor_scale"] != a[2]["tensor_scale"]
