"""GPU parity of the MXFP4 quantizer (UFP4_MXFP4) against the CPU oracle.

The reading (the pages name MXFP4 only as a comparison format): the OCP
microscaling definition, 32-element blocks with an E8M0 scale, E2M1 elements.
The GPU stores the scale byte at both of the block's 16-block places of the
scale layout; the oracle keeps one byte per block.  Bars as for the other
grids: bit-exact codes and scale bytes without the transform (RTNE and SR);
with it, codes within one grid step on at most 1e-4 of the elements where the
block scales agree (the fp32 butterflies round differently from the oracle's
fp64 product, which can move a block maximum across a power of two).
"""
import numpy as np
import pytest
import torch

from fp4_quantized_numerics_gb300 import inputs
from tests import layouts

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def U():
    from fp4_quantized_numerics_gb300 import build, ufp4
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return ufp4


def _gpu(U, x, dtype, col, rht, rnd, seed=5):
    t = torch.from_numpy(np.ascontiguousarray(x)).to(dtype).cuda()
    q = U.ufp4_quantize(t, U.UFP4_MXFP4, rht=rht, rht_seed=2, round=rnd, sr_seed=seed, sr_counter=3,
                        colwise=col)
    torch.cuda.synchronize()
    cb, sb = q.codes.cpu().numpy(), q.scales.cpu().numpy()
    codes = layouts.unpack_codes(cb, q.rows, q.k)
    s16, spad = layouts.unpack_scales(sb, q.rows, q.k)
    return dict(t=t, q=q, codes=codes, s16=s16, spad=spad, pad=layouts.code_padding(cb, q.rows, q.k),
                ts=float(q.tensor_scale.item()))


def _si(c):
    c = c.astype(np.int32)
    return np.where(c & 8, -(c & 7), c & 7)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("col", [False, True])
@pytest.mark.parametrize("rht,rnd", [(False, 0), (False, 1), (True, 0), (True, 1)])
@pytest.mark.parametrize("rows,cols", [(256, 1024), (96, 1056), (160, 32)])
def test_mx_matches_oracle(U, oracle, dtype, col, rht, rnd, rows, cols):
    # 96 x 1056: a padding 32-block in kpad row-wise (k = 1056) and column-wise
    # (k = 96), rows off the 128-row scale tile; 160 x 32: one block per row
    x = inputs.normal(30 + rows, (rows, cols)) * np.float32(4.0)
    xr = torch.from_numpy(x).to(dtype).float().numpy()     # what the GPU sees
    g = _gpu(U, x, dtype, col, rht, rnd)
    r = oracle.quantize_mx(xr, rht=rht, rht_seed=2, round_mode=rnd, sr_seed=5, sr_counter=3, colwise=col)
    assert g["ts"] == 1.0
    np.testing.assert_array_equal(g["s16"][:, 0::2], g["s16"][:, 1::2])   # both 16-block places
    assert not g["pad"].any() and not g["spad"].any()
    s32 = g["s16"][:, 0::2]
    if not rht:
        np.testing.assert_array_equal(s32, r["scales"])
        np.testing.assert_array_equal(g["codes"], r["codes"])
    else:
        same = s32 == r["scales"]
        assert (~same).mean() <= 1e-3 and (np.abs(s32.astype(int) - r["scales"]) <= 1).all()
        m = np.repeat(same, 32, axis=1)
        d = np.abs(_si(g["codes"]) - _si(r["codes"]))[m]
        assert d.max() <= 1 and (d > 0).mean() <= 1e-4


def test_mx_closed_form_block(U):
    # max 0.75 -> s = -3: every value lands on the grid exactly
    x = np.zeros((128, 64), np.float32)
    x[:, :5] = [0.75, 0.375, -0.0625, 0.25, 0.0]
    g = _gpu(U, x, torch.float32, False, False, 0)
    assert (g["s16"][:, 0] == 124).all() and (g["s16"][:, 2] == 0).all()   # second block all zero
    np.testing.assert_array_equal(g["codes"][0, :5], [7, 5, 9, 4, 0])


def test_mx_dequantize_and_stats(U, oracle):
    x = inputs.normal(40, (128, 512)) * np.float32(2.0)
    for rht in (False, True):
        g = _gpu(U, x, torch.float32, False, rht, 0)
        d = U.ufp4_dequantize(g["q"]).cpu().numpy().astype(np.float64)
        ref = oracle.dequantize_mx(g["codes"], g["s16"][:, 0::2])
        np.testing.assert_array_equal(d, ref)                   # v(m) 2^s is exact in fp32
        inv = U.ufp4_dequantize(g["q"], inverse_rht=rht, rht_seed=2).cpu().numpy().astype(np.float64)
        iref = oracle.dequantize_mx(g["codes"], g["s16"][:, 0::2], inverse_rht=rht, rht_seed=2)
        assert np.abs(inv - iref).max() <= 1e-6 * np.abs(iref).max()
        st = U.ufp4_stats(g["t"], g["q"], rht=rht, rht_seed=2)
        r = oracle.quantize_mx(x, rht=rht, rht_seed=2)
        ro = oracle.stats_mx(r["y"], r["codes"], r["scales"])
        tol = 1.0 if not rht else 10.0
        assert abs(st["alpha"] - ro["alpha"]) <= 1e-6 * tol
        assert abs(st["sqnr_db"] - ro["sqnr_db"]) <= 1e-4 * tol
        assert abs(st["mean_bias"] - ro["mean_bias"]) <= 1e-5 * tol


def test_mx_refused_where_unsupported(U):
    x = torch.from_numpy(inputs.normal(41, (128, 256))).to(torch.bfloat16).cuda()
    q = U.ufp4_quantize(x, U.UFP4_MXFP4)
    with pytest.raises(U.UFP4Error) as e:                       # MX and NVFP4-style operands do not mix
        U.ufp4_gemm(q, U.ufp4_quantize(x, U.UFP4_E2M1))
    assert e.value.status == U.UFP4_ERR_UNSUPPORTED
    with pytest.raises(U.UFP4Error) as e:
        U.ufp4_quantize_dual(x, U.UFP4_MXFP4)
    assert e.value.status == U.UFP4_ERR_UNSUPPORTED
    with pytest.raises(U.UFP4Error) as e:
        U.ufp4_quantize_grouped(x, U.UFP4_MXFP4, [100, 28])
    assert e.value.status == U.UFP4_ERR_UNSUPPORTED
    with pytest.raises(U.UFP4Error) as e:                       # no tensor amax for MX
        U.ufp4_quantize(x, U.UFP4_MXFP4, amax_in=torch.ones(1, device="cuda"))
    assert e.value.status == U.UFP4_ERR_INVALID
    y = torch.from_numpy(inputs.normal(42, (128, 48))).to(torch.bfloat16).cuda()
    with pytest.raises(U.UFP4Error) as e:                       # k not a multiple of 32
        U.ufp4_quantize(y, U.UFP4_MXFP4)
    assert e.value.status == U.UFP4_ERR_INVALID


def test_mx_nonfinite_flag(U):
    x = torch.from_numpy(inputs.normal(43, (64, 256))).to(torch.bfloat16).cuda()
    ws = U.workspace(x.device)
    x[3, 70] = float("nan")
    U.ufp4_quantize(x, U.UFP4_MXFP4, ws=ws)
    assert U.ufp4_check(ws) == U.UFP4_ERR_NONFINITE
    x[3, 70] = 1.0
    U.ufp4_quantize(x, U.UFP4_MXFP4, ws=ws, colwise=True)
    assert U.ufp4_check(ws) == U.UFP4_OK


def _mx_consumed(U, oracle, q):
    """fp64 values of a GPU MXFP4 operand (its codes and its per-32 scale
    bytes, one of the two 16-block places each), dequantized by the oracle."""
    torch.cuda.synchronize()
    codes = layouts.unpack_codes(q.codes.cpu().numpy(), q.rows, q.k)
    s16, _ = layouts.unpack_scales(q.scales.cpu().numpy(), q.rows, q.k)
    return oracle.dequantize_mx(codes, np.ascontiguousarray(s16[:, 0::2]))


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 200, 320), (130, 140, 4160), (64, 48, 32)])
def test_mx_gemm_matches_oracle(U, oracle, M, N, K):
    """C = A B^T of two MXFP4 operands on the tensor cores (E2M1 elements,
    UE8M0 scale per 32, scale_vec::2X) within 1e-5 relative Frobenius of the
    oracle's fp64 product of its own MX-dequantized operands (the codes and
    scales are bit-exact without the transform)."""
    a = inputs.normal(61, (M, K))
    b = inputs.normal(62, (N, K), std=0.02)
    qa = U.ufp4_quantize(torch.from_numpy(a).to(torch.bfloat16).cuda(), U.UFP4_MXFP4)
    qb = U.ufp4_quantize(torch.from_numpy(b).to(torch.bfloat16).cuda(), U.UFP4_MXFP4)
    c = U.ufp4_gemm(qa, qb).cpu().numpy().astype(np.float64)
    ra, rb = oracle.quantize_mx(a), oracle.quantize_mx(b)
    ref = oracle.gemm_f64(oracle.dequantize_mx(ra["codes"], ra["scales"]),
                          oracle.dequantize_mx(rb["codes"], rb["scales"]))
    assert np.linalg.norm(c - ref) <= 1e-5 * np.linalg.norm(ref)


def test_mx_training_gemms_and_rht(U, oracle):
    """fwd_y, bwd_dx (B column-wise) and bwd_dw (both column-wise, SR on dY)
    with MXFP4 operands, transform off against the oracle's operands and on
    against the operands the kernel consumed; and a spread of block
    exponents across 2^40 (rows scaled 2^-20 .. 2^20) that a per-tensor
    scale could not hold."""
    T, H, F = 192, 256, 320
    x = inputs.normal(63, (T, H))
    w = inputs.normal(64, (F, H), std=0.02)
    dy = inputs.normal(65, (T, F), std=1e-3)
    cases = ((x, w, False, False, 0), (dy, w, False, True, 1), (dy, x, True, True, 1))
    for rht in (False, True):
        for a, b, ca, cb, rnd in cases:
            qa = U.ufp4_quantize(torch.from_numpy(a).to(torch.bfloat16).cuda(), U.UFP4_MXFP4, rht=rht, rht_seed=2,
                                 colwise=ca, round=rnd, sr_seed=3)
            qb = U.ufp4_quantize(torch.from_numpy(b).to(torch.bfloat16).cuda(), U.UFP4_MXFP4, rht=rht, rht_seed=2,
                                 colwise=cb)
            c = U.ufp4_gemm(qa, qb).cpu().numpy().astype(np.float64)
            if not rht:
                ra = oracle.quantize_mx(a, colwise=ca, round_mode=rnd, sr_seed=3)
                rb = oracle.quantize_mx(b, colwise=cb)
                A = oracle.dequantize_mx(ra["codes"], ra["scales"])
                B = oracle.dequantize_mx(rb["codes"], rb["scales"])
            else:
                A, B = _mx_consumed(U, oracle, qa), _mx_consumed(U, oracle, qb)
            ref = oracle.gemm_f64(A, B)
            assert np.linalg.norm(c - ref) <= 1e-5 * np.linalg.norm(ref)
    wide = inputs.normal(66, (128, 256)) * np.float32(2.0) ** np.linspace(-20, 20, 128, dtype=np.float32)[:, None]
    wide = inputs.to_bf16_f32(wide)
    qa = U.ufp4_quantize(torch.from_numpy(wide).to(torch.bfloat16).cuda(), U.UFP4_MXFP4)
    qb = U.ufp4_quantize(torch.from_numpy(w[:, :256]).to(torch.bfloat16).cuda(), U.UFP4_MXFP4)
    c = U.ufp4_gemm(qa, qb).cpu().numpy().astype(np.float64)
    ref = oracle.gemm_f64(_mx_consumed(U, oracle, qa), _mx_consumed(U, oracle, qb))
    for r in (0, 64, 127):   # every row to 1e-5 of its own norm, small rows included
        assert np.linalg.norm(c[r] - ref[r]) <= 1e-5 * np.linalg.norm(ref[r])
