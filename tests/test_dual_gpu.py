"""GPU parity of the dual-orientation quantizer (ufp4_quantize_dual).

One read of X yields both the row-wise quantization of X and the column-wise
one (the quantization of X^T) that the three training GEMMs consume.  Each
result must equal the single-orientation path bit for bit (same kernels'
arithmetic, same tensor scale, SR numbering and padding), and, on a small
case, the CPU oracle directly: bit-exact with the transform off; with it on,
the bound of the single-orientation tests (codes within one grid step on at
most 1e-4 of the elements).
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


def _host(q):
    torch.cuda.synchronize()
    return (q.codes.cpu().numpy(), q.scales.cpu().numpy(), float(q.tensor_scale.item()))


def _assert_same(a, b):
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    assert a[2] == b[2]


def _single(U, x, grid, rht, rnd, sr_counter, colwise, amax=None):
    return _host(U.ufp4_quantize(x, grid, rht=rht, rht_seed=7, round=rnd, sr_seed=11, sr_counter=sr_counter,
                                 colwise=colwise, amax_in=amax))


DUAL_CASES = [(dt, grid, rht, rnd) for dt in (torch.bfloat16, torch.float32) for grid in (0, 1, 2)
              for rht in (False, True) for rnd in (0, 1)]


@pytest.mark.parametrize("dtype,grid,rht,rnd", DUAL_CASES)
@pytest.mark.parametrize("rows,cols", [(256, 1024), (272, 1040), (48, 4112)])
def test_dual_equals_single(U, dtype, grid, rht, rnd, rows, cols):
    # 272 x 1040: a ragged last column chunk, row count off the 128-row scale
    # tile, and a column-wise K (272) with a padding block; 48 x 4112: many
    # chunks per row block, few row blocks
    x = torch.from_numpy(inputs.normal(5 + rows, (rows, cols))).to(dtype).cuda()
    qr, qc = U.ufp4_quantize_dual(x, grid, rht=rht, rht_seed=7, round=rnd, sr_seed=11, sr_counter_row=3,
                                  sr_counter_col=4)
    _assert_same(_host(qr), _single(U, x, grid, rht, rnd, 3, False))
    _assert_same(_host(qc), _single(U, x, grid, rht, rnd, 4, True))


def test_dual_strided_input_and_partial_amax(U):
    # ld > cols (a view into a wider buffer), amax given for one orientation
    wide = torch.from_numpy(inputs.outlier(3, rows=512, cols=1536)["x"]).to(torch.bfloat16).cuda()
    x = wide[:, :1024]
    am = torch.tensor([float(x.float().abs().max()) * 2.0], device="cuda")
    qr, qc = U.ufp4_quantize_dual(x, 1, rht=True, rht_seed=7, amax_row=am)
    _assert_same(_host(qr), _single(U, x, 1, True, 0, 0, False, amax=am))
    _assert_same(_host(qc), _single(U, x, 1, True, 0, 0, True))


def test_dual_fallback_mixed_parameters(U):
    # different rounding per orientation: the call runs two single passes
    x = torch.from_numpy(inputs.normal(9, (128, 512))).to(torch.bfloat16).cuda()
    ws = U.workspace(x.device)
    out_r = U.QTensor.empty(128, 512, 0, x.device)
    out_c = U.QTensor.empty(512, 128, 0, x.device)
    import ctypes
    pr = U.qparams(0, True, 7, 0, 11, 0, False, None)
    pc = U.qparams(0, True, 7, 1, 11, 5, True, None)
    qr, qc = out_r.c(), out_c.c()
    st = U.lib().ufp4_quantize_dual(x.data_ptr(), 0, 128, 512, 512, ctypes.byref(pr), ctypes.byref(pc),
                                    ctypes.byref(qr), ctypes.byref(qc), ws.data_ptr(), ws.numel(), None)
    assert st == 0
    _assert_same(_host(out_r), _single(U, x, 0, True, 0, 0, False))
    _assert_same(_host(out_c), _single(U, x, 0, True, 1, 5, True))


@pytest.mark.parametrize("grid,rht,rnd", [(0, False, 0), (1, False, 1), (1, True, 0), (0, True, 1), (2, False, 1),
                                          (2, True, 0)])
def test_dual_matches_oracle(U, oracle, grid, rht, rnd):
    xn = inputs.smoke(0)["x"]   # 256 x 1024 N(0,1), BF16-representable
    x = torch.from_numpy(np.ascontiguousarray(xn)).to(torch.bfloat16).cuda()
    qr, qc = U.ufp4_quantize_dual(x, grid, rht=rht, rht_seed=2, round=rnd, sr_seed=1, sr_counter_row=0,
                                  sr_counter_col=1)
    for q, col, ctr in ((qr, False, 0), (qc, True, 1)):
        codes_b, scales_b, ts = _host(q)
        codes = layouts.unpack_codes(codes_b, q.rows, q.k)
        scales, spad = layouts.unpack_scales(scales_b, q.rows, q.k)
        assert not layouts.code_padding(codes_b, q.rows, q.k).any()
        assert not spad.any()
        r = oracle.quantize(xn, grid, rht=rht, rht_seed=2, round_mode=rnd, sr_seed=1, sr_counter=ctr, colwise=col)
        if not rht:
            np.testing.assert_array_equal(codes, r["codes"])
            np.testing.assert_array_equal(scales, r["scales"])
            assert ts == np.float32(r["tensor_scale"])
        else:
            si = lambda c: np.where(c.astype(np.int32) & 8, -(c.astype(np.int32) & 7), c.astype(np.int32) & 7)
            d = np.abs(si(codes) - si(r["codes"]))
            assert d.max() <= 1 and (d > 0).mean() <= 1e-4
            assert abs(ts / r["tensor_scale"] - 1) <= 1e-6


def test_dual_nonfinite_flag(U):
    x = torch.from_numpy(inputs.normal(4, (64, 256))).to(torch.bfloat16).cuda()
    x[5, 17] = float("inf")
    ws = U.workspace(x.device)
    U.ufp4_quantize_dual(x, 1, rht=True, ws=ws)
    assert U.ufp4_check(ws) == U.UFP4_ERR_NONFINITE
    y = torch.from_numpy(inputs.normal(4, (64, 256))).to(torch.bfloat16).cuda()
    U.ufp4_quantize_dual(y, 1, rht=True, ws=ws)
    assert U.ufp4_check(ws) == 0


@pytest.mark.parametrize("grid,rht,rnd", [(1, True, 0), (1, True, 1), (0, False, 0), (0, True, 1)])
@pytest.mark.parametrize("rows,cols", [(3584, 4864), (3584, 4928), (64, 128)])
def test_single_pass_capacity_boundary(U, grid, rht, rnd, rows, cols):
    """BF16 dual quantization with both tensor maxima computed: tensors of up
    to 14 x 128 x 64 tiles per SM (3584 x 4864 is 2128 tiles, the limit on
    152 SMs) take the single on-chip pass; one tile column more (3584 x 4928)
    the two-pass route.  Both equal the single-orientation calls bit for
    bit, and a repeated call (the grid-barrier counter is re-armed) too."""
    x = torch.from_numpy(inputs.normal(9, (rows, cols))).to(torch.bfloat16).cuda()
    kw = dict(rht=rht, rht_seed=7, round=rnd, sr_seed=11, sr_counter_row=3, sr_counter_col=4)
    qr, qc = U.ufp4_quantize_dual(x, grid, **kw)
    r1, c1 = _host(qr), _host(qc)
    _assert_same(r1, _single(U, x, grid, rht, rnd, 3, False))
    _assert_same(c1, _single(U, x, grid, rht, rnd, 4, True))
    qr2, qc2 = U.ufp4_quantize_dual(x, grid, **kw)
    _assert_same(_host(qr2), r1)
    _assert_same(_host(qc2), c1)
    assert U.ufp4_check(U.workspace(x.device)) == U.UFP4_OK
