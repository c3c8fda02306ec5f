"""GPU parity of the fused (RHT +) quantizer against the CPU oracle.

Acceptance bar (bit-exact where the arithmetic is defined to the bit):
  * RHT off: codes, block scales and the tensor scale identical to the
    oracle, RTNE and SR (same seed and counter), both grids, both
    orientations, BF16 and FP32 inputs; padding bytes zero.
  * RHT on: the fp32 butterflies round differently from the oracle's fp64
    transform, so at most 1e-4 of the codes may differ, each by one grid
    step; the tensor scale agrees to 1e-6 relative.
"""
import numpy as np
import pytest
import torch

from fp4_quantized_numerics_gb300 import inputs
from tests import layouts, parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def U():
    from fp4_quantized_numerics_gb300 import build, ufp4
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return ufp4


def _gpu_quant(U, x, grid, rht, rnd, colwise, dtype=torch.bfloat16, sr_seed=1, sr_counter=0,
               amax_in=None):
    xt = torch.from_numpy(np.ascontiguousarray(x)).to(dtype).cuda()
    esz = 2 if dtype == torch.bfloat16 else 4
    if (xt.shape[1] * esz) % 16:   # the ABI wants 16-byte row strides: pad ld
        ld = (xt.shape[1] * esz + 15) // 16 * 16 // esz
        wide = torch.zeros(xt.shape[0], ld, dtype=dtype, device="cuda")
        wide[:, : xt.shape[1]] = xt
        xt = wide[:, : xt.shape[1]]
    am = None if amax_in is None else torch.tensor([amax_in], dtype=torch.float32, device="cuda")
    q = U.ufp4_quantize(xt, grid, rht=rht, rht_seed=2, round=rnd, sr_seed=sr_seed,
                        sr_counter=sr_counter, colwise=colwise, amax_in=am)
    torch.cuda.synchronize()
    codes_b = q.codes.cpu().numpy()
    codes = layouts.unpack_codes(codes_b, q.rows, q.k)
    cpad = layouts.code_padding(codes_b, q.rows, q.k)
    scales, spad = layouts.unpack_scales(q.scales.cpu().numpy(), q.rows, q.k)
    return dict(codes=codes, scales=scales, tensor_scale=float(q.tensor_scale.item()),
                cpad=cpad, spad=spad, q=q, xt=xt)


def _signed_index(codes):
    c = codes.astype(np.int32)
    return np.where(c & 8, -(c & 7), c & 7)


def _compare(g, r, rht):
    assert not g["cpad"].any(), "code padding must be zero"
    assert not g["spad"].any(), "scale padding must be zero"
    if not rht:
        np.testing.assert_array_equal(g["scales"], r["scales"])
        np.testing.assert_array_equal(g["codes"], r["codes"])
        assert g["tensor_scale"] == np.float32(r["tensor_scale"])
    else:
        assert abs(g["tensor_scale"] / r["tensor_scale"] - 1) <= 1e-6
        parity.assert_codes_close(g["codes"], r["codes"])
        assert (g["scales"] != r["scales"]).mean() <= 1e-3


# grid 2 = clamped E2M1 ({0, .5, 1, 1.5, 2}, the pages' failed uniform-grid ablation)
CASES = [(grid, rht, rnd, col) for grid in (0, 1, 2) for rht in (False, True)
         for rnd in (0, 1) for col in (False, True)]


@pytest.mark.parametrize("grid,rht,rnd,col", CASES)
def test_smoke_config_all_modes(U, oracle, grid, rht, rnd, col):
    x = inputs.smoke(0)["x"]
    g = _gpu_quant(U, x, grid, rht, rnd, col)
    r = oracle.quantize(x, grid, rht=rht, rht_seed=2, round_mode=rnd, sr_seed=1, sr_counter=0,
                        colwise=col)
    _compare(g, r, rht)


@pytest.mark.parametrize("shape,col", [((300, 80), False), ((37, 208), False), ((48, 12), True),
                                       ((144, 260), True), ((16, 16), False), ((16, 4), True)])
@pytest.mark.parametrize("grid", [0, 1, 2])
def test_ragged_shapes(U, oracle, shape, col, grid):
    x = inputs.normal(31, shape)
    for rht in (False, True):
        for rnd in (0, 1):
            g = _gpu_quant(U, x, grid, rht, rnd, col)
            r = oracle.quantize(x, grid, rht=rht, rht_seed=2, round_mode=rnd, sr_seed=1, colwise=col)
            _compare(g, r, rht)


@pytest.mark.parametrize("grid", [0, 1, 2])
def test_fp32_input(U, oracle, grid):
    x = np.random.default_rng(5).standard_normal((96, 160)).astype(np.float32)
    for col in (False, True):
        for rnd in (0, 1):
            g = _gpu_quant(U, x, grid, False, rnd, col, dtype=torch.float32)
            r = oracle.quantize(x, grid, round_mode=rnd, sr_seed=1, colwise=col)
            _compare(g, r, False)


@pytest.mark.parametrize("grid", [0, 1, 2])
def test_outlier_config(U, oracle, grid):
    x = inputs.outlier(0)["x"]
    for rht in (False, True):
        g = _gpu_quant(U, x, grid, rht, 0, False)
        r = oracle.quantize(x, grid, rht=rht, rht_seed=2)
        _compare(g, r, rht)


def test_amax_in_and_special_tensors(U, oracle):
    x = inputs.normal(32, (64, 64))
    for grid in (0, 1, 2):
        g = _gpu_quant(U, x, grid, False, 0, False, amax_in=3.0)
        r = oracle.quantize(x, grid, amax_in=3.0)
        _compare(g, r, False)
    z = np.zeros((32, 64), np.float32)
    g = _gpu_quant(U, z, 1, True, 0, False)
    assert not g["codes"].any() and not g["scales"].any() and g["tensor_scale"] == 1.0
    s = np.zeros((32, 64), np.float32)
    s[3, 40] = -2.5
    g = _gpu_quant(U, s, 0, False, 0, False)
    r = oracle.quantize(s, 0)
    _compare(g, r, False)


def test_sr_reproducible_and_counter_sensitive(U):
    x = inputs.normal(33, (128, 256), std=1e-3)
    a = _gpu_quant(U, x, 1, True, 1, False, sr_seed=3, sr_counter=7)
    b = _gpu_quant(U, x, 1, True, 1, False, sr_seed=3, sr_counter=7)
    c = _gpu_quant(U, x, 1, True, 1, False, sr_seed=3, sr_counter=8)
    np.testing.assert_array_equal(a["codes"], b["codes"])
    assert (a["codes"] != c["codes"]).any()


def test_sr_large_counter_and_seed_bits(U, oracle):
    x = inputs.normal(34, (64, 128))
    seed, ctr = 0xDEADBEEF12345678, 0x0123456789ABCDEF
    g = _gpu_quant(U, x, 0, False, 1, True, sr_seed=seed, sr_counter=ctr)
    r = oracle.quantize(x, 0, round_mode=1, sr_seed=seed, sr_counter=ctr, colwise=True)
    _compare(g, r, False)


def test_nonfinite_input_is_reported(U):
    x = torch.randn(64, 64, device="cuda").to(torch.bfloat16)
    ws = torch.empty(U.lib().ufp4_workspace_bytes(), dtype=torch.uint8, device="cuda")
    U.ufp4_quantize(x, 0, ws=ws)
    assert U.ufp4_check(ws) == U.UFP4_OK
    x[5, 7] = float("nan")
    U.ufp4_quantize(x, 0, ws=ws)
    assert U.ufp4_check(ws) == U.UFP4_ERR_NONFINITE
    x[5, 7] = float("inf")
    U.ufp4_quantize(x, 1, rht=True, ws=ws)
    assert U.ufp4_check(ws) == U.UFP4_ERR_NONFINITE
    x[5, 7] = 1.0
    U.ufp4_quantize(x, 1, colwise=True, ws=ws)
    assert U.ufp4_check(ws) == U.UFP4_OK


@pytest.mark.parametrize("grid", [0, 1, 2])
def test_dequantize_matches_oracle(U, oracle, grid):
    """Codes from the RHT-off path are bit-exact, so both sides decode the
    same codes; the inverse transform (fp32 butterflies vs fp64) must agree
    to 1e-6 relative."""
    x = inputs.normal(35, (130, 96))
    g = _gpu_quant(U, x, grid, False, 0, False)
    r = oracle.quantize(x, grid)
    out = U.ufp4_dequantize(g["q"]).cpu().numpy()
    ref = oracle.dequantize(r["codes"], r["scales"], r["tensor_scale"], grid)
    np.testing.assert_array_equal(out, ref.astype(np.float32))
    out = U.ufp4_dequantize(g["q"], inverse_rht=True, rht_seed=2).cpu().numpy()
    ref = oracle.dequantize(r["codes"], r["scales"], r["tensor_scale"], grid, inverse_rht=True,
                            rht_seed=2)
    assert np.linalg.norm(out - ref) / np.linalg.norm(ref) <= 1e-6
    assert np.abs(out - ref).max() <= 1e-6 * np.abs(ref).max()


@pytest.mark.parametrize("grid", [0, 1, 2])
def test_stats_match_oracle(U, oracle, grid):
    x = inputs.smoke(0)["x"]
    for rht in (False, True):
        for col in (False, True):
            g = _gpu_quant(U, x, grid, rht, 0, col)
            st = U.ufp4_stats(g["xt"], g["q"], rht=rht, rht_seed=2, colwise=col)
            r = oracle.quantize(x, grid, rht=rht, rht_seed=2, colwise=col)
            ro = oracle.stats(r["y"], r["codes"], r["scales"], r["tensor_scale"], grid)
            tol = 1.0 if not rht else 10.0   # RHT: <= 1e-4 of codes may differ by a step
            assert abs(st["alpha"] - ro["alpha"]) <= 1e-6 * tol
            assert abs(st["sqnr_db"] - ro["sqnr_db"]) <= 1e-4 * tol
            assert abs(st["mean_bias"] - ro["mean_bias"]) <= 1e-5 * tol
            if not rht:
                assert st["bias_count"] == ro["bias_count"]


def _strided(x, dtype, extra):
    """x as a view whose rows sit `extra` elements apart beyond its width:
    16-byte aligned rows that are not 32-byte aligned when extra * esz = 16."""
    xt = torch.from_numpy(np.ascontiguousarray(x)).to(dtype).cuda()
    wide = torch.zeros(x.shape[0], x.shape[1] + extra, dtype=dtype, device="cuda")
    wide[:, : x.shape[1]] = xt
    return wide[:, : x.shape[1]]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("colwise", [False, True])
def test_rows_16_byte_aligned_only(U, oracle, dtype, rht, colwise):
    """The ABI asks only for 16-byte aligned rows: a row stride of 8 BF16 / 4
    FP32 elements beyond a 32-byte multiple puts every odd row off a 32-byte
    boundary.  Quantization, dual quantization, grouped quantization and
    stats must all read such inputs (RHT off: bit-exact)."""
    esz = 2 if dtype == torch.bfloat16 else 4
    x = inputs.normal(71, (96, 128))
    xs = _strided(x, dtype, 16 // esz)
    assert (xs.stride(0) * esz) % 32 == 16
    q = U.ufp4_quantize(xs, 1, rht=rht, rht_seed=2, colwise=colwise)
    torch.cuda.synchronize()
    got = dict(codes=layouts.unpack_codes(q.codes.cpu().numpy(), q.rows, q.k),
               scales=layouts.unpack_scales(q.scales.cpu().numpy(), q.rows, q.k)[0],
               tensor_scale=float(q.tensor_scale.item()),
               cpad=layouts.code_padding(q.codes.cpu().numpy(), q.rows, q.k),
               spad=layouts.unpack_scales(q.scales.cpu().numpy(), q.rows, q.k)[1])
    ref = oracle.quantize(x, 1, rht=rht, rht_seed=2, colwise=colwise)
    _compare(got, ref, rht)
    st = U.ufp4_stats(xs, q, rht=rht, rht_seed=2, colwise=colwise)
    rs = oracle.stats(ref["y"], ref["codes"], ref["scales"], ref["tensor_scale"], 1)
    if not rht:   # the statistics kernels sum fp32 partials (as test_stats_match_oracle allows)
        assert abs(st["alpha"] - rs["alpha"]) <= 1e-6
        assert st["bias_count"] == rs["bias_count"]
    if not colwise:
        qr, qc = U.ufp4_quantize_dual(xs, 1, rht=rht, rht_seed=2)
        torch.cuda.synchronize()
        assert torch.equal(qr.codes, q.codes) and torch.equal(qr.scales, q.scales)
        counts = [37, 0, 59]
        qg = U.ufp4_quantize_grouped(xs, 1, counts, rht=rht, rht_seed=2)
        torch.cuda.synchronize()
        gc = layouts.unpack_codes(qg.codes.cpu().numpy(), qg.rows, qg.k)
        rg = oracle.quantize_grouped(x, counts, 1, rht=rht, rht_seed=2)
        for e, off in ((0, 0), (2, 128)):
            if not rht:
                np.testing.assert_array_equal(gc[off:off + counts[e]], rg[e]["codes"])
            else:
                parity.assert_codes_close(gc[off:off + counts[e]], rg[e]["codes"])


@pytest.mark.parametrize("grid", [0, 1, 2])
@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("layout", ["bf16", "fp32", "strided", "colwise"])
def test_quantize_stats_fused(U, oracle, grid, rht, layout):
    """ufp4_quantize_stats: the quantized tensor is ufp4_quantize's bit for
    bit; the statistics agree with ufp4_stats (separate pass) and with the
    oracle's.  BF16 / FP32 contiguous row-wise take the one-pass kernel; the
    strided and column-wise layouts the two-pass route."""
    dtype = torch.float32 if layout == "fp32" else torch.bfloat16
    x = inputs.normal(72, (512, 768)) if dtype == torch.bfloat16 else \
        inputs.rng(72).standard_normal((512, 768), dtype=np.float32)
    xt = _strided(x, dtype, 8) if layout == "strided" else torch.from_numpy(x).to(dtype).cuda()
    col = layout == "colwise"
    rnd = 1 if grid == 1 else 0
    kw = dict(rht=rht, rht_seed=2, round=rnd, sr_seed=5, colwise=col)
    q, st = U.ufp4_quantize_stats(xt, grid, **kw)
    q0 = U.ufp4_quantize(xt, grid, **kw)
    s0 = U.ufp4_stats(xt, q0, **kw)
    torch.cuda.synchronize()
    for f in ("codes", "scales", "tensor_scale"):
        assert torch.equal(getattr(q, f), getattr(q0, f)), f
    assert torch.equal(q.eplane, q0.eplane) if q.eplane is not None else True
    assert st["bias_count"] == s0["bias_count"]
    assert abs(st["alpha"] - s0["alpha"]) <= 1e-6
    assert abs(st["sqnr_db"] - s0["sqnr_db"]) <= 1e-4
    assert abs(st["mean_bias"] - s0["mean_bias"]) <= 1e-5
    r = oracle.quantize(x, grid, rht=rht, rht_seed=2, round_mode=rnd, sr_seed=5, colwise=col)
    ro = oracle.stats(r["y"], r["codes"], r["scales"], r["tensor_scale"], grid)
    assert abs(st["alpha"] - ro["alpha"]) <= 1e-5
    assert abs(st["sqnr_db"] - ro["sqnr_db"]) <= 1e-3
