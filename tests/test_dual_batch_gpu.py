"""GPU parity of the batched dual quantization (ufp4_quantize_dual_batch).

A training step quantizes its operands one after another; the batch call
runs the amax pass of one tensor inside the quantization launch of the
tensor before it (k_dual_tile_amax: CTAs that finish their share of the
amax chunks join the quantization tiles through a shared counter).  Every
result must equal the tensor's own ufp4_quantize_dual bit for bit -- codes,
scales, E1M2 correction plane and tensor scale -- whatever the route of each
tensor (folded amax, separate amax pass, amax given, on-chip single pass,
FP32 staged kernels), and, sampled, the CPU oracle.

Sizes: a tensor takes the two-pass tile route (and so can have its amax
folded) when it has more than 14 x 152 = 2128 tiles of 128 x 64, e.g.
3584 x 4928; smaller ones with both maxima to compute take the on-chip
single pass.
"""
import numpy as np
import pytest
import torch

from tests import layouts

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def U():
    from fp4_quantized_numerics_gb300 import build, ufp4
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return ufp4


def _x(seed, rows, cols, dtype=torch.bfloat16, std=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(rows, cols, generator=g, device="cuda") * std).to(dtype)


def _host(q):
    torch.cuda.synchronize()
    ep = None if q.eplane is None else q.eplane.cpu().numpy()
    return q.codes.cpu().numpy(), q.scales.cpu().numpy(), float(q.tensor_scale.item()), ep


def _assert_same(a, b, what):
    np.testing.assert_array_equal(a[0], b[0], err_msg=what + " codes")
    np.testing.assert_array_equal(a[1], b[1], err_msg=what + " scales")
    assert a[2] == b[2], what + " tensor scale"
    assert (a[3] is None) == (b[3] is None)
    if a[3] is not None:
        np.testing.assert_array_equal(a[3], b[3], err_msg=what + " correction plane")


def _dual_kw(job):
    return {k: v for k, v in job.items() if k not in ("x", "grid")}


def _check_batch(U, jobs):
    """The batch's results against one ufp4_quantize_dual per job."""
    ws = U.workspace(jobs[0]["x"].device)
    outs = U.ufp4_quantize_dual_batch(jobs, ws=ws)
    assert U.ufp4_check(ws) == U.UFP4_OK
    got = [(_host(r), _host(c)) for r, c in outs]
    for i, job in enumerate(jobs):
        r, c = U.ufp4_quantize_dual(job["x"], job["grid"], ws=ws, **_dual_kw(job))
        _assert_same(got[i][0], _host(r), "job %d row-wise" % i)
        _assert_same(got[i][1], _host(c), "job %d column-wise" % i)
    return outs


def test_training_step_operands(U):
    """dY (SR, the arithmetic-heavy pass) first, then X (its amax pass runs
    inside dY's quantization launch), then W (on-chip single pass)."""
    dy = _x(1, 3584, 4928, std=1e-3)
    x = _x(2, 3584, 4928)
    w = _x(3, 512, 4928, std=0.02)
    common = dict(grid=1, rht=True, rht_seed=5)
    _check_batch(U, [dict(x=dy, round=1, sr_seed=3, sr_counter_row=1, sr_counter_col=2, **common),
                     dict(x=x, **common), dict(x=w, **common)])


@pytest.mark.parametrize("grid,rnd", [(0, 0), (0, 1), (1, 0), (2, 1)])
def test_chain_of_three_ragged(U, grid, rnd):
    """Three tile-route tensors, each needing its maxima: two folded amax
    passes (the partial areas alternate).  Ragged shapes: row counts off the
    128-row tile, column counts (multiples of 16, as row-wise blocks need)
    off the 64-column tile and the 512-column amax chunk; the quantized
    tensor's grid and rounding vary."""
    a = _x(4, 3600, 4944)   # 29 x 78 = 2262 tiles
    b = _x(5, 4112, 4432, std=3.0)   # 33 x 70 = 2310 tiles
    c = _x(6, 2336, 7472)   # 19 x 117 = 2223 tiles
    kw = dict(grid=grid, rht=True, rht_seed=9)
    _check_batch(U, [dict(x=a, round=rnd, sr_seed=7, sr_counter_row=5, **kw), dict(x=b, round=rnd, sr_seed=8, **kw),
                     dict(x=c, **kw)])


def test_routes_that_do_not_fold(U):
    """Given maxima, a next tensor without the transform (its amax pass is
    not the tensor-core one), an FP32 tensor and a resident one in between:
    each keeps its own route and the results still equal single calls."""
    a = _x(7, 3584, 4928)
    b = _x(8, 3584, 4928)
    c = _x(9, 3584, 4928)
    d = _x(10, 256, 1024, dtype=torch.float32)
    e = _x(11, 3584, 4928)
    am = torch.tensor([float(a.float().abs().max()) * 0.5], device="cuda")   # saturating caller amax
    jobs = [dict(x=a, grid=1, rht=True, rht_seed=3, amax_row=am, amax_col=am),   # needs no amax pass
            dict(x=b, grid=1, rht=True, rht_seed=3, amax_col=am),                # folded (row maximum missing)
            dict(x=c, grid=1, rht=False),                                        # not folded: no transform
            dict(x=d, grid=0, rht=True, rht_seed=3),                             # FP32: staged kernels
            dict(x=e, grid=0, rht=True, rht_seed=3, round=1, sr_seed=2)]         # after FP32: own amax pass
    _check_batch(U, jobs)


def test_unbalanced_pairs(U):
    """Folded pairs whose two kinds of work differ a lot in size, so that the
    CTAs of one kind run out early and finish the other kind's work: a tiny
    quantization (maxima given, so it takes the tile route) before a large
    amax pass, and a large quantization before a tiny amax pass (a small
    tensor with one maximum given takes the tile route too)."""
    a = _x(18, 128, 256)
    b = _x(19, 3584, 4928)
    c = _x(20, 3584, 4928)
    d = _x(21, 64, 128)
    am = torch.tensor([40.0], device="cuda")
    _check_batch(U, [dict(x=a, grid=1, rht=True, amax_row=am, amax_col=am), dict(x=b, grid=1, rht=True),
                     dict(x=c, grid=0, rht=True, round=1, sr_seed=6), dict(x=d, grid=1, rht=True, amax_row=am)])


def test_nonfinite_flag_covers_every_job(U):
    """The flag is cleared once per batch and raised by any job."""
    ws = U.workspace("cuda")
    a, b = _x(12, 3584, 4928), _x(13, 3584, 4928)
    jobs = [dict(x=a, grid=1, rht=True, round=1), dict(x=b, grid=1, rht=True)]
    for bad in (0, 1):
        t = (a, b)[bad]
        keep = t[100, 200].clone()
        t[100, 200] = float("nan")
        U.ufp4_quantize_dual_batch(jobs, ws=ws)
        assert U.ufp4_check(ws) == U.UFP4_ERR_NONFINITE, bad
        t[100, 200] = keep
        U.ufp4_quantize_dual_batch(jobs, ws=ws)
        assert U.ufp4_check(ws) == U.UFP4_OK, bad


def test_repeated_batches_agree(U):
    """The shared tile counter hands tiles to whichever CTA asks first; the
    results must not depend on that (ten batches, bit-identical)."""
    dy, x = _x(14, 3584, 4928, std=1e-3), _x(15, 3584, 4928)
    jobs = [dict(x=dy, grid=1, rht=True, round=1, sr_seed=4), dict(x=x, grid=1, rht=True)]
    first = [(_host(r), _host(c)) for r, c in U.ufp4_quantize_dual_batch(jobs)]
    for _ in range(10):
        again = [(_host(r), _host(c)) for r, c in U.ufp4_quantize_dual_batch(jobs)]
        for i in range(2):
            _assert_same(again[i][0], first[i][0], "row-wise %d" % i)
            _assert_same(again[i][1], first[i][1], "column-wise %d" % i)


def test_batch_matches_oracle_sampled(U, oracle):
    """The folded tensor's results against the oracle on sampled rows: the
    oracle quantizes the sampled rows of x (row-wise) and of x^T
    (column-wise) with the tensor amax of the whole rotated tensor, which it
    also computes; codes within one grid step on at most 1e-4 of the
    elements (the transform's bar), scales within one E4M3 step where a code
    differs, tensor scale within 1e-6."""
    dy, x = _x(16, 3584, 4928, std=1e-3), _x(17, 3584, 4928)
    jobs = [dict(x=dy, grid=1, rht=True, rht_seed=2, round=1, sr_seed=1), dict(x=x, grid=1, rht=True, rht_seed=2)]
    (_, _), (qr, qc) = U.ufp4_quantize_dual_batch(jobs)
    xn = x.float().cpu().numpy()
    A = {col: float(oracle.tensor_amax(xn, rht=True, rht_seed=2, colwise=col)) for col in (False, True)}
    rng = np.random.default_rng(0)
    for q, col in ((qr, False), (qc, True)):
        codes_b, scales_b, ts, _ = _host(q)
        codes = layouts.unpack_codes(codes_b, q.rows, q.k)
        scales, _ = layouts.unpack_scales(scales_b, q.rows, q.k)
        t = xn.T if col else xn
        rows = rng.choice(q.rows, 24, replace=False)
        r = oracle.quantize(np.ascontiguousarray(t[rows]), 1, rht=True, rht_seed=2, amax_in=A[col])
        si = lambda c: np.where(c.astype(np.int32) & 8, -(c.astype(np.int32) & 7), c.astype(np.int32) & 7)
        d = np.abs(si(codes[rows]) - si(r["codes"]))
        assert d.max() <= 1 and (d > 0).mean() <= 1e-4
        assert abs(ts / r["tensor_scale"] - 1) <= 1e-6
        ds = np.abs(scales[rows].astype(np.int32) - r["scales"].astype(np.int32))
        assert ds.max() <= 1 and (ds > 0).mean() <= 1e-3
