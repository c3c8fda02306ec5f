"""GPU parity of the grouped (mixture-of-experts) quantization and GEMMs.

A small MoE layer with ragged, tiny and zero-token experts: X [sum T_e x H],
W [E * F x H] (expert e = rows eF..eF+F-1), dY [sum T_e x F].  Every segment
is checked against the oracle's per-segment quantization (bit-exact with RHT
off, within the RHT tolerance with it on), and the three grouped GEMMs
(fwd_y, bwd_dx, bwd_dw) against the oracle's fp64 per-expert products.
"""
import ctypes

import numpy as np
import pytest
import torch

from fp4_quantized_numerics_gb300 import inputs
from tests import layouts, parity

pytestmark = pytest.mark.gpu

COUNTS = [37, 0, 130, 5, 256, 64, 1]
H, F = 96, 80


@pytest.fixture(scope="module")
def U():
    from fp4_quantized_numerics_gb300 import build, ufp4
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return ufp4


def _data():
    g = np.random.default_rng(7)
    T = sum(COUNTS)
    x = inputs.to_bf16_f32(g.standard_normal((T, H), dtype=np.float32))
    w = inputs.to_bf16_f32(g.standard_normal((len(COUNTS) * F, H), dtype=np.float32) * np.float32(0.02))
    dy = inputs.to_bf16_f32(g.standard_normal((T, F), dtype=np.float32) * np.float32(1e-3))
    return x, w, dy


def _gpu_segments(U, q, seg_rows, colwise):
    """Per-segment (codes, scales, tensor_scale) views of a grouped QTensor."""
    torch.cuda.synchronize()
    codes = layouts.unpack_codes(q.codes.cpu().numpy(), q.rows, q.k)
    scales, _ = layouts.unpack_scales(q.scales.cpu().numpy(), q.rows, q.k)
    ts = q.tensor_scale.cpu().numpy()
    offs = U.grouped_offsets(seg_rows, colwise)
    out = []
    for e, T in enumerate(seg_rows):
        if T == 0:
            out.append(None)
            continue
        o = offs[e]
        if not colwise:
            out.append((codes[o:o + T], scales[o:o + T], float(ts[e])))
        else:
            t16 = (T + 15) // 16 * 16
            out.append((codes[:, o:o + t16], scales[:, o // 16:(o + t16) // 16], float(ts[e])))
    return out


def _check_segments(got, ref, rht):
    """Per segment bit-exact (RHT off); with RHT on, the code bar over the
    whole grouped tensor (every segment's codes counted together)."""
    tally = parity.CodeTally()
    for g, r in zip(got, ref):
        if r is None:
            assert g is None
            continue
        codes, scales, ts = g
        if not rht:
            np.testing.assert_array_equal(scales, r["scales"])
            np.testing.assert_array_equal(codes, r["codes"])
            assert ts == np.float32(r["tensor_scale"])
        else:
            assert abs(ts / r["tensor_scale"] - 1) <= 1e-6
            tally.add(codes, r["codes"])
    if rht:
        tally.check()


@pytest.mark.parametrize("grid", [0, 1, 2])
@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("colwise", [False, True])
def test_grouped_quantize_matches_oracle(U, oracle, grid, rht, colwise):
    x, w, dy = _data()
    for arr, seg, rnd in ((x, COUNTS, 0), (dy, COUNTS, 1), (w, [F] * len(COUNTS), 0)):
        t = torch.from_numpy(arr).to(torch.bfloat16).cuda()
        q = U.ufp4_quantize_grouped(t, grid, seg, rht=rht, rht_seed=2, round=rnd, sr_seed=3,
                                    colwise=colwise)
        got = _gpu_segments(U, q, seg, colwise)
        ref = oracle.quantize_grouped(arr, seg, grid, rht=rht, rht_seed=2, round_mode=rnd, sr_seed=3,
                                      colwise=colwise)
        _check_segments(got, ref, rht)


def _deq(oracle, r, grid):
    return oracle.dequantize(r["codes"], r["scales"], r["tensor_scale"], grid)


def _consumed_segments(U, oracle, q, seg_rows, colwise, grid):
    """Per segment dict(codes, scales, tensor_scale) of the GPU's grouped
    tensor, i.e. the operands the grouped GEMM consumes."""
    out = []
    for g in _gpu_segments(U, q, seg_rows, colwise):
        out.append(None if g is None else dict(codes=g[0], scales=g[1], tensor_scale=g[2]))
    return out


@pytest.mark.parametrize("grid", [0, 1])
@pytest.mark.parametrize("rht", [False, True])
def test_grouped_training_gemms(U, oracle, grid, rht):
    """fwd_y, bwd_dx and bwd_dw of every expert.  RHT off: against the
    oracle's own operands (bit-exact codes).  RHT on: the GPU's codes pass the
    code bar against the oracle's, and each GEMM is compared with the fp64
    product of the GPU operands it consumed."""
    x, w, dy = _data()
    E = len(COUNTS)
    tx, tw, tdy = (torch.from_numpy(a).to(torch.bfloat16).cuda() for a in (x, w, dy))
    wseg = [F] * E
    kw = dict(rht=rht, rht_seed=2)
    qx_r = U.ufp4_quantize_grouped(tx, grid, COUNTS, **kw)
    qx_c = U.ufp4_quantize_grouped(tx, grid, COUNTS, colwise=True, **kw)
    qdy_r = U.ufp4_quantize_grouped(tdy, grid, COUNTS, round=1, sr_seed=3, **kw)
    qdy_c = U.ufp4_quantize_grouped(tdy, grid, COUNTS, round=1, sr_seed=3, colwise=True, **kw)
    qw_r = U.ufp4_quantize_grouped(tw, grid, wseg, **kw)
    qw_c = U.ufp4_quantize_grouped(tw, grid, wseg, colwise=True, **kw)
    rx_r = oracle.quantize_grouped(x, COUNTS, grid, **kw)
    rx_c = oracle.quantize_grouped(x, COUNTS, grid, colwise=True, **kw)
    rdy_r = oracle.quantize_grouped(dy, COUNTS, grid, round_mode=1, sr_seed=3, **kw)
    rdy_c = oracle.quantize_grouped(dy, COUNTS, grid, round_mode=1, sr_seed=3, colwise=True, **kw)
    rw_r = oracle.quantize_grouped(w, wseg, grid, **kw)
    rw_c = oracle.quantize_grouped(w, wseg, grid, colwise=True, **kw)
    if rht:
        pairs = ((qx_r, rx_r, COUNTS, False), (qx_c, rx_c, COUNTS, True), (qdy_r, rdy_r, COUNTS, False),
                 (qdy_c, rdy_c, COUNTS, True), (qw_r, rw_r, wseg, False), (qw_c, rw_c, wseg, True))
        got = []
        for q, r, seg, col in pairs:
            g = _consumed_segments(U, oracle, q, seg, col, grid)
            _check_segments([None if t is None else (t["codes"], t["scales"], t["tensor_scale"]) for t in g],
                            r, True)
            got.append(g)
        rx_r, rx_c, rdy_r, rdy_c, rw_r, rw_c = got

    T = sum(COUNTS)
    y = torch.full((T, F), 9.0, device="cuda")
    dx = torch.full((T, H), 9.0, device="cuda")
    dw = torch.full((E * F, H), 9.0, device="cuda")
    xo = U.grouped_offsets(COUNTS, False)
    ko = U.grouped_offsets(COUNTS, True)
    wo = U.grouped_offsets(wseg, False)
    wk = U.grouped_offsets(wseg, True)
    starts = np.concatenate([[0], np.cumsum(COUNTS)])
    fy, fdx, fdw = [], [], []
    for e, Te in enumerate(COUNTS):
        s0 = int(starts[e])
        fy.append(dict(M=Te, N=F, K=H, a_row=xo[e], a_k=0, b_row=wo[e], b_k=0, a_seg=e, b_seg=e,
                       c=y[s0:s0 + Te] if Te else y[:1]))
        fdx.append(dict(M=Te, N=H, K=F, a_row=xo[e], a_k=0, b_row=0, b_k=wk[e], a_seg=e, b_seg=e,
                        c=dx[s0:s0 + Te] if Te else dx[:1]))
        k16 = (Te + 15) // 16 * 16
        fdw.append(dict(M=F, N=H, K=k16, a_row=0, a_k=ko[e], b_row=0, b_k=ko[e], a_seg=e, b_seg=e,
                        c=dw[e * F:(e + 1) * F]))
    U.ufp4_gemm_grouped(qx_r, qw_r, fy)
    U.ufp4_gemm_grouped(qdy_r, qw_c, fdx)
    U.ufp4_gemm_grouped(qdy_c, qx_c, fdw)
    torch.cuda.synchronize()
    y, dx, dw = y.cpu().numpy(), dx.cpu().numpy(), dw.cpu().numpy()
    for e, Te in enumerate(COUNTS):
        s0 = int(starts[e])
        if Te == 0:
            np.testing.assert_array_equal(dw[e * F:(e + 1) * F], 0.0)   # K = 0: zeros
            continue
        ref = oracle.gemm_f64(_deq(oracle, rx_r[e], grid), _deq(oracle, rw_r[e], grid))
        assert np.linalg.norm(y[s0:s0 + Te] - ref) <= 1e-5 * np.linalg.norm(ref)
        ref = oracle.gemm_f64(_deq(oracle, rdy_r[e], grid), _deq(oracle, rw_c[e], grid))
        assert np.linalg.norm(dx[s0:s0 + Te] - ref) <= 1e-5 * np.linalg.norm(ref)
        ref = oracle.gemm_f64(_deq(oracle, rdy_c[e], grid), _deq(oracle, rx_c[e], grid))
        assert np.linalg.norm(dw[e * F:(e + 1) * F] - ref) <= 1e-5 * np.linalg.norm(ref)
    # rows of y / dx that belong to no expert do not exist (sum T_e rows); all written
    assert not np.any(y == 9.0) and not np.any(dx == 9.0)


def _filled(U, rows, k, grid, n, dev="cuda"):
    """A grouped QTensor whose buffers hold a sentinel, so that any byte a
    call leaves unwritten shows up in the comparison."""
    q = U.QTensor.empty(rows, k, grid, dev)
    q.codes.fill_(0xA5)
    q.scales.fill_(0x5A)
    if q.eplane is not None:
        q.eplane.fill_(0x3C)
    q.tensor_scale = torch.full((max(n, 1),), -7.0, device=dev)
    return q


def _same(a, b):
    torch.cuda.synchronize()
    assert torch.equal(a.codes, b.codes)
    assert torch.equal(a.scales, b.scales)
    assert torch.equal(a.tensor_scale, b.tensor_scale)
    assert (a.eplane is None) == (b.eplane is None)
    if a.eplane is not None:
        assert torch.equal(a.eplane, b.eplane)


@pytest.mark.parametrize("counts,cols", [(COUNTS, H), ([128, 1, 0, 255, 129, 16, 200], 80),
                                         ([300], 208), ([0, 5], 32)])
@pytest.mark.parametrize("grid", [0, 1, 2])
@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("rnd", [0, 1])
def test_grouped_dual_equals_two_grouped_calls(U, grid, rht, rnd, counts, cols):
    """ufp4_quantize_grouped_dual (segment-aligned 128 x 64 tiles, one read per
    pass) gives each orientation bit for bit what its own
    ufp4_quantize_grouped call gives: codes, scales, correction planes, every
    segment's tensor scale, padding rows and blocks (segments of 1, 16, 128,
    129, 255 rows, empty ones, column counts off the 64-column tile)."""
    g = np.random.default_rng(11)
    T = sum(counts)
    x = inputs.to_bf16_f32(g.standard_normal((T, cols), dtype=np.float32) *
                           np.float32(2.0) ** g.integers(-3, 4, size=(T, 1)).astype(np.float32))
    t = torch.from_numpy(x).to(torch.bfloat16).cuda()
    n = len(counts)
    kw = dict(rht=rht, rht_seed=5, round=rnd, sr_seed=9)
    rr, kc = U.grouped_rows(counts), U.grouped_kpad(counts)
    dr, dc = _filled(U, rr, cols, grid, n), _filled(U, cols, kc, grid, n)
    U.ufp4_quantize_grouped_dual(t, grid, counts, sr_counter_row=3, sr_counter_col=4, out_row=dr, out_col=dc, **kw)
    sr, sc = _filled(U, rr, cols, grid, n), _filled(U, cols, kc, grid, n)
    U.ufp4_quantize_grouped(t, grid, counts, sr_counter=3, out=sr, **kw)
    U.ufp4_quantize_grouped(t, grid, counts, sr_counter=4, colwise=True, out=sc, **kw)
    _same(dr, sr)
    _same(dc, sc)
    assert U.ufp4_check() == U.UFP4_OK


@pytest.mark.parametrize("rht", [False, True])
def test_grouped_dual_matches_oracle(U, oracle, rht):
    """The grouped dual call against the oracle's per-segment quantization
    (dY-like input with SR): bit-exact without the transform, the code bar
    with it."""
    x, w, dy = _data()
    t = torch.from_numpy(dy).to(torch.bfloat16).cuda()
    qr, qc = U.ufp4_quantize_grouped_dual(t, 1, COUNTS, rht=rht, rht_seed=2, round=1, sr_seed=3)
    for q, col in ((qr, False), (qc, True)):
        got = _gpu_segments(U, q, COUNTS, col)
        ref = oracle.quantize_grouped(dy, COUNTS, 1, rht=rht, rht_seed=2, round_mode=1, sr_seed=3, colwise=col)
        _check_segments(got, ref, rht)


def test_grouped_dual_nonfinite_flag(U):
    """A NaN in one segment raises the workspace's non-finite flag."""
    x = torch.zeros(200, 64, dtype=torch.bfloat16, device="cuda")
    x[150, 3] = float("nan")
    ws = U.workspace()
    U.ufp4_quantize_grouped_dual(x, 1, [100, 100], ws=ws)
    assert U.ufp4_check(ws) == U.UFP4_ERR_NONFINITE
    U.ufp4_quantize_grouped_dual(torch.ones(200, 64, dtype=torch.bfloat16, device="cuda"), 1, [100, 100], ws=ws)
    assert U.ufp4_check(ws) == U.UFP4_OK


@pytest.mark.parametrize("case", ["fp32", "mixed_round", "mixed_rht"])
def test_grouped_dual_two_call_route(U, case):
    """Where one read cannot serve both orientations (FP32 input, different
    rounding modes or transforms) the grouped dual call runs the two grouped
    quantizations in turn: each result still equals its own call."""
    counts = [37, 0, 130, 5]
    g = np.random.default_rng(13)
    x = inputs.to_bf16_f32(g.standard_normal((sum(counts), 96), dtype=np.float32))
    dtype = torch.float32 if case == "fp32" else torch.bfloat16
    t = torch.from_numpy(x).to(dtype).cuda()
    n = len(counts)
    rr, kc = U.grouped_rows(counts), U.grouped_kpad(counts)
    dr, dc = _filled(U, rr, 96, 1, n), _filled(U, 96, kc, 1, n)
    pr = U.qparams(1, True, 2, 0, 3, 0, False)
    pc = U.qparams(1, case != "mixed_rht", 2, 1 if case == "mixed_round" else 0, 3, 0, True)
    qr, qc = dr.c(), dc.c()
    ws = U.workspace()
    st = U.lib().ufp4_quantize_grouped_dual(t.data_ptr(), U._dtype_code(t), 96, t.stride(0), U._i64_array(counts), n,
                                            ctypes.byref(pr), ctypes.byref(pc), ctypes.byref(qr), ctypes.byref(qc),
                                            ws.data_ptr(), ws.numel(), U._stream(None))
    assert st == U.UFP4_OK
    sr, sc = _filled(U, rr, 96, 1, n), _filled(U, 96, kc, 1, n)
    U.ufp4_quantize_grouped(t, 1, counts, rht=True, rht_seed=2, sr_seed=3, out=sr)
    U.ufp4_quantize_grouped(t, 1, counts, rht=case != "mixed_rht", rht_seed=2,
                            round=1 if case == "mixed_round" else 0, sr_seed=3, colwise=True, out=sc)
    _same(dr, sr)
    _same(dc, sc)
