"""GPU checks of the E1M2 correction plane (ufp4_qtensor.eplane).

An E1M2 value m/2 is (R + E)/2 with R the code's nibble read as an E2M1 code
and E the plane's nibble read as an E2M1 code (include/ufp4.h).  The plane
that every quantize path writes must satisfy that identity nibble by nibble
(same sign bit, E2M1(m) + E2M1(e) = m), including the zero padding; and the
GEMM that loads the planes must give the bits of the GEMM that expands them
on chip (which the GEMM parity tests pin to the oracle).
"""
import numpy as np
import pytest
import torch

from fp4_quantized_numerics_gb300 import inputs

pytestmark = pytest.mark.gpu

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


@pytest.fixture(scope="module")
def U():
    from fp4_quantized_numerics_gb300 import build, ufp4
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return ufp4


def _nibbles(buf):
    b = buf.cpu().numpy().astype(np.int32)
    return np.stack([b & 15, b >> 4], axis=-1).reshape(-1)


def _check_plane(q):
    assert q.eplane is not None and q.eplane.numel() == q.codes.numel()
    torch.cuda.synchronize()
    c, e = _nibbles(q.codes), _nibbles(q.eplane)
    np.testing.assert_array_equal(c & 8, e & 8)                     # sign kept
    np.testing.assert_array_equal(E2M1[c & 7] + E2M1[e & 7], (c & 7).astype(np.float64))
    assert ((c & 7) > 0).mean() > 0.3                                # not a trivially zero tensor


def _strip(U, q):
    """The same quantized tensor without its plane (the GEMM then expands on chip)."""
    s = U.QTensor(q.codes, q.scales, q.tensor_scale, q.rows, q.k, q.grid)
    if hasattr(q, "seg_rows"):
        s.seg_rows = q.seg_rows
    return s


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rht,rnd", [(False, 0), (True, 0), (True, 1), (False, 1)])
@pytest.mark.parametrize("colwise", [False, True])
@pytest.mark.parametrize("rows,cols", [(256, 1024), (272, 1040), (48, 4112)])
def test_single_plane(U, dtype, rht, rnd, colwise, rows, cols):
    x = torch.from_numpy(inputs.normal(60 + rows, (rows, cols))).to(dtype).cuda()
    q = U.ufp4_quantize(x, U.UFP4_E1M2, rht=rht, rht_seed=7, round=rnd, sr_seed=5, colwise=colwise)
    _check_plane(q)
    # the plane does not change the codes or scales
    q0 = U.ufp4_quantize(x, U.UFP4_E1M2, rht=rht, rht_seed=7, round=rnd, sr_seed=5, colwise=colwise,
                         out=U.QTensor.empty(q.rows, q.k, U.UFP4_E1M2, x.device, eplane=False))
    assert q0.eplane is None
    torch.cuda.synchronize()
    assert torch.equal(q0.codes, q.codes) and torch.equal(q0.scales, q.scales)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rht,rnd", [(False, 0), (True, 0), (True, 1)])
@pytest.mark.parametrize("rows,cols", [(256, 1024), (272, 1040)])
def test_dual_planes(U, dtype, rht, rnd, rows, cols):
    x = torch.from_numpy(inputs.normal(70 + rows, (rows, cols))).to(dtype).cuda()
    qr, qc = U.ufp4_quantize_dual(x, U.UFP4_E1M2, rht=rht, rht_seed=7, round=rnd, sr_seed=5,
                                  sr_counter_row=1, sr_counter_col=2)
    _check_plane(qr)
    _check_plane(qc)


@pytest.mark.parametrize("colwise", [False, True])
def test_grouped_planes(U, colwise):
    counts = [100, 0, 37, 256, 16]
    x = torch.from_numpy(inputs.normal(80, (sum(counts), 512))).to(torch.bfloat16).cuda()
    q = U.ufp4_quantize_grouped(x, U.UFP4_E1M2, counts, rht=True, rht_seed=2, round=1, sr_seed=3,
                                colwise=colwise)
    _check_plane(q)


def test_plane_rejected_for_other_grids(U):
    x = torch.from_numpy(inputs.normal(81, (128, 256))).to(torch.bfloat16).cuda()
    q = U.QTensor.empty(128, 256, U.UFP4_E2M1, x.device)
    assert q.eplane is None
    q.eplane = torch.empty_like(q.codes)
    with pytest.raises(U.UFP4Error):
        U.ufp4_quantize(x, U.UFP4_E2M1, out=q)


@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (300, 200, 320), (129, 257, 1040), (64, 48, 16),
                                   (256, 384, 2048), (130, 140, 4160), (1000, 600, 1536)])
def test_gemm_planes_equal_onchip_expansion(U, M, N, K):
    a = torch.from_numpy(inputs.normal(90, (M, K))).to(torch.bfloat16).cuda()
    b = torch.from_numpy(inputs.normal(91, (N, K), std=0.02)).to(torch.bfloat16).cuda()
    qa = U.ufp4_quantize(a, U.UFP4_E1M2, rht=True, rht_seed=2)
    qb = U.ufp4_quantize(b, U.UFP4_E1M2, rht=True, rht_seed=2)
    c_pl = U.ufp4_gemm(qa, qb)
    c_a = U.ufp4_gemm(_strip(U, qa), qb)          # one plane missing: on-chip expansion
    c_none = U.ufp4_gemm(_strip(U, qa), _strip(U, qb))
    torch.cuda.synchronize()
    assert torch.equal(c_pl, c_none) and torch.equal(c_a, c_none)
    assert c_none.abs().max() > 0


def test_grouped_gemm_planes_equal_onchip_expansion(U):
    counts = [130, 0, 64, 200]
    H, F = 256, 320
    x = torch.from_numpy(inputs.normal(92, (sum(counts), H))).to(torch.bfloat16).cuda()
    w = torch.from_numpy(inputs.normal(93, (len(counts) * F, H), std=0.02)).to(torch.bfloat16).cuda()
    qx = U.ufp4_quantize_grouped(x, U.UFP4_E1M2, counts, rht=True, rht_seed=2)
    qw = U.ufp4_quantize_grouped(w, U.UFP4_E1M2, [F] * len(counts), rht=True, rht_seed=2)
    xo = U.grouped_offsets(counts, False)
    wo = U.grouped_offsets([F] * len(counts), False)
    starts = np.concatenate([[0], np.cumsum(counts)])
    outs = []
    for planes in (True, False):
        y = torch.full((sum(counts), F), 9.0, device="cuda")
        groups = [dict(M=t, N=F, K=H, a_row=xo[e], a_k=0, b_row=wo[e], b_k=0, a_seg=e, b_seg=e,
                       c=y[int(starts[e]):int(starts[e]) + t] if t else y[:1]) for e, t in enumerate(counts)]
        U.ufp4_gemm_grouped(qx if planes else _strip(U, qx), qw if planes else _strip(U, qw), groups)
        outs.append(y)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and outs[0].abs().max() > 0
