"""GPU checks through the test-only probe build of the library (tests/probe).

libufp4_probe.so is libufp4 with csrc/quantize.cu compiled under -DUFP4_PROBE:
the same kernels, plus hooks that record the values each quantization path
hands to its block scale, and two probe calls.  Two properties that the
library's outputs only show indirectly are checked directly here:

  * the forward transform: every rotated value y the quantizer computes, in
    every path (row-wise, column-wise, both orientations from one read, the
    strided and grouped kernels; BF16 and FP32 input), against the oracle's
    y = (1/4) H16 diag(d) x, computed in fp64 and rounded once.  Bar: 1e-6
    relative, per element, measured against the l2 norm of the element's
    16-block (an element-wise relative error is meaningless where the
    transform cancels to near zero; the block norm is the transform's
    output scale, and the fp32 butterflies' error bound is about 2.4e-7 of
    it).
  * the block-scale division a / qmax, which the kernels compute with
    Markstein's FMA correction of a reciprocal product: equal bit for bit to
    IEEE division for every finite non-negative fp32 a, qmax = 6, 3.5, 2.
"""
import contextlib
import ctypes

import numpy as np
import pytest
import torch

from fp4_quantized_numerics_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def probe():
    """(binding module, probe library with the binding's argument types)."""
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tests.probe import build as pbuild
    from fp4_quantized_numerics_gb300 import ufp4 as U
    path = pbuild.build_probe()
    saved = U._lib, U.LIB_PATH
    U._lib, U.LIB_PATH = None, path
    try:
        P = U.lib()
    finally:
        U._lib, U.LIB_PATH = saved
    P.ufp4probe_capture.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    P.ufp4probe_capture.restype = ctypes.c_int
    P.ufp4probe_div_qmax.argtypes = [ctypes.c_float, ctypes.c_uint32, ctypes.c_uint32,
                                     ctypes.POINTER(ctypes.c_ulonglong), ctypes.POINTER(ctypes.c_uint32)]
    P.ufp4probe_div_qmax.restype = ctypes.c_int
    return U, P


@contextlib.contextmanager
def _through(U, P, row_y=None, col_y=None):
    """Route the binding's calls to the probe library, capturing into the
    given fp32 device buffers."""
    saved = U._lib
    U._lib = P
    try:
        assert P.ufp4probe_capture(None if row_y is None else row_y.data_ptr(),
                                   None if col_y is None else col_y.data_ptr()) == 0
        yield
        torch.cuda.synchronize()
    finally:
        P.ufp4probe_capture(None, None)
        U._lib = saved


def _check_rotation(y_gpu, y_ref, rows_valid=None):
    """|y_gpu - y_ref| <= 1e-6 * ||block||_2 element by element."""
    g = y_gpu.astype(np.float64)
    r = y_ref.astype(np.float64)
    if rows_valid is not None:
        g, r = g[rows_valid], r[rows_valid]
    norm = np.sqrt((r.reshape(r.shape[0], -1, 16) ** 2).sum(-1, keepdims=True))
    err = np.abs(g - r).reshape(norm.shape[0], -1, 16)
    assert np.all(err <= 1e-6 * norm), "max rel err %g" % float((err / np.maximum(norm, 1e-300)).max())
    return float((g == r).mean())


def _input(shape, seed, dtype):
    """N(0,1) data; BF16-representable for BF16 input, full fp32 otherwise."""
    if dtype == torch.bfloat16:
        return inputs.normal(seed, shape)
    return inputs.rng(seed).standard_normal(shape, dtype=np.float32)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("colwise", [False, True])
@pytest.mark.parametrize("shape", [(256, 1024), (272, 96), (4096, 512)])
def test_forward_rht_single(probe, oracle, dtype, colwise, shape):
    U, P = probe
    x = _input(shape, 61, dtype)
    xt = torch.from_numpy(x).to(dtype).cuda()
    out_rows, k = (shape[1], shape[0]) if colwise else shape
    y = torch.full((out_rows, k), float("nan"), device="cuda")
    with _through(U, P, row_y=None if colwise else y, col_y=y if colwise else None):
        U.ufp4_quantize(xt, U.UFP4_E1M2, rht=True, rht_seed=2, colwise=colwise)
    ref = oracle.quantize(x, 1, rht=True, rht_seed=2, colwise=colwise)["y"]
    _check_rotation(y.cpu().numpy(), ref)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rnd", [0, 1])
def test_forward_rht_dual(probe, oracle, dtype, rnd):
    """Both orientations from one read (the benchmark's step): row-wise
    blocks and column-wise units of the same tiles."""
    U, P = probe
    x = _input((384, 320), 62, dtype)
    xt = torch.from_numpy(x).to(dtype).cuda()
    yr = torch.full((384, 320), float("nan"), device="cuda")
    yc = torch.full((320, 384), float("nan"), device="cuda")
    with _through(U, P, row_y=yr, col_y=yc):
        U.ufp4_quantize_dual(xt, U.UFP4_E1M2, rht=True, rht_seed=2, round=rnd, sr_seed=3)
    _check_rotation(yr.cpu().numpy(), oracle.quantize(x, 1, rht=True, rht_seed=2)["y"])
    _check_rotation(yc.cpu().numpy(), oracle.quantize(x, 1, rht=True, rht_seed=2, colwise=True)["y"])


def test_forward_rht_strided_and_grouped(probe, oracle):
    """The strided kernels (row stride > cols) and the grouped row-wise path."""
    U, P = probe
    x = _input((200, 128), 63, torch.bfloat16)
    wide = torch.zeros(200, 136, dtype=torch.bfloat16, device="cuda")
    wide[:, :128] = torch.from_numpy(x).to(torch.bfloat16).cuda()
    xt = wide[:, :128]
    y = torch.full((200, 128), float("nan"), device="cuda")
    with _through(U, P, row_y=y):
        U.ufp4_quantize(xt, U.UFP4_E2M1, rht=True, rht_seed=2)
    _check_rotation(y.cpu().numpy(), oracle.quantize(x, 0, rht=True, rht_seed=2)["y"])

    counts = [37, 0, 130, 33]
    xg = _input((sum(counts), 64), 64, torch.bfloat16)
    rows = U.grouped_rows(counts)
    yg = torch.full((rows, 64), float("nan"), device="cuda")
    with _through(U, P, row_y=yg):
        U.ufp4_quantize_grouped(torch.from_numpy(xg).to(torch.bfloat16).cuda(), U.UFP4_E1M2, counts,
                                rht=True, rht_seed=2)
    ref = np.zeros((rows, 64), np.float32)
    offs, start = U.grouped_offsets(counts, False), 0
    valid = []
    for e, T in enumerate(counts):
        if T:
            ref[offs[e]:offs[e] + T] = oracle.quantize(xg[start:start + T], 1, rht=True, rht_seed=2)["y"]
            valid.extend(range(offs[e], offs[e] + T))
        start += T
    _check_rotation(yg.cpu().numpy(), ref, np.array(valid))


def test_forward_rht_outlier_columns(probe, oracle):
    """The outlier-heavy 4096 x 4096 input (column offsets, 4 columns x 100):
    wide dynamic range inside a block is where fp32 butterflies round."""
    U, P = probe
    x = inputs.outlier(0)["x"]
    xt = torch.from_numpy(x).to(torch.bfloat16).cuda()
    y = torch.full(x.shape, float("nan"), device="cuda")
    with _through(U, P, row_y=y):
        U.ufp4_quantize(xt, U.UFP4_E2M1, rht=True, rht_seed=2)
    same = _check_rotation(y.cpu().numpy(), oracle.quantize(x, 0, rht=True, rht_seed=2)["y"])
    assert same > 0.99   # most rotated values are bit-identical to the correctly rounded ones


@pytest.mark.parametrize("qmax", [6.0, 3.5, 2.0])
def test_block_scale_division_exhaustive(probe, qmax):
    """div_qmax(a, qmax) == IEEE a / qmax for every finite a >= 0 (2^31 - 2^23
    bit patterns), the division behind every block scale."""
    U, P = probe
    n, first = ctypes.c_ulonglong(0), ctypes.c_uint32(0)
    assert P.ufp4probe_div_qmax(qmax, 0, 0x7F800000, ctypes.byref(n), ctypes.byref(first)) == 0
    assert n.value == 0, "first mismatch at bits 0x%08x" % first.value


def test_gemm_wait_timeout_reports_and_recovers(probe, oracle):
    """The GEMM's bounded waits: with a short budget (about a millisecond)
    and the MMA thread held on a barrier nothing arrives on, the kernel
    gives up, returns normally and raises the flag; ufp4_check reports
    UFP4_ERR_TIMEOUT once and clears it; the next GEMM with the default
    budget is correct.  Nothing faults: every role leaves its loop, drains
    the copies it started and the tensor memory is freed."""
    U, P = probe
    P.ufp4probe_gemm_waits.argtypes = [ctypes.c_longlong, ctypes.c_int]
    P.ufp4probe_gemm_waits.restype = None
    d = inputs.smoke(0)
    a = torch.from_numpy(d["a"]).to(torch.bfloat16).cuda()
    b = torch.from_numpy(d["b"]).to(torch.bfloat16).cuda()
    with _through(U, P):
        assert U.ufp4_check() == U.UFP4_OK
        for grid in (U.UFP4_E2M1, U.UFP4_E1M2):
            qa, qb = U.ufp4_quantize(a, grid), U.ufp4_quantize(b, grid)
            P.ufp4probe_gemm_waits(2_000_000, 1)
            try:
                U.ufp4_gemm(qa, qb)
                torch.cuda.synchronize()
            finally:
                P.ufp4probe_gemm_waits(0, 0)
            assert U.ufp4_check() == U.UFP4_ERR_TIMEOUT
            assert U.ufp4_check() == U.UFP4_OK          # the flag was cleared
            c = U.ufp4_gemm(qa, qb).cpu().numpy().astype(np.float64)
            assert U.ufp4_check() == U.UFP4_OK
            ra, rb = oracle.quantize(d["a"], grid), oracle.quantize(d["b"], grid)
            ref = oracle.gemm_f64(oracle.dequantize(ra["codes"], ra["scales"], ra["tensor_scale"], grid),
                                  oracle.dequantize(rb["codes"], rb["scales"], rb["tensor_scale"], grid))
            assert np.linalg.norm(c - ref) <= 1e-5 * np.linalg.norm(ref)
