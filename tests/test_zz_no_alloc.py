"""ufp4_quantize_noalloc against ufp4_quantize (GPU, through the C ABI).

The no-allocation entry point serves callers that cannot allocate device
memory when they quantize; it keeps its scratch in a fixed array inside the
library instead of a caller workspace.  Its results must equal those of the
regular entry point bit for bit (same kernels), on two calls in a row --
the second call reuses the array the first one left behind.  This file is
named to be collected last.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    from fp4_quantized_numerics_gb300 import build, ufp4
    build.build()
    L = ufp4.lib()
    f = L.ufp4_quantize_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  ctypes.POINTER(ufp4.QParamsC), ctypes.POINTER(ufp4.QTensorC), ctypes.c_void_p]
    f.restype = ctypes.c_int
    return ufp4, f


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    assert torch.cuda.is_available(), "GPU test"
    U, f = _noalloc_fn()
    cases = [  # (rows, cols, grid, rht, round, colwise, seed)
        (512, 1024, U.UFP4_E1M2, True, U.UFP4_RTNE, False, 1),
        (384, 640, U.UFP4_E2M1, True, U.UFP4_SR, True, 2),
    ]
    for rows, cols, grid, rht, rnd, col, seed in cases:
        g = torch.Generator(device="cuda")
        g.manual_seed(seed)
        x = torch.randn(rows, cols, generator=g, device="cuda").to(torch.bfloat16)
        kw = dict(rht=rht, rht_seed=2, round=rnd, sr_seed=3, sr_counter=seed, colwise=col)
        ref = U.ufp4_quantize(x, grid, **kw)
        out_rows, k = (cols, rows) if col else (rows, cols)
        got = U.QTensor.empty(out_rows, k, grid)
        got.codes.fill_(0xAB)
        got.scales.fill_(0xCD)
        p = U.qparams(grid, **kw)
        qc = got.c()
        st = f(x.data_ptr(), U.UFP4_BF16, rows, cols, x.stride(0), ctypes.byref(p), ctypes.byref(qc),
               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == U.UFP4_OK, U.ufp4_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(got.codes, ref.codes)
        assert torch.equal(got.scales, ref.scales)
        assert torch.equal(got.tensor_scale, ref.tensor_scale)


def test_noalloc_rejects_bad_arguments_without_launching():
    U, f = _noalloc_fn()
    p = U.qparams(U.UFP4_E1M2)
    qc = U.QTensorC(0x1000, 0x1000, 0x1000, 32, 48, U.UFP4_E1M2, 0)   # k mismatch
    assert f(0x20000, U.UFP4_BF16, 32, 64, 64, ctypes.byref(p), ctypes.byref(qc), None) == U.UFP4_ERR_INVALID
