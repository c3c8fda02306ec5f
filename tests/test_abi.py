"""CPU-only checks of the libufp4 C ABI: the library loads, exports every
symbol include/ufp4.h declares, its size helpers agree with the documented
layouts, and invalid arguments are rejected on the host before any launch.
No call here reaches the GPU."""
import ctypes
import os
import re

import pytest

from tests.layouts import kpad, rpad

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from fp4_quantized_numerics_gb300 import build, ufp4
    build.build()
    return ufp4.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "ufp4.h")).read()
    return sorted(set(re.findall(r"UFP4_API[^;(]*?\b(ufp4_\w+)\s*\(", src)))


def test_header_declares_expected_calls():
    names = _declared()
    for n in ["ufp4_quantize", "ufp4_dequantize", "ufp4_gemm", "ufp4_stats", "ufp4_check",
              "ufp4_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    from fp4_quantized_numerics_gb300 import ufp4
    for n in _declared():
        assert hasattr(L, n), n
    assert set(_declared()) == set(ufp4.EXPORTED)


def test_size_helpers(L):
    for k in [16, 48, 64, 1024, 1040]:
        assert L.ufp4_kpad(k) == kpad(k)
        for r in [1, 127, 128, 300]:
            assert L.ufp4_codes_bytes(r, k) == r * kpad(k) // 2
            assert L.ufp4_scales_bytes(r, k) == rpad(r) * kpad(k) // 16
    assert L.ufp4_codes_bytes(0, 16) == 0
    assert L.ufp4_workspace_bytes() >= 16 * 1024


def test_status_strings(L):
    from fp4_quantized_numerics_gb300 import ufp4
    for s in range(6):
        assert len(ufp4.ufp4_status_string(s)) > 0
    assert ufp4.ufp4_status_string(99) == "unknown status"


def _q(**kw):
    from fp4_quantized_numerics_gb300 import ufp4
    base = dict(grid=0, rht=False, rht_seed=0, round=0, sr_seed=0, sr_counter=0, colwise=False)
    base.update(kw)
    return ufp4.qparams(**base)


def _qt(rows, k, grid=0, ptr=0x1000):
    from fp4_quantized_numerics_gb300 import ufp4
    return ufp4.QTensorC(ptr, ptr, ptr, rows, k, grid, 0)


def test_quantize_rejects_bad_arguments_on_host(L):
    from fp4_quantized_numerics_gb300 import ufp4
    ws, x = 0x10000, 0x20000
    wsb = L.ufp4_workspace_bytes()
    INV = ufp4.UFP4_ERR_INVALID

    def call(p, out, rows=32, cols=64, ld=64, dtype=0, xp=x, w=ws, wb=wsb):
        return L.ufp4_quantize(xp, dtype, rows, cols, ld, ctypes.byref(p) if p is not None else None,
                               ctypes.byref(out) if out is not None else None, w, wb, None)

    assert call(None, _qt(32, 64)) == INV                              # no params
    assert call(_q(), None) == INV                                     # no output
    assert call(_q(grid=7), _qt(32, 64, 7)) == INV                     # bad grid
    assert call(_q(round=3), _qt(32, 64)) == INV                       # bad rounding
    assert call(_q(), _qt(32, 64), dtype=5) == INV                     # bad dtype
    assert call(_q(), _qt(32, 48)) == INV                              # shape mismatch
    assert call(_q(), _qt(32, 64, grid=1)) == INV                      # grid mismatch
    assert call(_q(), _qt(32, 40), cols=40, ld=40) == INV              # k % 16
    assert call(_q(), _qt(32, 64), ld=32) == INV                       # ld < cols
    assert call(_q(), _qt(32, 64), xp=x + 2) == INV                    # misaligned x
    assert call(_q(), _qt(32, 64), ld=68) == INV                       # row stride not 16 B
    assert call(_q(), _qt(32, 64), w=0) == INV                         # no workspace
    assert call(_q(), _qt(32, 64), wb=16) == INV                       # workspace too small
    assert call(_q(), _qt(32, 64, ptr=0x1001)) == INV                  # misaligned codes
    q = _qt(32, 64)
    q.eplane = 0x4000
    assert call(_q(), q) == INV                                        # E plane on an E2M1 tensor
    q = _qt(32, 64, grid=1)
    q.eplane = 0x4008
    assert call(_q(grid=1), q) == INV                                  # misaligned E plane
    p = _q(grid=3)                                                     # MXFP4 wants block 32
    p.block = 16
    assert call(p, _qt(32, 64, grid=3)) == ufp4.UFP4_ERR_UNSUPPORTED
    assert call(_q(grid=3), _qt(32, 48, grid=3), cols=48, ld=48) == INV   # MXFP4: k % 32
    p = _q(grid=3)
    p.amax_in = 0x4000
    assert call(p, _qt(32, 64, grid=3)) == INV                         # MXFP4: no tensor amax
    assert call(_q(colwise=True), _qt(64, 30), rows=30) == INV         # colwise rows % 16
    assert call(_q(colwise=True), _qt(62, 32), rows=32, cols=62, ld=64) == INV  # colwise cols % 4
    p = _q()
    p.block = 32
    assert call(p, _qt(32, 64)) == ufp4.UFP4_ERR_UNSUPPORTED
    p = _q()
    p.reserved = 1
    assert call(p, _qt(32, 64)) == INV


def test_zero_sized_quantize_is_a_noop(L):
    from fp4_quantized_numerics_gb300 import ufp4
    p = _q()
    out = ufp4.QTensorC(0, 0, 0, 0, 64, 0, 0)
    assert L.ufp4_quantize(None, 0, 0, 64, 64, ctypes.byref(p), ctypes.byref(out), 0x10000,
                           L.ufp4_workspace_bytes(), None) == ufp4.UFP4_OK


def test_gemm_and_dequant_reject_bad_arguments_on_host(L):
    from fp4_quantized_numerics_gb300 import ufp4
    INV = ufp4.UFP4_ERR_INVALID
    a, b = _qt(128, 256), _qt(64, 128)
    assert L.ufp4_gemm(ctypes.byref(a), ctypes.byref(b), 0x4000, 64, None) == INV   # K mismatch
    b = _qt(64, 256, grid=1)
    assert L.ufp4_gemm(ctypes.byref(a), ctypes.byref(b), 0x4000, 64, None) == ufp4.UFP4_ERR_UNSUPPORTED
    b = _qt(64, 256)
    assert L.ufp4_gemm(ctypes.byref(a), ctypes.byref(b), 0x4000, 32, None) == INV   # ldc < N
    assert L.ufp4_gemm(ctypes.byref(a), ctypes.byref(b), 0x4004, 64, None) == INV   # c alignment
    assert L.ufp4_gemm(ctypes.byref(a), ctypes.byref(b), 0, 64, None) == INV        # no C
    a, b = _qt(128, 256, grid=1), _qt(64, 256, grid=1)
    a.eplane = 0x4001
    assert L.ufp4_gemm(ctypes.byref(a), ctypes.byref(b), 0x4000, 64, None) == INV   # E plane alignment
    q = _qt(16, 32)
    assert L.ufp4_dequantize(ctypes.byref(q), 2, 0, 0x4000, 32, None) == INV
    assert L.ufp4_dequantize(ctypes.byref(q), 0, 0, 0x4000, 30, None) == INV
    z = _qt(0, 32)
    assert L.ufp4_dequantize(ctypes.byref(z), 0, 0, 0, 0, None) == ufp4.UFP4_OK


def test_stats_rejects_bad_arguments_on_host(L):
    from fp4_quantized_numerics_gb300 import ufp4
    p = _q()
    q = _qt(32, 64)
    out = ufp4.StatsC()
    assert L.ufp4_stats(0x20000, 0, 32, 64, 64, ctypes.byref(p), ctypes.byref(q), 0x10000,
                        L.ufp4_workspace_bytes(), None, None) == ufp4.UFP4_ERR_INVALID
    assert L.ufp4_stats(0x20000, 0, 32, 64, 64, ctypes.byref(p), ctypes.byref(q), 0, 0,
                        ctypes.byref(out), None) == ufp4.UFP4_ERR_INVALID


def test_binding_refuses_cpu_tensors():
    import torch
    from fp4_quantized_numerics_gb300 import ufp4
    with pytest.raises(TypeError):
        ufp4.ufp4_quantize(torch.zeros(16, 16, dtype=torch.bfloat16), 0)


def test_sizes_beyond_the_index_limits_are_refused_on_host(L):
    """Tensors past the kernels' 32-bit block indexing (UFP4_MAX_DIM,
    UFP4_MAX_BLOCKS in include/ufp4.h) return UFP4_ERR_UNSUPPORTED before
    any launch; the pointers are never touched."""
    from fp4_quantized_numerics_gb300 import ufp4
    UNS = ufp4.UFP4_ERR_UNSUPPORTED
    ws, x, wsb = 0x10000, 0x20000, L.ufp4_workspace_bytes()
    # 2^20 rows x 2^16 cols: 2^32 blocks of 16
    rows, cols = 1 << 20, 1 << 16
    p = _q()
    assert L.ufp4_quantize(x, 0, rows, cols, cols, ctypes.byref(p), ctypes.byref(_qt(rows, cols)), ws, wsb,
                           None) == UNS
    pc = _q(colwise=True)
    assert L.ufp4_quantize(x, 0, rows, cols, cols, ctypes.byref(pc), ctypes.byref(_qt(cols, rows)), ws, wsb,
                           None) == UNS
    # one dimension past 2^31
    big = 1 << 31
    assert L.ufp4_quantize(x, 0, 16, big, big, ctypes.byref(p), ctypes.byref(_qt(16, big)), ws, wsb,
                           None) == UNS
    q = _qt(rows, cols)
    assert L.ufp4_dequantize(ctypes.byref(q), 0, 0, 0x4000, cols, None) == UNS
    a, b = _qt(rows, cols), _qt(128, cols)
    assert L.ufp4_gemm(ctypes.byref(a), ctypes.byref(b), 0x4000, 128, None) == UNS
    # just inside the limit still passes validation (it then fails on the fake
    # pointers only if it reached the GPU, which a CPU test must not do: use a
    # too-small workspace to stop it one check later)
    rows_ok = (1 << 31) // (kpad(cols) // 16) - 1
    assert L.ufp4_quantize(x, 0, rows_ok, cols, cols, ctypes.byref(p), ctypes.byref(_qt(rows_ok, cols)), ws, 16,
                           None) == ufp4.UFP4_ERR_INVALID


def test_dual_and_grouped_reject_bad_arguments_on_host(L):
    from fp4_quantized_numerics_gb300 import ufp4
    INV, UNS = ufp4.UFP4_ERR_INVALID, ufp4.UFP4_ERR_UNSUPPORTED
    ws, x, wsb = 0x10000, 0x20000, L.ufp4_workspace_bytes()

    def dual(pr, pc, qr, qc, rows=64, cols=128):
        return L.ufp4_quantize_dual(x, 0, rows, cols, cols, ctypes.byref(pr) if pr else None,
                                    ctypes.byref(pc) if pc else None, ctypes.byref(qr), ctypes.byref(qc),
                                    ws, wsb, None)

    qr, qc = _qt(64, 128), _qt(128, 64)
    assert dual(None, _q(colwise=True), qr, qc) == INV                     # no row params
    assert dual(_q(colwise=True), _q(colwise=True), qr, qc) == INV         # row params must be row-wise
    assert dual(_q(), _q(), qr, qc) == INV                                 # column params must be column-wise
    assert dual(_q(), _q(colwise=True), _qt(64, 128), _qt(64, 128)) == INV   # column result shape
    assert dual(_q(grid=3), _q(grid=3, colwise=True), _qt(64, 128, 3), _qt(128, 64, 3)) == UNS   # MXFP4

    def seg(v):
        return (ctypes.c_int64 * len(v))(*v)

    # grouped row counts: rows round up to 128 per segment, k to 64 (empty segments take none)
    assert L.ufp4_grouped_rows(seg([100, 0, 37]), 3) == 256
    assert L.ufp4_grouped_kpad(seg([100, 0, 37]), 3) == 192

    def grouped(p, out, counts, cols=128, n=None):
        return L.ufp4_quantize_grouped(x, 0, cols, cols, seg(counts), len(counts) if n is None else n,
                                       ctypes.byref(p), ctypes.byref(out), ws, wsb, None)

    out = _qt(256, 128)
    assert grouped(_q(), out, [100, 0, 37], n=0) == INV                    # no segments
    assert grouped(_q(), out, [100, 0, 37], n=300) == INV                  # too many segments
    assert grouped(_q(), out, [100, -1, 37]) == INV                        # negative count
    assert grouped(_q(), _qt(200, 128), [100, 0, 37]) == INV               # rows != sum of rpad
    p = _q()
    p.amax_in = 0x4000
    assert grouped(p, out, [100, 0, 37]) == INV                            # amax is per segment
    assert grouped(_q(grid=3), _qt(256, 128, 3), [100, 0, 37]) == UNS      # MXFP4

    def gdual(pr, pc, qr, qc, counts, cols=128):
        return L.ufp4_quantize_grouped_dual(x, 0, cols, cols, seg(counts), len(counts),
                                            ctypes.byref(pr) if pr else None, ctypes.byref(pc) if pc else None,
                                            ctypes.byref(qr), ctypes.byref(qc), ws, wsb, None)

    gqr, gqc = _qt(256, 128), _qt(128, 192)
    assert gdual(None, _q(colwise=True), gqr, gqc, [100, 0, 37]) == INV           # no row params
    assert gdual(_q(colwise=True), _q(colwise=True), gqr, gqc, [100, 0, 37]) == INV
    assert gdual(_q(), _q(), gqr, gqc, [100, 0, 37]) == INV                       # column params row-wise
    assert gdual(_q(), _q(colwise=True), gqr, _qt(128, 128), [100, 0, 37]) == INV  # column k != sum of kpad
    assert gdual(_q(), _q(colwise=True), _qt(200, 128), gqc, [100, 0, 37]) == INV  # row count
    assert gdual(_q(grid=3), _q(grid=3, colwise=True), _qt(256, 128, 3), _qt(128, 192, 3),
                 [100, 0, 37]) == UNS                                             # MXFP4
    assert gdual(_q(), _q(colwise=True), _qt(0, 128), _qt(128, 0), [0, 0]) == ufp4.UFP4_OK   # nothing to do

    def ggemm(a, b, groups, n=None):
        arr = (ufp4.GemmGroupC * max(len(groups), 1))(*groups)
        return L.ufp4_gemm_grouped(ctypes.byref(a), ctypes.byref(b), arr, len(groups) if n is None else n, None)

    a, b = _qt(256, 128), _qt(256, 128)
    g = ufp4.GemmGroupC(100, 64, 128, 0, 0, 0, 0, 0, 0, 0x4000, 64)
    assert ggemm(a, b, [g], n=300) == INV                                  # too many groups
    assert ggemm(a, _qt(256, 128, 1), [g]) == UNS                          # grids differ
    assert ggemm(_qt(256, 128, 3), _qt(256, 128, 3), [g]) == UNS          # MXFP4
    bad = [ufp4.GemmGroupC(100, 64, 128, 64, 0, 0, 0, 0, 0, 0x4000, 64),   # a_row not on a 128-row tile
           ufp4.GemmGroupC(100, 64, 120, 0, 0, 0, 0, 0, 0, 0x4000, 64),    # K % 16
           ufp4.GemmGroupC(300, 64, 128, 0, 0, 0, 0, 0, 0, 0x4000, 64),    # rows past A
           ufp4.GemmGroupC(100, 64, 128, 0, 32, 0, 0, 0, 0, 0x4000, 64),   # a_k not on a 64 boundary
           ufp4.GemmGroupC(100, 64, 128, 0, 0, 0, 0, 0, 0, 0x4004, 64),    # C alignment
           ufp4.GemmGroupC(100, 64, 128, 0, 0, 0, 0, 0, 0, 0x4000, 32)]    # ldc < N
    for gg in bad:
        assert ggemm(a, b, [gg]) == INV, (gg.M, gg.K, gg.a_row, gg.a_k, gg.c, gg.ldc)
