"""Thin ctypes binding of libufp4 (include/ufp4.h).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels.  PyTorch provides device memory and the current stream.  There
is no fallback: if libufp4.so is missing or a tensor is not on a CUDA device,
the calls raise.

The functions carry the C names:
  ufp4_quantize(x, grid, ...) -> QTensor
  ufp4_dequantize(q, ...)     -> fp32 tensor
  ufp4_gemm(a, b, ...)        -> fp32 tensor (C = A B^T)
  ufp4_stats(x, q, ...)       -> dict
  ufp4_check(...), ufp4_status_string(...)
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libufp4.so")

UFP4_E2M1, UFP4_E1M2, UFP4_E2M1C, UFP4_MXFP4 = 0, 1, 2, 3
UFP4_BLOCK, UFP4_MX_BLOCK = 16, 32
UFP4_RTNE, UFP4_SR = 0, 1
UFP4_BF16, UFP4_FP32 = 0, 1
UFP4_OK, UFP4_ERR_INVALID, UFP4_ERR_UNSUPPORTED, UFP4_ERR_NONFINITE, UFP4_ERR_CUDA, \
    UFP4_ERR_TIMEOUT = range(6)

EXPORTED = ["ufp4_kpad", "ufp4_codes_bytes", "ufp4_scales_bytes", "ufp4_workspace_bytes",
            "ufp4_quantize", "ufp4_check", "ufp4_dequantize", "ufp4_gemm", "ufp4_stats",
            "ufp4_status_string", "ufp4_quantize_noalloc", "ufp4_grouped_rows",
            "ufp4_grouped_kpad", "ufp4_quantize_grouped", "ufp4_gemm_grouped", "ufp4_quantize_dual",
            "ufp4_gemm_amax", "ufp4_quantize_stats", "ufp4_quantize_grouped_dual"]


class QParamsC(ctypes.Structure):
    _fields_ = [("grid", ctypes.c_int32), ("block", ctypes.c_int32), ("rht", ctypes.c_int32),
                ("round", ctypes.c_int32), ("rht_seed", ctypes.c_uint64),
                ("sr_seed", ctypes.c_uint64), ("sr_counter", ctypes.c_uint64),
                ("colwise", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("amax_in", ctypes.c_void_p)]


class QTensorC(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("tensor_scale", ctypes.c_void_p), ("rows", ctypes.c_int64),
                ("k", ctypes.c_int64), ("grid", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("eplane", ctypes.c_void_p)]


class StatsC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_double) for n in
                ("alpha", "sqnr_db", "mean_bias", "sum_aq", "sum_aa", "sum_err2", "bias_count")]


class GemmGroupC(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("a_row", ctypes.c_int64), ("a_k", ctypes.c_int64), ("b_row", ctypes.c_int64),
                ("b_k", ctypes.c_int64), ("a_seg", ctypes.c_int32), ("b_seg", ctypes.c_int32),
                ("c", ctypes.c_void_p), ("ldc", ctypes.c_int64)]


class UFP4Error(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what, ufp4_status_string(status), status))


_lib = None


def lib():
    """The loaded libufp4 (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libufp4.so is not built (run fp4_quantized_numerics_gb300.build.build())")
        L = ctypes.CDLL(LIB_PATH)
        i64, vp = ctypes.c_int64, ctypes.c_void_p
        L.ufp4_kpad.argtypes = [i64]
        L.ufp4_kpad.restype = i64
        L.ufp4_codes_bytes.argtypes = [i64, i64]
        L.ufp4_codes_bytes.restype = i64
        L.ufp4_scales_bytes.argtypes = [i64, i64]
        L.ufp4_scales_bytes.restype = i64
        L.ufp4_workspace_bytes.argtypes = []
        L.ufp4_workspace_bytes.restype = ctypes.c_size_t
        L.ufp4_quantize.argtypes = [vp, ctypes.c_int32, i64, i64, i64, ctypes.POINTER(QParamsC),
                                    ctypes.POINTER(QTensorC), vp, ctypes.c_size_t, vp]
        L.ufp4_quantize.restype = ctypes.c_int
        L.ufp4_quantize_dual.argtypes = [vp, ctypes.c_int32, i64, i64, i64, ctypes.POINTER(QParamsC),
                                         ctypes.POINTER(QParamsC), ctypes.POINTER(QTensorC),
                                         ctypes.POINTER(QTensorC), vp, ctypes.c_size_t, vp]
        L.ufp4_quantize_dual.restype = ctypes.c_int
        L.ufp4_check.argtypes = [vp, vp]
        L.ufp4_check.restype = ctypes.c_int
        L.ufp4_dequantize.argtypes = [ctypes.POINTER(QTensorC), ctypes.c_int32, ctypes.c_uint64,
                                      vp, i64, vp]
        L.ufp4_dequantize.restype = ctypes.c_int
        L.ufp4_gemm.argtypes = [ctypes.POINTER(QTensorC), ctypes.POINTER(QTensorC), vp, i64, vp]
        L.ufp4_gemm.restype = ctypes.c_int
        L.ufp4_gemm_amax.argtypes = [ctypes.POINTER(QTensorC), ctypes.POINTER(QTensorC), vp, i64,
                                     ctypes.c_int32, ctypes.c_uint64, vp, vp]
        L.ufp4_gemm_amax.restype = ctypes.c_int
        L.ufp4_stats.argtypes = [vp, ctypes.c_int32, i64, i64, i64, ctypes.POINTER(QParamsC),
                                 ctypes.POINTER(QTensorC), vp, ctypes.c_size_t,
                                 ctypes.POINTER(StatsC), vp]
        L.ufp4_stats.restype = ctypes.c_int
        L.ufp4_quantize_stats.argtypes = [vp, ctypes.c_int32, i64, i64, i64, ctypes.POINTER(QParamsC),
                                          ctypes.POINTER(QTensorC), vp, ctypes.c_size_t,
                                          ctypes.POINTER(StatsC), vp]
        L.ufp4_quantize_stats.restype = ctypes.c_int
        i64p = ctypes.POINTER(ctypes.c_int64)
        L.ufp4_grouped_rows.argtypes = [i64p, ctypes.c_int32]
        L.ufp4_grouped_rows.restype = i64
        L.ufp4_grouped_kpad.argtypes = [i64p, ctypes.c_int32]
        L.ufp4_grouped_kpad.restype = i64
        L.ufp4_quantize_grouped.argtypes = [vp, ctypes.c_int32, i64, i64, i64p, ctypes.c_int32,
                                            ctypes.POINTER(QParamsC), ctypes.POINTER(QTensorC), vp,
                                            ctypes.c_size_t, vp]
        L.ufp4_quantize_grouped.restype = ctypes.c_int
        L.ufp4_quantize_grouped_dual.argtypes = [vp, ctypes.c_int32, i64, i64, i64p, ctypes.c_int32,
                                                 ctypes.POINTER(QParamsC), ctypes.POINTER(QParamsC),
                                                 ctypes.POINTER(QTensorC), ctypes.POINTER(QTensorC), vp,
                                                 ctypes.c_size_t, vp]
        L.ufp4_quantize_grouped_dual.restype = ctypes.c_int
        L.ufp4_gemm_grouped.argtypes = [ctypes.POINTER(QTensorC), ctypes.POINTER(QTensorC),
                                        ctypes.POINTER(GemmGroupC), ctypes.c_int32, vp]
        L.ufp4_gemm_grouped.restype = ctypes.c_int
        L.ufp4_status_string.argtypes = [ctypes.c_int]
        L.ufp4_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def ufp4_status_string(status):
    return lib().ufp4_status_string(int(status)).decode()


def _check(status, what):
    if status != UFP4_OK:
        raise UFP4Error(status, what)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _cuda(t, name):
    if not (isinstance(t, torch.Tensor) and t.is_cuda):
        raise TypeError("%s must be a CUDA tensor (libufp4 has no CPU path)" % name)


_workspaces = {}


def workspace(device=None):
    """A per-device scratch buffer of ufp4_workspace_bytes() (allocated once)."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    if dev.index is None:
        dev = torch.device(dev.type, torch.cuda.current_device())
    key = (dev.type, dev.index)
    ws = _workspaces.get(key)
    if ws is None:
        ws = torch.empty(int(lib().ufp4_workspace_bytes()), dtype=torch.uint8, device=dev)
        _workspaces[key] = ws
    return ws


class QTensor:
    """Quantized tensor: device codes / scales / tensor scale in the layouts
    of include/ufp4.h, logical shape rows x k; E1M2 tensors may carry the
    correction plane (eplane) that the quantizer writes and the GEMM loads."""

    def __init__(self, codes, scales, tensor_scale, rows, k, grid, eplane=None):
        self.codes, self.scales, self.tensor_scale = codes, scales, tensor_scale
        self.rows, self.k, self.grid = int(rows), int(k), int(grid)
        self.eplane = eplane

    @classmethod
    def empty(cls, rows, k, grid, device="cuda", eplane=None):
        """eplane: allocate the E1M2 correction plane (default: for E1M2)."""
        L = lib()
        codes = torch.empty(max(int(L.ufp4_codes_bytes(rows, k)), 1), dtype=torch.uint8, device=device)
        scales = torch.empty(max(int(L.ufp4_scales_bytes(rows, k)), 1), dtype=torch.uint8, device=device)
        ts = torch.empty(1, dtype=torch.float32, device=device)
        if eplane is None:
            eplane = int(grid) == UFP4_E1M2
        ep = torch.empty_like(codes) if eplane and int(grid) == UFP4_E1M2 else None
        return cls(codes, scales, ts, rows, k, grid, ep)

    @property
    def kpad(self):
        return int(lib().ufp4_kpad(self.k))

    def c(self):
        return QTensorC(self.codes.data_ptr(), self.scales.data_ptr(), self.tensor_scale.data_ptr(),
                        self.rows, self.k, self.grid, 0,
                        None if self.eplane is None else self.eplane.data_ptr())

    def codes_2d(self):
        """codes as uint8 [rows, kpad/2] (a view)."""
        return self.codes[: self.rows * (self.kpad // 2)].view(self.rows, self.kpad // 2)


def _dtype_code(x):
    if x.dtype == torch.bfloat16:
        return UFP4_BF16
    if x.dtype == torch.float32:
        return UFP4_FP32
    raise TypeError("libufp4 quantizes bf16 or fp32 tensors, got %s" % x.dtype)


def qparams(grid, rht=False, rht_seed=0, round=UFP4_RTNE, sr_seed=0, sr_counter=0,
            colwise=False, amax_in=None):
    block = UFP4_MX_BLOCK if int(grid) == UFP4_MXFP4 else UFP4_BLOCK
    return QParamsC(int(grid), block, int(bool(rht)), int(round), int(rht_seed) & (2**64 - 1),
                    int(sr_seed) & (2**64 - 1), int(sr_counter) & (2**64 - 1), int(bool(colwise)), 0,
                    None if amax_in is None else amax_in.data_ptr())


def ufp4_quantize(x, grid, rht=False, rht_seed=0, round=UFP4_RTNE, sr_seed=0, sr_counter=0,
                  colwise=False, amax_in=None, out=None, ws=None, stream=None):
    """Fused (RHT +) block quantization of a 2-D bf16/fp32 CUDA tensor.
    Row-wise: blocks along the last dim, result rows x cols.  colwise=True:
    blocks down the columns, result is the quantization of x.T."""
    _cuda(x, "x")
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit stride in its last dim")
    rows, cols = x.shape
    out_rows, k = (cols, rows) if colwise else (rows, cols)
    if out is None:
        out = QTensor.empty(out_rows, k, grid, x.device)
    if ws is None:
        ws = workspace(x.device)
    p = qparams(grid, rht, rht_seed, round, sr_seed, sr_counter, colwise, amax_in)
    qc = out.c()
    st = lib().ufp4_quantize(x.data_ptr(), _dtype_code(x), rows, cols, x.stride(0), ctypes.byref(p),
                             ctypes.byref(qc), ws.data_ptr(), ws.numel(), _stream(stream))
    _check(st, "ufp4_quantize")
    return out


def ufp4_quantize_dual(x, grid, rht=False, rht_seed=0, round=UFP4_RTNE, sr_seed=0, sr_counter_row=0,
                       sr_counter_col=0, amax_row=None, amax_col=None, out_row=None, out_col=None, ws=None,
                       stream=None):
    """Row-wise and column-wise quantization of x (results x and x.T
    quantized along their last dim) from one read of x per pass."""
    _cuda(x, "x")
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit stride in its last dim")
    rows, cols = x.shape
    if out_row is None:
        out_row = QTensor.empty(rows, cols, grid, x.device)
    if out_col is None:
        out_col = QTensor.empty(cols, rows, grid, x.device)
    if ws is None:
        ws = workspace(x.device)
    pr = qparams(grid, rht, rht_seed, round, sr_seed, sr_counter_row, False, amax_row)
    pc = qparams(grid, rht, rht_seed, round, sr_seed, sr_counter_col, True, amax_col)
    qr, qc = out_row.c(), out_col.c()
    st = lib().ufp4_quantize_dual(x.data_ptr(), _dtype_code(x), rows, cols, x.stride(0), ctypes.byref(pr),
                                  ctypes.byref(pc), ctypes.byref(qr), ctypes.byref(qc), ws.data_ptr(),
                                  ws.numel(), _stream(stream))
    _check(st, "ufp4_quantize_dual")
    return out_row, out_col


def ufp4_check(ws=None, stream=None):
    return lib().ufp4_check(None if ws is None else ws.data_ptr(), _stream(stream))


def ufp4_dequantize(q, inverse_rht=False, rht_seed=0, out=None, stream=None):
    _cuda(q.codes, "q.codes")
    if out is None:
        out = torch.empty(q.rows, q.k, dtype=torch.float32, device=q.codes.device)
    qc = q.c()
    st = lib().ufp4_dequantize(ctypes.byref(qc), int(bool(inverse_rht)), int(rht_seed),
                               out.data_ptr(), out.stride(0), _stream(stream))
    _check(st, "ufp4_dequantize")
    return out


def ufp4_gemm(a, b, out=None, stream=None):
    """C = A B^T (fp32), A: M x K and B: N x K quantized along K."""
    _cuda(a.codes, "a.codes")
    _cuda(b.codes, "b.codes")
    if out is None:   # row stride rounded up to 4 floats (16 bytes), as the ABI requires
        ld = (b.rows + 3) // 4 * 4
        out = torch.empty(a.rows, ld, dtype=torch.float32, device=a.codes.device)[:, : b.rows]
    ac, bc = a.c(), b.c()
    st = lib().ufp4_gemm(ctypes.byref(ac), ctypes.byref(bc), out.data_ptr(), out.stride(0),
                         _stream(stream))
    _check(st, "ufp4_gemm")
    return out


def ufp4_gemm_amax(a, b, rht=False, rht_seed=0, out=None, amax=None, stream=None):
    """C = A B^T as ufp4_gemm, and the tensor amax of C's row-wise
    quantization (rotated with rht_seed when rht) from the epilogue.
    Returns (C, amax); pass amax as the amax_in of ufp4_quantize(C, ...)."""
    _cuda(a.codes, "a.codes")
    _cuda(b.codes, "b.codes")
    if out is None:
        ld = (b.rows + 3) // 4 * 4
        out = torch.empty(a.rows, ld, dtype=torch.float32, device=a.codes.device)[:, : b.rows]
    if amax is None:
        amax = torch.empty(1, dtype=torch.float32, device=a.codes.device)
    ac, bc = a.c(), b.c()
    st = lib().ufp4_gemm_amax(ctypes.byref(ac), ctypes.byref(bc), out.data_ptr(), out.stride(0),
                              int(bool(rht)), int(rht_seed) & (2**64 - 1), amax.data_ptr(), _stream(stream))
    _check(st, "ufp4_gemm_amax")
    return out, amax


def ufp4_quantize_stats(x, grid, rht=False, rht_seed=0, round=UFP4_RTNE, sr_seed=0, sr_counter=0,
                        colwise=False, amax_in=None, out=None, ws=None, stream=None):
    """ufp4_quantize and ufp4_stats of its result in one call (one read of x
    where the layout allows).  Returns (QTensor, stats dict); synchronises."""
    _cuda(x, "x")
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit stride in its last dim")
    rows, cols = x.shape
    out_rows, k = (cols, rows) if colwise else (rows, cols)
    if out is None:
        out = QTensor.empty(out_rows, k, grid, x.device)
    if ws is None:
        ws = workspace(x.device)
    p = qparams(grid, rht, rht_seed, round, sr_seed, sr_counter, colwise, amax_in)
    qc = out.c()
    res = StatsC()
    st = lib().ufp4_quantize_stats(x.data_ptr(), _dtype_code(x), rows, cols, x.stride(0), ctypes.byref(p),
                                   ctypes.byref(qc), ws.data_ptr(), ws.numel(), ctypes.byref(res),
                                   _stream(stream))
    _check(st, "ufp4_quantize_stats")
    return out, {n: getattr(res, n) for n, _ in StatsC._fields_}


def ufp4_stats(x, q, rht=False, rht_seed=0, round=UFP4_RTNE, sr_seed=0, sr_counter=0,
               colwise=False, amax_in=None, ws=None, stream=None):
    """alpha, SQNR and mean rounding bias of quantization q of x (synchronises)."""
    _cuda(x, "x")
    rows, cols = x.shape
    if ws is None:
        ws = workspace(x.device)
    p = qparams(q.grid, rht, rht_seed, round, sr_seed, sr_counter, colwise, amax_in)
    qc = q.c()
    out = StatsC()
    st = lib().ufp4_stats(x.data_ptr(), _dtype_code(x), rows, cols, x.stride(0), ctypes.byref(p),
                          ctypes.byref(qc), ws.data_ptr(), ws.numel(), ctypes.byref(out),
                          _stream(stream))
    _check(st, "ufp4_stats")
    return {n: getattr(out, n) for n, _ in StatsC._fields_}


# ------------------------------------------------------------ grouped (MoE)
def _i64_array(vals):
    arr = (ctypes.c_int64 * len(vals))(*[int(v) for v in vals])
    return arr


def grouped_rows(seg_rows):
    return int(lib().ufp4_grouped_rows(_i64_array(seg_rows), len(seg_rows)))


def grouped_kpad(seg_rows):
    return int(lib().ufp4_grouped_kpad(_i64_array(seg_rows), len(seg_rows)))


def grouped_offsets(seg_rows, colwise):
    """Row offsets (row-wise) or k offsets (column-wise) of each segment."""
    offs, o = [], 0
    for t in seg_rows:
        offs.append(o)
        if t > 0:
            o += ((t + 63) // 64 * 64) if colwise else ((t + 127) // 128 * 128)
    return offs


def ufp4_quantize_grouped(x, grid, seg_rows, rht=False, rht_seed=0, round=UFP4_RTNE, sr_seed=0,
                          sr_counter=0, colwise=False, out=None, ws=None, stream=None):
    """Quantize the row segments of x, one tensor scale per segment (layouts:
    include/ufp4.h, grouped tensors).  Returns a QTensor whose tensor_scale
    holds one S_dec per segment."""
    _cuda(x, "x")
    cols = x.shape[1]
    n = len(seg_rows)
    if colwise:
        rows, k = cols, grouped_kpad(seg_rows)
    else:
        rows, k = grouped_rows(seg_rows), cols
    if out is None:
        out = QTensor.empty(rows, k, grid, x.device)
        out.tensor_scale = torch.empty(max(n, 1), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = workspace(x.device)
    p = qparams(grid, rht, rht_seed, round, sr_seed, sr_counter, colwise)
    qc = out.c()
    st = lib().ufp4_quantize_grouped(x.data_ptr(), _dtype_code(x), cols, x.stride(0),
                                     _i64_array(seg_rows), n, ctypes.byref(p), ctypes.byref(qc),
                                     ws.data_ptr(), ws.numel(), _stream(stream))
    _check(st, "ufp4_quantize_grouped")
    out.seg_rows = list(seg_rows)
    return out


def ufp4_quantize_grouped_dual(x, grid, seg_rows, rht=False, rht_seed=0, round=UFP4_RTNE, sr_seed=0,
                               sr_counter_row=0, sr_counter_col=0, out_row=None, out_col=None, ws=None,
                               stream=None):
    """Row-wise and column-wise grouped quantization of x from one read of x
    per pass; each result as its own ufp4_quantize_grouped call."""
    _cuda(x, "x")
    cols = x.shape[1]
    n = len(seg_rows)
    if out_row is None:
        out_row = QTensor.empty(grouped_rows(seg_rows), cols, grid, x.device)
        out_row.tensor_scale = torch.empty(max(n, 1), dtype=torch.float32, device=x.device)
    if out_col is None:
        out_col = QTensor.empty(cols, grouped_kpad(seg_rows), grid, x.device)
        out_col.tensor_scale = torch.empty(max(n, 1), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = workspace(x.device)
    pr = qparams(grid, rht, rht_seed, round, sr_seed, sr_counter_row, False)
    pc = qparams(grid, rht, rht_seed, round, sr_seed, sr_counter_col, True)
    qr, qc = out_row.c(), out_col.c()
    st = lib().ufp4_quantize_grouped_dual(x.data_ptr(), _dtype_code(x), cols, x.stride(0),
                                          _i64_array(seg_rows), n, ctypes.byref(pr), ctypes.byref(pc),
                                          ctypes.byref(qr), ctypes.byref(qc), ws.data_ptr(), ws.numel(),
                                          _stream(stream))
    _check(st, "ufp4_quantize_grouped_dual")
    out_row.seg_rows = list(seg_rows)
    out_col.seg_rows = list(seg_rows)
    return out_row, out_col


def ufp4_gemm_grouped(a, b, groups, stream=None):
    """groups: list of dicts with keys M, N, K, a_row, a_k, b_row, b_k, a_seg,
    b_seg and c (an fp32 CUDA tensor view of M x N with unit column stride)."""
    arr = (GemmGroupC * max(len(groups), 1))()
    for i, g in enumerate(groups):
        c = g["c"]
        arr[i] = GemmGroupC(g["M"], g["N"], g["K"], g["a_row"], g["a_k"], g["b_row"], g["b_k"],
                            g["a_seg"], g["b_seg"], c.data_ptr(), c.stride(0))
    ac, bc = a.c(), b.c()
    st = lib().ufp4_gemm_grouped(ctypes.byref(ac), ctypes.byref(bc), arr, len(groups), _stream(stream))
    _check(st, "ufp4_gemm_grouped")
