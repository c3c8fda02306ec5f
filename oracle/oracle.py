"""Python face of the CPU oracle (test infrastructure only).

Only tests/, the smoke check and the benchmark's cpu_baseline / reference legs
may import this module.  It wraps ufp4_oracle.c through ctypes and works on
numpy arrays; it never touches the CUDA library or its Python binding.

Sources: the three pages on arXiv:2606.20381 ("Rethinking Shrinkage Bias in
LLM FP4 Pretraining"), cited as in ufp4_oracle.c ([ZC] zhichai.net post,
[AN] autonainews.com article, [HP] hotpaper.ai card).

Layouts produced here are the plain ones: one code per element (rows x k,
unpacked), row-major scales (rows x k/16), packed codes with element 2j in the
low nibble of byte j.  Column-wise quantization is literally "transpose, then
quantize row-wise".
"""
import ctypes
import os

import numpy as np

from . import build as _build

E2M1, E1M2, E2M1C = 0, 1, 2
MXFP4 = 3      # E2M1 elements, E8M0 scale per 32 elements (see quantize_mx)
RTNE, SR = 0, 1

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build_oracle()
        L = ctypes.CDLL(path)
        u32p = ctypes.POINTER(ctypes.c_uint32)
        L.ref_philox4x32_10.argtypes = [u32p, u32p, u32p]
        L.ref_rht_signs.argtypes = [ctypes.c_uint64, ctypes.POINTER(ctypes.c_int32)]
        L.ref_hadamard16.argtypes = [ctypes.c_int32, ctypes.c_int32]
        L.ref_hadamard16.restype = ctypes.c_int32
        L.ref_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.ref_e4m3_decode.restype = ctypes.c_double
        L.ref_e4m3_encode.argtypes = [ctypes.c_float]
        L.ref_e4m3_encode.restype = ctypes.c_uint8
        L.ref_grid_value.argtypes = [ctypes.c_int, ctypes.c_int]
        L.ref_grid_value.restype = ctypes.c_double
        L.ref_grid_qmax.argtypes = [ctypes.c_int]
        L.ref_grid_qmax.restype = ctypes.c_double
        L.ref_grid_levels.argtypes = [ctypes.c_int]
        L.ref_grid_levels.restype = ctypes.c_int
        L.ref_round_rtne.argtypes = [ctypes.c_int, ctypes.c_float]
        L.ref_round_rtne.restype = ctypes.c_int
        L.ref_round_sr.argtypes = [ctypes.c_int, ctypes.c_float, ctypes.c_uint32]
        L.ref_round_sr.restype = ctypes.c_int
        L.ref_sr_bits.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
        L.ref_sr_bits.restype = ctypes.c_uint32
        vp = ctypes.c_void_p
        L.ref_quantize.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_uint64,
                                   ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64,
                                   ctypes.c_uint64, vp, vp, vp, vp, vp]
        L.ref_quantize.restype = ctypes.c_int
        L.ref_quantize_strided.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_uint64,
                                           ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64,
                                           ctypes.c_uint64, ctypes.c_uint64, vp, vp, vp, vp, vp]
        L.ref_quantize_strided.restype = ctypes.c_int
        L.ref_tensor_amax.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                      ctypes.c_uint64]
        L.ref_tensor_amax.restype = ctypes.c_float
        L.ref_dequantize.argtypes = [vp, vp, ctypes.c_float, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_uint64, vp]
        L.ref_gemm_f64.argtypes = [vp, vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp]
        L.ref_gemm_entries.argtypes = [vp, vp, ctypes.c_int64, vp, vp, ctypes.c_int64, vp]
        L.ref_stats.argtypes = [vp, vp, vp, ctypes.c_float, ctypes.c_int64, ctypes.c_int64,
                                ctypes.c_int, vp]
        L.ref_e8m0_decode.argtypes = [ctypes.c_uint8]
        L.ref_e8m0_decode.restype = ctypes.c_double
        L.ref_mx_shared_exp.argtypes = [ctypes.c_float]
        L.ref_mx_shared_exp.restype = ctypes.c_int
        L.ref_quantize_mx.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                      ctypes.c_uint64, ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64,
                                      vp, vp, vp]
        L.ref_quantize_mx.restype = ctypes.c_int
        L.ref_dequantize_mx.argtypes = [vp, vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                        ctypes.c_uint64, vp]
        L.ref_stats_mx.argtypes = [vp, vp, vp, ctypes.c_int64, ctypes.c_int64, vp]
        _lib = L
    return _lib


def _p(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


# --------------------------------------------------------------- primitives
def philox4x32_10(ctr, key):
    """Philox4x32-10 (Salmon et al., SC'11) of a 4-word counter and 2-word key."""
    c = (ctypes.c_uint32 * 4)(*[int(v) & 0xFFFFFFFF for v in ctr])
    k = (ctypes.c_uint32 * 2)(*[int(v) & 0xFFFFFFFF for v in key])
    o = (ctypes.c_uint32 * 4)()
    lib().ref_philox4x32_10(c, k, o)
    return [int(v) for v in o]


def rht_signs(seed):
    d = (ctypes.c_int32 * 16)()
    lib().ref_rht_signs(ctypes.c_uint64(seed), d)
    return np.array(list(d), dtype=np.int32)


def hadamard16():
    return np.array([[lib().ref_hadamard16(i, j) for j in range(16)] for i in range(16)],
                    dtype=np.int64)


def e4m3_decode(c):
    return lib().ref_e4m3_decode(int(c))


def e4m3_encode(v):
    return int(lib().ref_e4m3_encode(float(v)))


def grid_value(grid, m):
    return lib().ref_grid_value(grid, int(m))


def grid_qmax(grid):
    return lib().ref_grid_qmax(grid)


def grid_levels(grid):
    return lib().ref_grid_levels(grid)


def round_rtne(grid, a):
    return lib().ref_round_rtne(grid, float(a))


def round_sr(grid, a, r):
    """SR of a >= 0 with the 16 random bits r (the low 16 bits are used)."""
    return lib().ref_round_sr(grid, float(a), int(r) & 0xFFFFFFFF)


def sr_bits(sr_seed, sr_counter, i):
    """The 16 random bits of logical element i (see ref_sr_bits)."""
    return int(lib().ref_sr_bits(sr_seed, sr_counter, i))


# ------------------------------------------------------------------ tensors
def quantize(x, grid, rht=False, rht_seed=0, round_mode=RTNE, sr_seed=0, sr_counter=0,
             colwise=False, amax_in=None, elem_base=0, sr_row_stride=None):
    """Quantize a 2-D fp32 array with 16-blocks along its last dim (row-wise),
    or along its first dim (colwise: the result is the quantization of x.T).

    Returns dict(codes=u8[rows_out, k] (one code per element), scales=u8
    [rows_out, k//16] (row-major E4M3), tensor_scale=float (S_dec),
    y=f32[rows_out, k] (the tensor actually quantized: rotated when rht)).
    """
    x = np.asarray(x, dtype=np.float32)
    if colwise:
        x = x.T
    x = np.ascontiguousarray(x)
    rows, k = x.shape
    codes = np.zeros((rows, k), dtype=np.uint8)
    scales = np.zeros((rows, max(k // 16, 0)), dtype=np.uint8)
    ts = np.zeros(1, dtype=np.float32)
    y = np.zeros((rows, k), dtype=np.float32)
    am = None if amax_in is None else np.array([amax_in], dtype=np.float32)
    stride = k if sr_row_stride is None else sr_row_stride
    rc = lib().ref_quantize_strided(_p(x), rows, k, k, grid, int(bool(rht)), ctypes.c_uint64(rht_seed),
                                    round_mode, ctypes.c_uint64(sr_seed), ctypes.c_uint64(sr_counter),
                                    ctypes.c_uint64(elem_base), ctypes.c_uint64(stride), _p(am), _p(codes),
                                    _p(scales), _p(ts), _p(y))
    if rc != 0:
        raise ValueError("ref_quantize failed (%d): k must be a multiple of 16" % rc)
    return dict(codes=codes, scales=scales, tensor_scale=float(ts[0]), y=y)


def tensor_amax(x, rht=False, rht_seed=0, colwise=False):
    """A_t of the quantization of x (of x.T when colwise), the step of
    quantize() that needs the whole tensor."""
    x = np.asarray(x, dtype=np.float32)
    if colwise:
        x = x.T
    x = np.ascontiguousarray(x)
    rows, k = x.shape
    return float(lib().ref_tensor_amax(_p(x), rows, k, k, int(bool(rht)), ctypes.c_uint64(rht_seed)))


def rpad128(t):
    return (t + 127) // 128 * 128


def kpad64(t):
    return (t + 63) // 64 * 64


def quantize_grouped(x, seg_rows, grid, rht=False, rht_seed=0, round_mode=RTNE, sr_seed=0,
                     sr_counter=0, colwise=False):
    """Per-segment quantization of the row segments of x, each with its own
    tensor scale (mixture-of-experts tokens).  Row-wise: segment e is the
    quantization of its rows, placed at row offset roff_e = sum rpad128 of the
    earlier segments in an output of row length cols.  Column-wise: segment e
    (T_e x cols) is zero-padded to a multiple of 16 rows and becomes cols x
    T16_e at k offset koff_e = sum kpad64 of the earlier segments, in an
    output of row length Ktot = sum kpad64.  Stochastic rounding indexes each
    element by its place in that whole output.  Returns a list of per-segment
    dicts (as quantize) plus 'off' (roff_e or koff_e)."""
    x = np.asarray(x, dtype=np.float32)
    rows, cols = x.shape
    starts = np.concatenate([[0], np.cumsum(seg_rows)]).astype(np.int64)
    ktot = int(sum(kpad64(int(t)) for t in seg_rows if t > 0))
    out, off = [], 0
    for e, T in enumerate(seg_rows):
        T = int(T)
        seg = x[starts[e]:starts[e] + T]
        if not colwise:
            r = quantize(seg, grid, rht, rht_seed, round_mode, sr_seed, sr_counter,
                         elem_base=off * cols) if T > 0 else None
            if r is not None:
                r["off"] = off
            out.append(r)
            off += rpad128(T) if T > 0 else 0
        else:
            if T == 0:
                out.append(None)
                continue
            t16 = (T + 15) // 16 * 16
            padded = np.zeros((t16, cols), np.float32)
            padded[:T] = seg
            r = quantize(padded, grid, rht, rht_seed, round_mode, sr_seed, sr_counter, colwise=True,
                         elem_base=off, sr_row_stride=ktot)
            r["off"] = off
            out.append(r)
            off += kpad64(T)
    return out


def pack_codes(codes):
    """Two codes per byte: element 2j in bits 3..0, element 2j+1 in bits 7..4."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def dequantize(codes, scales, tensor_scale, grid, inverse_rht=False, rht_seed=0):
    """fp64 value of every element: v(m) * e_b * S_dec (then the inverse RHT)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows, k = codes.shape
    out = np.zeros((rows, k), dtype=np.float64)
    lib().ref_dequantize(_p(codes), _p(scales), ctypes.c_float(tensor_scale), rows, k, grid,
                         int(bool(inverse_rht)), ctypes.c_uint64(rht_seed), _p(out))
    return out


def gemm_f64(a, b):
    """C = a @ b.T in fp64 with a plain triple loop (a: M x K, b: N x K)."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    b = np.ascontiguousarray(b, dtype=np.float64)
    M, K = a.shape
    N = b.shape[0]
    c = np.zeros((M, N), dtype=np.float64)
    lib().ref_gemm_f64(_p(a), _p(b), M, N, K, _p(c))
    return c


def gemm_entries(a, b, mi, ni):
    a = np.ascontiguousarray(a, dtype=np.float64)
    b = np.ascontiguousarray(b, dtype=np.float64)
    mi = np.ascontiguousarray(mi, dtype=np.int64)
    ni = np.ascontiguousarray(ni, dtype=np.int64)
    out = np.zeros(len(mi), dtype=np.float64)
    lib().ref_gemm_entries(_p(a), _p(b), a.shape[1], _p(mi), _p(ni), len(mi), _p(out))
    return out


def stats(y, codes, scales, tensor_scale, grid):
    """alpha, SQNR and mean rounding bias of one quantization (see ufp4_oracle.c)."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows, k = codes.shape
    out = np.zeros(7, dtype=np.float64)
    lib().ref_stats(_p(y), _p(codes), _p(scales), ctypes.c_float(tensor_scale), rows, k,
                    grid, _p(out))
    keys = ["alpha", "sqnr_db", "mean_bias", "sum_aq", "sum_aa", "sum_err2", "bias_count"]
    return dict(zip(keys, [float(v) for v in out]))


# ------------------------------------------------------------------- MXFP4
def e8m0_decode(b):
    return lib().ref_e8m0_decode(int(b))


def mx_shared_exp(a):
    return int(lib().ref_mx_shared_exp(float(a)))


def quantize_mx(x, rht=False, rht_seed=0, round_mode=RTNE, sr_seed=0, sr_counter=0, colwise=False):
    """MXFP4 quantization (E2M1 elements, one E8M0 scale per 32 elements along
    the last dim, or along the first when colwise; see ufp4_oracle.c).
    Returns dict(codes=u8[rows_out, k], scales=u8[rows_out, k//32] (biased
    exponents), y=f32[rows_out, k])."""
    x = np.asarray(x, dtype=np.float32)
    if colwise:
        x = x.T
    x = np.ascontiguousarray(x)
    rows, k = x.shape
    codes = np.zeros((rows, k), dtype=np.uint8)
    scales = np.zeros((rows, max(k // 32, 0)), dtype=np.uint8)
    y = np.zeros((rows, k), dtype=np.float32)
    rc = lib().ref_quantize_mx(_p(x), rows, k, k, int(bool(rht)), ctypes.c_uint64(rht_seed), round_mode,
                               ctypes.c_uint64(sr_seed), ctypes.c_uint64(sr_counter), _p(codes), _p(scales),
                               _p(y))
    if rc != 0:
        raise ValueError("ref_quantize_mx failed (%d): k must be a multiple of 32" % rc)
    return dict(codes=codes, scales=scales, y=y)


def dequantize_mx(codes, scales, inverse_rht=False, rht_seed=0):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows, k = codes.shape
    out = np.zeros((rows, k), dtype=np.float64)
    lib().ref_dequantize_mx(_p(codes), _p(scales), rows, k, int(bool(inverse_rht)), ctypes.c_uint64(rht_seed),
                            _p(out))
    return out


def stats_mx(y, codes, scales):
    y = np.ascontiguousarray(y, dtype=np.float32)
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows, k = codes.shape
    out = np.zeros(7, dtype=np.float64)
    lib().ref_stats_mx(_p(y), _p(codes), _p(scales), rows, k, _p(out))
    keys = ["alpha", "sqnr_db", "mean_bias", "sum_aq", "sum_aa", "sum_err2", "bias_count"]
    return dict(zip(keys, [float(v) for v in out]))
