"""Test-side readers of the libufp4 output layouts (include/ufp4.h).

These restate the documented byte layouts independently of both the CUDA
library and the oracle, so GPU outputs can be compared with the oracle's
plain layouts (one code per element, row-major scales).
"""
import numpy as np


def kpad(k):
    return (k + 63) // 64 * 64


def rpad(r):
    return (r + 127) // 128 * 128


def unpack_codes(codes_bytes, rows, k):
    """uint8 [rows*kpad/2] packed -> uint8 [rows, k], element 2j = low nibble."""
    kp = kpad(k)
    b = np.asarray(codes_bytes, dtype=np.uint8)[: rows * kp // 2].reshape(rows, kp // 2)
    out = np.empty((rows, kp), dtype=np.uint8)
    out[:, 0::2] = b & 0xF
    out[:, 1::2] = b >> 4
    return out[:, :k]


def code_padding(codes_bytes, rows, k):
    """The padding nibbles k..kpad-1 of every row (must be zero)."""
    kp = kpad(k)
    b = np.asarray(codes_bytes, dtype=np.uint8)[: rows * kp // 2].reshape(rows, kp // 2)
    full = np.empty((rows, kp), dtype=np.uint8)
    full[:, 0::2] = b & 0xF
    full[:, 1::2] = b >> 4
    return full[:, k:]


def scale_index(rows, k):
    """Byte offsets of scale (r, b) for r < rpad(rows), b < kpad(k)/16."""
    kp = kpad(k)
    nkt = kp // 64
    r = np.arange(rpad(rows))[:, None]
    b = np.arange(kp // 16)[None, :]
    return ((r // 128) * nkt + b // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (b % 4)


def unpack_scales(scale_bytes, rows, k):
    """Tiled scale bytes -> (row-major [rows, k/16] scales, all padding entries)."""
    s = np.asarray(scale_bytes, dtype=np.uint8)
    idx = scale_index(rows, k)
    full = s[idx]
    pad = np.concatenate([full[rows:, :].ravel(), full[:rows, k // 16:].ravel()])
    return full[:rows, : k // 16], pad


def rows_of(q, rows):
    """Codes (one per element, [len(rows), k]) and row-major scales
    ([len(rows), k/16]) of selected rows of a device QTensor."""
    import torch
    rows = np.asarray(rows, dtype=np.int64)
    kp = kpad(q.k)
    c2 = q.codes_2d()
    idx = torch.as_tensor(rows, device=c2.device)
    b = c2.index_select(0, idx).cpu().numpy()
    codes = np.empty((len(rows), kp), dtype=np.uint8)
    codes[:, 0::2] = b & 0xF
    codes[:, 1::2] = b >> 4
    nkt = kp // 64
    bb = np.arange(q.k // 16)[None, :]
    r = rows[:, None]
    off = ((r // 128) * nkt + bb // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (bb % 4)
    s_all = q.scales
    sc = s_all[torch.as_tensor(off.ravel(), device=s_all.device)].cpu().numpy().reshape(off.shape)
    return codes[:, : q.k], sc
