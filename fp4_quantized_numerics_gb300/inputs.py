"""Seeded synthetic inputs for the UFP4 workloads.

This module holds no quantization arithmetic: it only draws random tensors
with the shapes and value distributions of the five workloads, so that the
CUDA path and the CPU oracle can be fed identical bytes.  Host arrays come
from numpy's PCG64 generator (same stream on every platform); the large
device-resident workloads can also be drawn directly on a CUDA device with a
seeded torch generator (used where only sampled outputs are checked).

N(0, s) always means standard deviation s.

Workloads (shapes of the models the pages train, [ZC] Key points,
Validation results; [HP] technical approach):
  smoke      256 x 1024 N(0,1) tensor; 256 x 256 x 256 GEMM operands.
  outlier    4096 x 4096 = N(0,1) + per-column offset N(0,0.5); 0.1% of the
             columns (4) scaled by 100 after the offset -- the coherent-mean
             outliers of [AN] "Systemic Instability".
  dense1p5b  X 8192 x 2048 N(0,1) with 0.05% columns (1) x50;
             W 5632 x 2048 N(0,0.02); dY 8192 x 5632 N(0,1e-3).
  moe7p9b    64 experts, 16384 tokens x top-6; per-expert token counts from a
             multinomial over Dirichlet(1) probabilities (zero allowed);
             X_e N(0,1) [T_e x 2048], W_e N(0,0.02) [1408 x 2048],
             dY_e N(0,1e-3) [T_e x 1408].
  moe124b    X 65536 x 8192 N(0,1), W 2048 x 8192 N(0,0.01),
             dY 65536 x 2048 N(0,1e-3); chain of 100 4096^3 GEMMs with fresh
             W_k N(0, 1/64) and X_0 N(0,1).
"""
import numpy as np

try:
    import torch
except ImportError:  # the oracle-only CPU tests do not need torch
    torch = None


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16_f32(a):
    """Round an fp32 array to bf16 (nearest-even) and return it as fp32, so
    the value is exactly what a bf16 tensor of the same data holds."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    nan = np.isnan(a)
    out = (r & 0xFFFFFFFF).astype(np.uint32).view(np.float32)
    out = np.where(nan, np.float32(np.nan), out)
    return out.astype(np.float32)


def bf16_bits(a_f32):
    """uint16 bit patterns of an fp32 array whose values are already bf16."""
    a = np.ascontiguousarray(a_f32, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def normal(seed, shape, std=1.0):
    return to_bf16_f32(rng(seed).standard_normal(shape, dtype=np.float32) * np.float32(std))


def smoke(seed=0):
    g = rng(seed)
    x = to_bf16_f32(g.standard_normal((256, 1024), dtype=np.float32))
    a = to_bf16_f32(g.standard_normal((256, 256), dtype=np.float32))
    b = to_bf16_f32(g.standard_normal((256, 256), dtype=np.float32))
    return dict(x=x, a=a, b=b)


def outlier(seed=0, rows=4096, cols=4096, frac=0.001, scale=100.0, offset_std=0.5):
    g = rng(seed)
    x = g.standard_normal((rows, cols), dtype=np.float32)
    x += (g.standard_normal(cols, dtype=np.float32) * np.float32(offset_std))[None, :]
    n_out = max(1, int(round(frac * cols)))
    idx = np.sort(g.choice(cols, size=n_out, replace=False))
    x[:, idx] *= np.float32(scale)
    return dict(x=to_bf16_f32(x), outlier_cols=idx)


def dense(seed=0, tokens=8192, hidden=2048, ffn=5632, out_frac=0.0005, out_scale=50.0):
    g = rng(seed)
    x = g.standard_normal((tokens, hidden), dtype=np.float32)
    n_out = max(1, int(round(out_frac * hidden)))
    idx = np.sort(g.choice(hidden, size=n_out, replace=False))
    x[:, idx] *= np.float32(out_scale)
    w = g.standard_normal((ffn, hidden), dtype=np.float32) * np.float32(0.02)
    dy = g.standard_normal((tokens, ffn), dtype=np.float32) * np.float32(1e-3)
    return dict(x=to_bf16_f32(x), w=to_bf16_f32(w), dy=to_bf16_f32(dy), outlier_cols=idx)


def moe_counts(seed=0, tokens=16384, topk=6, experts=64):
    g = rng(seed)
    p = g.dirichlet(np.ones(experts))
    return g.multinomial(tokens * topk, p).astype(np.int64)


def moe(seed=0, tokens=16384, topk=6, experts=64, hidden=2048, ffn=1408, counts=None):
    if counts is None:
        counts = moe_counts(seed, tokens, topk, experts)
    g = rng(seed + 1)
    total = int(counts.sum())
    x = to_bf16_f32(g.standard_normal((total, hidden), dtype=np.float32))
    w = to_bf16_f32(g.standard_normal((experts * ffn, hidden), dtype=np.float32) * np.float32(0.02))
    dy = to_bf16_f32(g.standard_normal((total, ffn), dtype=np.float32) * np.float32(1e-3))
    return dict(counts=counts, x=x, w=w, dy=dy)


# ------------------------------------------------------------ device draws
def device_normal(shape, std, seed, device="cuda", dtype=None):
    """A bf16 N(0, std) tensor drawn on the device with a seeded generator."""
    if dtype is None:
        dtype = torch.bfloat16
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def device_dense(seed=0, tokens=8192, hidden=2048, ffn=5632, device="cuda",
                 out_cols=1, out_scale=50.0):
    x = device_normal((tokens, hidden), 1.0, seed, device)
    g = rng(seed)
    idx = np.sort(g.choice(hidden, size=out_cols, replace=False))
    for c in idx:
        x[:, int(c)] = (x[:, int(c)].float() * out_scale).to(x.dtype)
    w = device_normal((ffn, hidden), 0.02, seed + 1, device)
    dy = device_normal((tokens, ffn), 1e-3, seed + 2, device)
    return dict(x=x, w=w, dy=dy, outlier_cols=idx)
