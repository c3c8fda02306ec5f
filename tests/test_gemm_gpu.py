"""GPU parity of the block-scaled FP4 GEMMs against the oracle's fp64 product.

Both sides quantize the same inputs (the oracle with its own code); with RHT
off the codes are bit-exact, so the oracle's fp64 product of its dequantized
operands is the exact value of the GPU's product.  Bar: relative Frobenius
error <= 1e-5 (fp32 accumulation in the tensor cores).
"""
import numpy as np
import pytest
import torch

from fp4_quantized_numerics_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = 1e-5


@pytest.fixture(scope="module")
def U():
    from fp4_quantized_numerics_gb300 import build, ufp4
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return ufp4


def _rel_fro(c, ref):
    return float(np.linalg.norm(c - ref) / max(np.linalg.norm(ref), 1e-300))


def _gemm_case(U, oracle, a, b, grid, rht=False, col_a=False, col_b=False, round_a=0):
    ta = torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).cuda()
    tb = torch.from_numpy(np.ascontiguousarray(b)).to(torch.bfloat16).cuda()
    qa = U.ufp4_quantize(ta, grid, rht=rht, rht_seed=2, colwise=col_a, round=round_a, sr_seed=3)
    qb = U.ufp4_quantize(tb, grid, rht=rht, rht_seed=2, colwise=col_b)
    c = U.ufp4_gemm(qa, qb)
    torch.cuda.synchronize()
    ra = oracle.quantize(a, grid, rht=rht, rht_seed=2, colwise=col_a, round_mode=round_a, sr_seed=3)
    rb = oracle.quantize(b, grid, rht=rht, rht_seed=2, colwise=col_b)
    A = oracle.dequantize(ra["codes"], ra["scales"], ra["tensor_scale"], grid)
    B = oracle.dequantize(rb["codes"], rb["scales"], rb["tensor_scale"], grid)
    ref = oracle.gemm_f64(A, B)
    return c.cpu().numpy().astype(np.float64), ref


@pytest.mark.parametrize("grid", [0, 1, 2])
def test_smoke_gemm_256(U, oracle, grid):
    d = inputs.smoke(0)
    c, ref = _gemm_case(U, oracle, d["a"], d["b"], grid)
    assert _rel_fro(c, ref) <= TOL


@pytest.mark.parametrize("grid", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (300, 200, 320), (129, 257, 1040),
                                   (64, 48, 16), (256, 384, 2048), (130, 140, 4160)])
def test_ragged_and_multistage(U, oracle, grid, M, N, K):
    a = inputs.normal(41, (M, K))
    b = inputs.normal(42, (N, K), std=0.02)
    c, ref = _gemm_case(U, oracle, a, b, grid)
    assert _rel_fro(c, ref) <= TOL


@pytest.mark.parametrize("grid", [0, 1])
def test_training_orientations(U, oracle, grid):
    """fwd_y = X W^T, bwd_dx = dY W (B = W column-wise), bwd_dw = dY^T X
    (both operands column-wise), with SR on dY as in the recipe."""
    T, H, F = 192, 256, 320
    x = inputs.normal(43, (T, H))
    w = inputs.normal(44, (F, H), std=0.02)
    dy = inputs.normal(45, (T, F), std=1e-3)
    c, ref = _gemm_case(U, oracle, x, w, grid)                                   # fwd_y
    assert c.shape == (T, F) and _rel_fro(c, ref) <= TOL
    c, ref = _gemm_case(U, oracle, dy, w, grid, col_b=True, round_a=1)          # bwd_dx
    assert c.shape == (T, H) and _rel_fro(c, ref) <= TOL
    c, ref = _gemm_case(U, oracle, dy, x, grid, col_a=True, col_b=True, round_a=1)  # bwd_dw
    assert c.shape == (F, H) and _rel_fro(c, ref) <= TOL


@pytest.mark.parametrize("grid", [0, 1])
def test_rht_gemm_close_to_unrotated_product(U, oracle, grid):
    """With the same signs on both operands the rotation cancels in A B^T; the
    GPU result must stay close to the oracle's quantized RHT product (codes
    may differ in <= 1e-4 of the elements)."""
    d = inputs.smoke(0)
    c, ref = _gemm_case(U, oracle, d["a"], d["b"], grid, rht=True)
    assert _rel_fro(c, ref) <= 1e-3
    exact = d["a"].astype(np.float64) @ d["b"].astype(np.float64).T
    assert _rel_fro(c, exact) <= (0.2 if grid == 0 else 0.15)


def test_gemm_k_zero_writes_zeros(U):
    q = U.QTensor.empty(64, 0, 0)
    out = torch.full((64, 64), 7.0, device="cuda")
    U.ufp4_gemm(q, U.QTensor.empty(64, 0, 0), out=out)
    torch.cuda.synchronize()
    assert not out.any()


def test_gemm_no_timeout_flag(U):
    assert U.ufp4_check() == U.UFP4_OK
