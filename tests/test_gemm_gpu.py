"""GPU parity of the block-scaled FP4 GEMMs against the oracle's fp64 product.

Both sides quantize the same inputs (the oracle with its own code).  With RHT
off the codes are bit-exact, so the oracle's fp64 product of its dequantized
operands is the exact value of the GPU's product.  With RHT on, the GPU's
codes first pass the code bar against the oracle's (at most 1e-4 one grid
step apart), and the GEMM is compared with the fp64 product of the operands
it consumed: the GPU's codes and scales, dequantized by the oracle.  Bar:
relative Frobenius error <= 1e-5 (fp32 accumulation in the tensor cores).
"""
import numpy as np
import pytest
import torch

from fp4_quantized_numerics_gb300 import inputs
from tests import layouts, parity

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


def consumed(oracle, q):
    """fp64 values of the operand a GPU GEMM consumed: the GPU's codes,
    scales and tensor scale, dequantized by the oracle."""
    torch.cuda.synchronize()
    codes = layouts.unpack_codes(q.codes.cpu().numpy(), q.rows, q.k)
    scales, _ = layouts.unpack_scales(q.scales.cpu().numpy(), q.rows, q.k)
    return codes, oracle.dequantize(codes, scales, float(q.tensor_scale[0].item()), q.grid)


def _gemm_case(U, oracle, a, b, grid, rht=False, col_a=False, col_b=False, round_a=0):
    ta = torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).cuda()
    tb = torch.from_numpy(np.ascontiguousarray(b)).to(torch.bfloat16).cuda()
    qa = U.ufp4_quantize(ta, grid, rht=rht, rht_seed=2, colwise=col_a, round=round_a, sr_seed=3)
    qb = U.ufp4_quantize(tb, grid, rht=rht, rht_seed=2, colwise=col_b)
    c = U.ufp4_gemm(qa, qb)
    torch.cuda.synchronize()
    ra = oracle.quantize(a, grid, rht=rht, rht_seed=2, colwise=col_a, round_mode=round_a, sr_seed=3)
    rb = oracle.quantize(b, grid, rht=rht, rht_seed=2, colwise=col_b)
    if rht:
        # the codes the kernel consumed, at the code bar against the oracle's
        ca, A = consumed(oracle, qa)
        cb, B = consumed(oracle, qb)
        tally = parity.CodeTally()
        tally.add(ca, ra["codes"])
        tally.add(cb, rb["codes"])
        tally.check()
    else:
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
@pytest.mark.parametrize("rht", [False, True])
def test_training_orientations(U, oracle, grid, rht):
    """fwd_y = X W^T, bwd_dx = dY W (B = W column-wise), bwd_dw = dY^T X
    (both operands column-wise), with SR on dY as in the recipe, the
    transform off and on (UFP4 rotates the operands of all three GEMMs)."""
    T, H, F = 192, 256, 320
    x = inputs.normal(43, (T, H))
    w = inputs.normal(44, (F, H), std=0.02)
    dy = inputs.normal(45, (T, F), std=1e-3)
    c, ref = _gemm_case(U, oracle, x, w, grid, rht=rht)                                   # fwd_y
    assert c.shape == (T, F) and _rel_fro(c, ref) <= TOL
    c, ref = _gemm_case(U, oracle, dy, w, grid, rht=rht, col_b=True, round_a=1)          # bwd_dx
    assert c.shape == (T, H) and _rel_fro(c, ref) <= TOL
    c, ref = _gemm_case(U, oracle, dy, x, grid, rht=rht, col_a=True, col_b=True, round_a=1)  # bwd_dw
    assert c.shape == (F, H) and _rel_fro(c, ref) <= TOL


@pytest.mark.parametrize("grid", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 200, 320), (130, 140, 4160)])
def test_rht_gemm_matches_consumed_operands(U, oracle, grid, M, N, K):
    """RHT on: 1e-5 against the fp64 product of the operands consumed, and,
    since the same signs rotate both operands, close to the unrotated
    product of the BF16 inputs (the quantization error only)."""
    a = inputs.normal(46, (M, K))
    b = inputs.normal(47, (N, K))
    c, ref = _gemm_case(U, oracle, a, b, grid, rht=True)
    assert _rel_fro(c, ref) <= TOL
    exact = a.astype(np.float64) @ b.astype(np.float64).T
    assert _rel_fro(c, exact) <= {0: 0.2, 1: 0.15, 2: 0.3}[grid]


def test_gemm_k_zero_writes_zeros(U):
    q = U.QTensor.empty(64, 0, 0)
    out = torch.full((64, 64), 7.0, device="cuda")
    U.ufp4_gemm(q, U.QTensor.empty(64, 0, 0), out=out)
    torch.cuda.synchronize()
    assert not out.any()


def test_gemm_no_timeout_flag(U):
    assert U.ufp4_check() == U.UFP4_OK


@pytest.mark.parametrize("grid", [0, 1])
@pytest.mark.parametrize("M,N,K", [(256, 512, 4096), (384, 300, 8192)])
def test_split_k_deterministic(U, oracle, grid, M, N, K):
    """Few output tiles and a long K: the GEMM splits K in two and adds the
    halves into a zeroed C (TMA reduce-add).  Two terms add the same in
    either order, so repeated runs agree bit for bit; and the result is
    within 1e-5 of the oracle's fp64 product."""
    a = inputs.normal(48, (M, K))
    b = inputs.normal(49, (N, K), std=0.02)
    ta = torch.from_numpy(a).to(torch.bfloat16).cuda()
    tb = torch.from_numpy(b).to(torch.bfloat16).cuda()
    qa, qb = U.ufp4_quantize(ta, grid), U.ufp4_quantize(tb, grid)
    c1 = U.ufp4_gemm(qa, qb).clone()
    c2 = torch.full_like(c1, 5.0)
    U.ufp4_gemm(qa, qb, out=c2)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)
    ra, rb = oracle.quantize(a, grid), oracle.quantize(b, grid)
    ref = oracle.gemm_f64(oracle.dequantize(ra["codes"], ra["scales"], ra["tensor_scale"], grid),
                          oracle.dequantize(rb["codes"], rb["scales"], rb["tensor_scale"], grid))
    assert _rel_fro(c1.cpu().numpy(), ref) <= TOL


@pytest.mark.parametrize("grid", [0, 1])
@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 208, 320), (128, 4096, 1024)])
def test_gemm_amax_fuses_next_quantization(U, oracle, grid, rht, M, N, K):
    """ufp4_gemm_amax: C as ufp4_gemm computes it, and the tensor amax of C's
    row-wise quantization from the epilogue.  Quantizing C with that amax
    given equals, bit for bit, quantizing C with the amax computed by the
    quantizer's own pass; without the transform it is max |C| exactly, with
    it the oracle's rotated amax of C within 1e-6."""
    a = inputs.normal(50, (M, K))
    b = inputs.normal(51, (N, K), std=0.05)
    qa = U.ufp4_quantize(torch.from_numpy(a).to(torch.bfloat16).cuda(), grid)
    qb = U.ufp4_quantize(torch.from_numpy(b).to(torch.bfloat16).cuda(), grid)
    c, am = U.ufp4_gemm_amax(qa, qb, rht=rht, rht_seed=2)
    c_plain = U.ufp4_gemm(qa, qb)
    q_given = U.ufp4_quantize(c, grid, rht=rht, rht_seed=2, amax_in=am)
    q_own = U.ufp4_quantize(c, grid, rht=rht, rht_seed=2)
    torch.cuda.synchronize()
    assert _rel_fro(c.cpu().numpy(), c_plain.cpu().numpy()) <= 1e-6   # plain may split K
    for f in ("codes", "scales", "tensor_scale"):
        assert torch.equal(getattr(q_given, f), getattr(q_own, f)), f
    ch = c.cpu().numpy()
    if not rht:
        assert am.item() == float(np.abs(ch).max())
    else:
        want = oracle.tensor_amax(ch, rht=True, rht_seed=2)
        assert abs(am.item() / want - 1) <= 1e-6


@pytest.mark.parametrize("grid", [0, 1, 3])
def test_repeated_gemms_agree_with_varied_block_scales(U, oracle, grid):
    """The scale warp's tensor-memory copies and the MMAs that read them are
    ordered by fences around an mbarrier, not by waiting for the copies to
    complete.  Rows and K blocks carry block scales spread over 2^-12..2^12,
    so an MMA that read a stage's scales before they landed (or a previous
    stage's) would be far off: 30 runs of a multi-tile, multi-stage GEMM in
    each grid (E2M1, E1M2 with loaded planes, MXFP4) agree bit for bit and
    with the oracle's fp64 product."""
    M, N, K = 512, 1024, 2048
    g = inputs.rng(77)
    a = g.standard_normal((M, K), dtype=np.float32)
    a *= np.float32(2.0) ** g.integers(-12, 13, size=(M, K // 32)).repeat(32, axis=1).astype(np.float32)
    b = g.standard_normal((N, K), dtype=np.float32)
    b *= np.float32(2.0) ** g.integers(-12, 13, size=(N, K // 32)).repeat(32, axis=1).astype(np.float32)
    a, b = inputs.to_bf16_f32(a), inputs.to_bf16_f32(b)
    ta = torch.from_numpy(a).to(torch.bfloat16).cuda()
    tb = torch.from_numpy(b).to(torch.bfloat16).cuda()
    qa, qb = U.ufp4_quantize(ta, grid), U.ufp4_quantize(tb, grid)
    first = U.ufp4_gemm(qa, qb).clone()
    for _ in range(29):
        c = torch.full_like(first, 3.0)
        U.ufp4_gemm(qa, qb, out=c)
        assert torch.equal(c, first)
    if grid == 3:
        ra, rb = oracle.quantize_mx(a), oracle.quantize_mx(b)
        A = oracle.dequantize_mx(ra["codes"], ra["scales"])
        B = oracle.dequantize_mx(rb["codes"], rb["scales"])
    else:
        ra, rb = oracle.quantize(a, grid), oracle.quantize(b, grid)
        A = oracle.dequantize(ra["codes"], ra["scales"], ra["tensor_scale"], grid)
        B = oracle.dequantize(rb["codes"], rb["scales"], rb["tensor_scale"], grid)
    assert _rel_fro(first.cpu().numpy(), oracle.gemm_f64(A, B)) <= TOL
