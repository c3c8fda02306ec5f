"""Parity at the workloads' full sizes, on sampled outputs.

The oracle computes each quantization's tensor amax over the whole tensor
(its own pass), then quantizes sampled output rows against that scale, and
GEMM entries from its own quantized rows -- nothing it uses comes from the
GPU.  Workloads: the dense-1.5B training step in the launch configuration the
benchmark times (E1M2, RHT on every operand, SR on dY), the MoE-7.9B grouped
layer (64 experts, 16384 tokens x top-6) and the MoE-124B large layer.
Bars: RHT off bit-exact codes/scales and GEMM blocks within 1e-5 relative
Frobenius; RHT on <= 1e-4 of codes one step apart, tensor scale 1e-6.
"""
import numpy as np
import pytest
import torch

import bench
from fp4_quantized_numerics_gb300 import inputs
from tests import layouts

pytestmark = pytest.mark.gpu
NS = 24   # sampled rows per quantization / GEMM block side


@pytest.fixture(scope="module")
def U():
    from fp4_quantized_numerics_gb300 import build, ufp4
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return ufp4


def _f32(t):
    return t.float().cpu().numpy()


def _check_rows(oracle, q, x, grid, rows_sample, rht, rnd, sr_counter, colwise, tol_frac=1e-4):
    """Sampled output rows of GPU quantization q of host array x vs the oracle."""
    A_t = oracle.tensor_amax(x, rht=rht, rht_seed=2, colwise=colwise)
    qmax = 6.0 if grid == 0 else 3.5
    ts = float(q.tensor_scale[0].item())
    want_ts = float(np.float32(np.float32(A_t) / np.float32(448 * qmax)))
    assert abs(ts / want_ts - 1) <= (1e-6 if rht else 0.0)
    gc, gs = layouts.rows_of(q, rows_sample)
    klen = x.shape[0] if colwise else x.shape[1]
    diff = 0
    for i, r in enumerate(rows_sample):
        vec = x[:, r] if colwise else x[r]
        ref = oracle.quantize(vec[None, :], grid, rht=rht, rht_seed=2, round_mode=rnd, sr_seed=3,
                              sr_counter=sr_counter, amax_in=A_t, elem_base=int(r) * klen)
        if not rht:
            np.testing.assert_array_equal(gc[i], ref["codes"][0])
            np.testing.assert_array_equal(gs[i], ref["scales"][0])
        else:
            si = lambda c: np.where(c & 8, -(c.astype(np.int32) & 7), c.astype(np.int32) & 7)
            d = np.abs(si(gc[i]) - si(ref["codes"][0]))
            assert d.max() <= 1
            diff += int((d > 0).sum())
    if rht:
        assert diff <= max(1, tol_frac * len(rows_sample) * klen * 4)


def _gemm_block(oracle, grid, a, b, a_col, b_col, ms, ns, rht, c_gpu, tol, rnd_a=0, ctr=0):
    """C[ms][:, ns] of A B^T with A = quant(a) (a.T if a_col) vs the oracle."""
    Aa = oracle.tensor_amax(a, rht=rht, rht_seed=2, colwise=a_col)
    Ab = oracle.tensor_amax(b, rht=rht, rht_seed=2, colwise=b_col)
    ka = a.shape[0] if a_col else a.shape[1]
    rows_a = np.stack([a[:, m] if a_col else a[m] for m in ms])
    rows_b = np.stack([b[:, n] if b_col else b[n] for n in ns])
    deq = []
    for rows, idx, A_t, rnd in ((rows_a, ms, Aa, rnd_a), (rows_b, ns, Ab, 0)):
        parts = []
        for j, r in enumerate(idx):
            q = oracle.quantize(rows[j:j + 1], grid, rht=rht, rht_seed=2, round_mode=rnd, sr_seed=3,
                                sr_counter=ctr, amax_in=A_t, elem_base=int(r) * ka)
            parts.append(oracle.dequantize(q["codes"], q["scales"], q["tensor_scale"], grid))
        deq.append(np.concatenate(parts))
    ref = oracle.gemm_f64(deq[0], deq[1])
    got = c_gpu[np.ix_(ms, ns)].astype(np.float64)
    assert np.linalg.norm(got - ref) <= tol * np.linalg.norm(ref)


def _sample(n, k, seed):
    return np.sort(np.random.default_rng(seed).choice(n, size=min(k, n), replace=False))


def test_dense_step_bench_configuration(U, oracle):
    """One step of the benchmark's workload, exactly as bench.py launches it."""
    d = inputs.device_dense(seed=0, device="cuda")
    step = bench.Step(U, d["x"], d["w"], d["dy"], U.UFP4_E1M2)
    step.quantize_all()
    step.gemms()
    torch.cuda.synchronize()
    x, w, dy = _f32(d["x"]), _f32(d["w"]), _f32(d["dy"])
    T, H = x.shape
    F = w.shape[0]
    g = 1
    _check_rows(oracle, step.qx_r, x, g, _sample(T, NS, 1), True, 0, 0, False)
    _check_rows(oracle, step.qw_r, w, g, _sample(F, NS, 2), True, 0, 0, False)
    _check_rows(oracle, step.qdy_r, dy, g, _sample(T, NS, 3), True, 1, 0, False)
    _check_rows(oracle, step.qw_c, w, g, _sample(H, NS, 4), True, 0, 0, True)
    _check_rows(oracle, step.qdy_c, dy, g, _sample(F, NS, 5), True, 1, 0, True)
    _check_rows(oracle, step.qx_c, x, g, _sample(H, NS, 6), True, 0, 0, True)
    # GEMM blocks: with RHT on, <= 1e-4 of the codes may sit one step apart,
    # which moves a K-long dot product by up to ~1e-3 of its norm.
    y = step.y.cpu().numpy()
    _gemm_block(oracle, g, x, w, False, False, _sample(T, NS, 7), _sample(F, NS, 8), True, y, 3e-3)


@pytest.mark.parametrize("grid", [0, 1])
def test_dense_gemms_full_size_exact_codes(U, oracle, grid):
    """fwd_y, bwd_dx, bwd_dw at 8192 x 5632 x 2048 with RHT off (codes are
    then bit-exact, so the oracle block is the exact value of the GPU's)."""
    d = inputs.device_dense(seed=1, device="cuda")
    x, w, dy = d["x"], d["w"], d["dy"]
    qx, qw = U.ufp4_quantize(x, grid), U.ufp4_quantize(w, grid)
    qdy = U.ufp4_quantize(dy, grid, round=U.UFP4_SR, sr_seed=3)
    qwc = U.ufp4_quantize(w, grid, colwise=True)
    qdyc = U.ufp4_quantize(dy, grid, colwise=True, round=U.UFP4_SR, sr_seed=3)
    qxc = U.ufp4_quantize(x, grid, colwise=True)
    y, dx, dw = U.ufp4_gemm(qx, qw), U.ufp4_gemm(qdy, qwc), U.ufp4_gemm(qdyc, qxc)
    torch.cuda.synchronize()
    xh, wh, dyh = _f32(x), _f32(w), _f32(dy)
    T, H = xh.shape
    F = wh.shape[0]
    _gemm_block(oracle, grid, xh, wh, False, False, _sample(T, NS, 11), _sample(F, NS, 12), False,
                y.cpu().numpy(), 1e-5)
    _gemm_block(oracle, grid, dyh, wh, False, True, _sample(T, NS, 13), _sample(H, NS, 14), False,
                dx.cpu().numpy(), 1e-5, rnd_a=1)
    _gemm_block(oracle, grid, dyh, xh, True, True, _sample(F, NS, 15), _sample(H, NS, 16), False,
                dw.cpu().numpy(), 1e-5, rnd_a=1)


def test_moe7p9b_grouped_full_size(U, oracle):
    """64 experts, 16384 tokens x top-6 (Dirichlet(1) routing, zero-token
    experts allowed): grouped RHT + E1M2 quantization and the grouped GEMMs."""
    m = inputs.moe(seed=0)
    counts = [int(c) for c in m["counts"]]
    E, H, F = len(counts), 2048, 1408
    tx = torch.from_numpy(m["x"]).to(torch.bfloat16).cuda()
    tw = torch.from_numpy(m["w"]).to(torch.bfloat16).cuda()
    tdy = torch.from_numpy(m["dy"]).to(torch.bfloat16).cuda()
    grid = 1
    qx = U.ufp4_quantize_grouped(tx, grid, counts, rht=True, rht_seed=2)
    qdyc = U.ufp4_quantize_grouped(tdy, grid, counts, rht=True, rht_seed=2, round=1, sr_seed=3, colwise=True)
    torch.cuda.synchronize()
    starts = np.concatenate([[0], np.cumsum(counts)])
    xo = U.grouped_offsets(counts, False)
    ko = U.grouped_offsets(counts, True)
    ts_x = q_ts = qx.tensor_scale.cpu().numpy()
    ts_dy = qdyc.tensor_scale.cpu().numpy()
    order = np.argsort(counts)
    for e in [int(order[-1]), int(order[len(order) // 2]), int(order[0])]:
        T = counts[e]
        if T == 0:
            continue
        seg = m["x"][starts[e]:starts[e] + T]
        rows = _sample(T, 8, e)
        A_t = oracle.tensor_amax(seg, rht=True, rht_seed=2)
        assert abs(ts_x[e] / float(np.float32(np.float32(A_t) / np.float32(1568))) - 1) <= 1e-6
        gc, _ = layouts.rows_of(qx, [xo[e] + r for r in rows])
        for i, r in enumerate(rows):
            ref = oracle.quantize(seg[r:r + 1], grid, rht=True, rht_seed=2, amax_in=A_t,
                                  elem_base=(xo[e] + int(r)) * H)
            assert (gc[i] != ref["codes"][0]).mean() <= 2e-3
        segd = m["dy"][starts[e]:starts[e] + T]
        A_d = oracle.tensor_amax(segd, rht=True, rht_seed=2, colwise=True)
        assert abs(ts_dy[e] / float(np.float32(np.float32(A_d) / np.float32(1568))) - 1) <= 1e-6
    # grouped fwd_y with RHT off: exact per-expert blocks
    qx0 = U.ufp4_quantize_grouped(tx, grid, counts)
    qw0 = U.ufp4_quantize_grouped(tw, grid, [F] * E)
    y = torch.zeros(sum(counts), F, device="cuda")
    wo = U.grouped_offsets([F] * E, False)
    groups = [dict(M=counts[e], N=F, K=H, a_row=xo[e], a_k=0, b_row=wo[e], b_k=0, a_seg=e, b_seg=e,
                   c=y[starts[e]:starts[e] + counts[e]] if counts[e] else y[:1]) for e in range(E)]
    U.ufp4_gemm_grouped(qx0, qw0, groups)
    torch.cuda.synchronize()
    yh = y.cpu().numpy()
    e = int(order[-1])
    T = counts[e]
    seg = m["x"][starts[e]:starts[e] + T]
    wseg = m["w"][e * F:(e + 1) * F]
    ms, ns = _sample(T, NS, 21), _sample(F, NS, 22)
    Ax, Aw = oracle.tensor_amax(seg), oracle.tensor_amax(wseg)
    qa = oracle.quantize(seg[ms], grid, amax_in=Ax)
    qb = oracle.quantize(wseg[ns], grid, amax_in=Aw)
    ref = oracle.gemm_f64(oracle.dequantize(qa["codes"], qa["scales"], qa["tensor_scale"], grid),
                          oracle.dequantize(qb["codes"], qb["scales"], qb["tensor_scale"], grid))
    got = yh[starts[e] + ms][:, ns]
    assert np.linalg.norm(got - ref) <= 1e-5 * np.linalg.norm(ref)


def test_moe124b_large_layer_full_size(U, oracle):
    """X 65536 x 8192, W 2048 x 8192, dY 65536 x 2048 (RHT off for exact
    GEMM blocks; the RHT path is covered by the tensor-scale check)."""
    dev = torch.device("cuda")
    x = inputs.device_normal((65536, 8192), 1.0, 31, dev)
    w = inputs.device_normal((2048, 8192), 0.01, 32, dev)
    grid = 1
    qx, qw = U.ufp4_quantize(x, grid), U.ufp4_quantize(w, grid)
    y = U.ufp4_gemm(qx, qw)
    qxr = U.ufp4_quantize(x, grid, rht=True, rht_seed=2)
    torch.cuda.synchronize()
    xh, wh = _f32(x), _f32(w)
    A_r = oracle.tensor_amax(xh, rht=True, rht_seed=2)
    assert abs(float(qxr.tensor_scale.item()) / float(np.float32(np.float32(A_r) / np.float32(1568))) - 1) <= 1e-6
    _check_rows(oracle, qx, xh, grid, _sample(65536, 8, 41), False, 0, 0, False)
    _gemm_block(oracle, grid, xh, wh, False, False, _sample(65536, NS, 42), _sample(2048, NS, 43), False,
                y.cpu().numpy(), 1e-5)


@pytest.mark.parametrize("grid", [0, 1])
def test_attenuation_chain_matches_oracle(U, oracle, grid):
    """A short compounding chain X_{k+1} = Q(X_k) Q(W_k)^T (re-quantized from
    fp32 each step): the GPU's prod eta tracks the oracle's, and E2M1 shrinks."""
    n, steps = 256, 8
    g = np.random.default_rng(9)
    X0 = inputs.to_bf16_f32(g.standard_normal((n, n), dtype=np.float32))
    Ws = [inputs.to_bf16_f32(g.standard_normal((n, n), dtype=np.float32) / np.float32(16))
          for _ in range(steps)]

    def eta(Y, X, W):
        Yr = X.astype(np.float64) @ W.astype(np.float64).T
        return float(np.vdot(Y, Yr) / np.vdot(Yr, Yr))

    Xg, Xo = X0.copy(), X0.copy()
    pg, po = 1.0, 1.0
    for W in Ws:
        qx = U.ufp4_quantize(torch.from_numpy(Xg).cuda(), grid)
        qw = U.ufp4_quantize(torch.from_numpy(W).to(torch.bfloat16).cuda(), grid)
        Yg = U.ufp4_gemm(qx, qw).cpu().numpy()
        pg *= eta(Yg.astype(np.float64), Xg, W)
        Xg = Yg.astype(np.float32)
        ra, rb = oracle.quantize(Xo, grid), oracle.quantize(W, grid)
        Yo = oracle.gemm_f64(oracle.dequantize(ra["codes"], ra["scales"], ra["tensor_scale"], grid),
                             oracle.dequantize(rb["codes"], rb["scales"], rb["tensor_scale"], grid))
        po *= eta(Yo, Xo, W)
        Xo = Yo.astype(np.float32)
    assert abs(pg / po - 1) <= 1e-3
    if grid == 0:
        assert pg < 0.99       # E2M1 attenuates
    else:
        assert abs(pg - 1) < 0.02
