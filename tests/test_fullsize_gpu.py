"""Parity at the workloads' full sizes, on sampled outputs.

The oracle computes each quantization's tensor amax over the whole tensor
(its own pass), then quantizes sampled output rows against that scale --
nothing it uses for the codes comes from the GPU.  Workloads: the dense-1.5B
training step and the MoE-124B large layer, each in the launch configuration
the benchmark times (E1M2, RHT on every operand, SR on dY, both orientations
from one read), and the MoE-7.9B grouped layer (64 experts, 16384 tokens x
top-6).  Bars (tests/parity.py): RHT off bit-exact codes and scales; RHT on
at most 1e-4 of the sampled codes one grid step apart, tensor scale 1e-6;
every GEMM within 1e-5 relative Frobenius of the fp64 product of the
operands it consumed, on sampled output blocks.
"""
import numpy as np
import pytest
import torch

import bench
from fp4_quantized_numerics_gb300 import inputs
from tests import layouts, parity

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


def _check_rows(oracle, q, x, grid, rows_sample, rht, rnd, sr_counter, colwise, tally=None):
    """Sampled output rows of GPU quantization q of host array x vs the
    oracle (its own tensor amax of the whole tensor).  With a tally the code
    bar is left to the caller."""
    A_t = oracle.tensor_amax(x, rht=rht, rht_seed=2, colwise=colwise)
    qmax = 6.0 if grid == 0 else 3.5
    ts = float(q.tensor_scale[0].item())
    want_ts = float(np.float32(np.float32(A_t) / np.float32(448 * qmax)))
    assert abs(ts / want_ts - 1) <= (1e-6 if rht else 0.0)
    gc, gs = layouts.rows_of(q, rows_sample)
    klen = x.shape[0] if colwise else x.shape[1]
    own = tally is None
    if own:
        tally = parity.CodeTally()
    for i, r in enumerate(rows_sample):
        vec = x[:, r] if colwise else x[r]
        ref = oracle.quantize(vec[None, :], grid, rht=rht, rht_seed=2, round_mode=rnd, sr_seed=3,
                              sr_counter=sr_counter, amax_in=A_t, elem_base=int(r) * klen)
        if not rht:
            np.testing.assert_array_equal(gc[i], ref["codes"][0])
            np.testing.assert_array_equal(gs[i], ref["scales"][0])
        else:
            tally.add(gc[i], ref["codes"][0])
    if rht and own:
        tally.check()


def _consumed_rows(oracle, q, rows, seg=0, k0=0, klen=None):
    """fp64 values of rows `rows`, k range [k0, k0 + klen), of GPU operand q
    (segment seg's tensor scale): what the GEMM multiplied."""
    codes, scales = layouts.rows_of(q, rows)
    klen = q.k - k0 if klen is None else klen
    ts = float(q.tensor_scale[seg].item())
    return oracle.dequantize(codes[:, k0:k0 + klen], scales[:, k0 // 16:(k0 + klen) // 16], ts, q.grid)


def _gemm_block_consumed(oracle, qa, qb, ms, ns, c_block, a_rows=None, b_rows=None, a_seg=0, b_seg=0,
                         a_k0=0, b_k0=0, K=None):
    """C block (rows ms, cols ns) against the fp64 product of the consumed
    operand rows (a_rows / b_rows: the operands' row indices, default ms / ns)."""
    A = _consumed_rows(oracle, qa, ms if a_rows is None else a_rows, a_seg, a_k0, K)
    B = _consumed_rows(oracle, qb, ns if b_rows is None else b_rows, b_seg, b_k0, K)
    parity.assert_gemm_close(c_block, oracle.gemm_f64(A, B))


def _gemm_block(oracle, grid, a, b, a_col, b_col, ms, ns, rht, c_gpu, tol, rnd_a=0, ctr=0):
    """C[ms][:, ns] of A B^T with A = quant(a) (a.T if a_col) vs the oracle's
    own quantization of the sampled rows (RHT off: bit-exact codes)."""
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


def _check_step(oracle, step, x, w, dy, seeds):
    """All six quantizations of a bench.Step (sampled rows vs the oracle) and
    its three GEMMs (sampled blocks vs the consumed operands)."""
    T, H = x.shape
    F = w.shape[0]
    g = step.grid
    s = iter(seeds)
    _check_rows(oracle, step.qx_r, x, g, _sample(T, NS, next(s)), True, 0, 0, False)
    _check_rows(oracle, step.qw_r, w, g, _sample(F, NS, next(s)), True, 0, 0, False)
    _check_rows(oracle, step.qdy_r, dy, g, _sample(T, NS, next(s)), True, 1, 0, False)
    _check_rows(oracle, step.qw_c, w, g, _sample(H, NS, next(s)), True, 0, 0, True)
    _check_rows(oracle, step.qdy_c, dy, g, _sample(F, NS, next(s)), True, 1, 0, True)
    _check_rows(oracle, step.qx_c, x, g, _sample(H, NS, next(s)), True, 0, 0, True)
    for qa, qb, c, (m, n) in ((step.qx_r, step.qw_r, step.y, (T, F)),      # fwd_y = X W^T
                              (step.qdy_r, step.qw_c, step.dx, (T, H)),    # bwd_dx = dY W
                              (step.qdy_c, step.qx_c, step.dw, (F, H))):   # bwd_dw = dY^T X
        ms, ns = _sample(m, NS, next(s)), _sample(n, NS, next(s))
        block = c[torch.as_tensor(ms, device=c.device)][:, torch.as_tensor(ns, device=c.device)]
        _gemm_block_consumed(oracle, qa, qb, ms, ns, block.cpu().numpy())


def test_dense_step_bench_configuration(U, oracle):
    """One step of the dense-1.5B workload, exactly as bench.py launches it:
    six codes checks and fwd_y, bwd_dx, bwd_dw at 1e-5."""
    d = inputs.device_dense(seed=0, device="cuda")
    step = bench.Step(U, d["x"], d["w"], d["dy"], U.UFP4_E1M2)
    step.quantize_all()
    step.gemms()
    torch.cuda.synchronize()
    _check_step(oracle, step, _f32(d["x"]), _f32(d["w"]), _f32(d["dy"]), range(1, 13))


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
    experts allowed), the benchmark's recipe: grouped RHT + E1M2
    quantization of X, W, dY both ways from one read per pass (SR on dY; each
    result equal to its own grouped call) and the three grouped GEMMs.  Sampled codes of three experts (largest, median, smallest
    nonzero) against the oracle, row-wise X and column-wise dY; sampled GEMM
    blocks of the same experts against the consumed operands; and the
    grouped fwd_y with RHT off against the oracle's own operands."""
    m = inputs.moe(seed=0)
    counts = [int(c) for c in m["counts"]]
    E, H, F = len(counts), 2048, 1408
    tx = torch.from_numpy(m["x"]).to(torch.bfloat16).cuda()
    tw = torch.from_numpy(m["w"]).to(torch.bfloat16).cuda()
    tdy = torch.from_numpy(m["dy"]).to(torch.bfloat16).cuda()
    grid = 1
    kw = dict(rht=True, rht_seed=2)
    wseg = [F] * E
    # both orientations of every operand from one read per pass, as the
    # benchmark launches them; each result equals its own grouped call
    qx, qxc = U.ufp4_quantize_grouped_dual(tx, grid, counts, **kw)
    qdy, qdyc = U.ufp4_quantize_grouped_dual(tdy, grid, counts, round=1, sr_seed=3, **kw)
    qw, qwc = U.ufp4_quantize_grouped_dual(tw, grid, wseg, **kw)
    for q, t, seg, col, extra in ((qx, tx, counts, False, {}), (qxc, tx, counts, True, {}),
                                  (qdy, tdy, counts, False, dict(round=1, sr_seed=3)),
                                  (qdyc, tdy, counts, True, dict(round=1, sr_seed=3)),
                                  (qw, tw, wseg, False, {}), (qwc, tw, wseg, True, {})):
        single = U.ufp4_quantize_grouped(t, grid, seg, colwise=col, **kw, **extra)
        assert torch.equal(q.codes, single.codes) and torch.equal(q.scales, single.scales)
        assert torch.equal(q.eplane, single.eplane) and torch.equal(q.tensor_scale, single.tensor_scale)
        del single
    T = sum(counts)
    y = torch.zeros(T, F, device="cuda")
    dx = torch.zeros(T, H, device="cuda")
    dw = torch.zeros(E * F, H, device="cuda")
    starts = np.concatenate([[0], np.cumsum(counts)])
    xo, ko = U.grouped_offsets(counts, False), U.grouped_offsets(counts, True)
    wo, wk = U.grouped_offsets(wseg, False), U.grouped_offsets(wseg, True)
    k16 = [(c + 15) // 16 * 16 for c in counts]
    U.ufp4_gemm_grouped(qx, qw, [dict(M=counts[e], N=F, K=H, a_row=xo[e], a_k=0, b_row=wo[e], b_k=0, a_seg=e,
                                      b_seg=e, c=y[starts[e]:starts[e] + counts[e]] if counts[e] else y[:1])
                                 for e in range(E)])
    U.ufp4_gemm_grouped(qdy, qwc, [dict(M=counts[e], N=H, K=F, a_row=xo[e], a_k=0, b_row=0, b_k=wk[e], a_seg=e,
                                        b_seg=e, c=dx[starts[e]:starts[e] + counts[e]] if counts[e] else dx[:1])
                                   for e in range(E)])
    U.ufp4_gemm_grouped(qdyc, qxc, [dict(M=F, N=H, K=k16[e], a_row=0, a_k=ko[e], b_row=0, b_k=ko[e], a_seg=e,
                                         b_seg=e, c=dw[e * F:(e + 1) * F]) for e in range(E)])
    torch.cuda.synchronize()
    ts_x = qx.tensor_scale.cpu().numpy()
    ts_dy = qdyc.tensor_scale.cpu().numpy()
    ktot = qdyc.k
    order = np.argsort(counts)
    nonzero = [int(e) for e in order if counts[e] > 0]
    tally_x, tally_dy = parity.CodeTally(), parity.CodeTally()
    yh, dxh, dwh = y.cpu().numpy(), dx.cpu().numpy(), dw.cpu().numpy()
    for e in sorted({nonzero[-1], nonzero[len(nonzero) // 2], nonzero[0]}):
        Te = counts[e]
        seg = m["x"][starts[e]:starts[e] + Te]
        A_t = oracle.tensor_amax(seg, rht=True, rht_seed=2)
        assert abs(ts_x[e] / float(np.float32(np.float32(A_t) / np.float32(1568))) - 1) <= 1e-6
        rows = _sample(Te, 8, e)
        gc, _ = layouts.rows_of(qx, [xo[e] + r for r in rows])
        for i, r in enumerate(rows):
            ref = oracle.quantize(seg[r:r + 1], grid, rht=True, rht_seed=2, amax_in=A_t,
                                  elem_base=(xo[e] + int(r)) * H)
            tally_x.add(gc[i], ref["codes"][0])
        # column-wise dY: rows of the result are columns of dY_e, tokens
        # zero-padded to 16, SR index c * Ktot + koff_e + t
        segd = np.zeros((k16[e], F), np.float32)
        segd[:Te] = m["dy"][starts[e]:starts[e] + Te]
        A_d = oracle.tensor_amax(segd, rht=True, rht_seed=2, colwise=True)
        assert abs(ts_dy[e] / float(np.float32(np.float32(A_d) / np.float32(1568))) - 1) <= 1e-6
        cols = _sample(F, 8, 100 + e)
        gc, _ = layouts.rows_of(qdyc, cols)
        for i, c in enumerate(cols):
            ref = oracle.quantize(segd[:, c][None, :], grid, rht=True, rht_seed=2, round_mode=1, sr_seed=3,
                                  amax_in=A_d, elem_base=int(c) * ktot + ko[e])
            tally_dy.add(gc[i][ko[e]:ko[e] + k16[e]], ref["codes"][0])
        # the three GEMMs of expert e on sampled blocks
        ms, ns = _sample(Te, NS, 200 + e), _sample(F, NS, 300 + e)
        _gemm_block_consumed(oracle, qx, qw, ms, ns, yh[starts[e] + ms][:, ns], a_rows=xo[e] + ms,
                             b_rows=wo[e] + ns, a_seg=e, b_seg=e)
        ns = _sample(H, NS, 400 + e)
        _gemm_block_consumed(oracle, qdy, qwc, ms, ns, dxh[starts[e] + ms][:, ns], a_rows=xo[e] + ms,
                             a_seg=e, b_seg=e, b_k0=wk[e], K=F)
        ms = _sample(F, NS, 500 + e)
        _gemm_block_consumed(oracle, qdyc, qxc, ms, ns, dwh[e * F + ms][:, ns], a_seg=e, b_seg=e,
                             a_k0=ko[e], b_k0=ko[e], K=k16[e])
    tally_x.check()
    tally_dy.check()
    # grouped fwd_y with RHT off: exact per-expert blocks
    qx0 = U.ufp4_quantize_grouped(tx, grid, counts)
    qw0 = U.ufp4_quantize_grouped(tw, grid, wseg)
    y0 = torch.zeros(T, F, device="cuda")
    groups = [dict(M=counts[e], N=F, K=H, a_row=xo[e], a_k=0, b_row=wo[e], b_k=0, a_seg=e, b_seg=e,
                   c=y0[starts[e]:starts[e] + counts[e]] if counts[e] else y0[:1]) for e in range(E)]
    U.ufp4_gemm_grouped(qx0, qw0, groups)
    torch.cuda.synchronize()
    e = nonzero[-1]
    Te = counts[e]
    seg = m["x"][starts[e]:starts[e] + Te]
    wseg_e = m["w"][e * F:(e + 1) * F]
    ms, ns = _sample(Te, NS, 21), _sample(F, NS, 22)
    Ax, Aw = oracle.tensor_amax(seg), oracle.tensor_amax(wseg_e)
    qa = oracle.quantize(seg[ms], grid, amax_in=Ax)
    qb = oracle.quantize(wseg_e[ns], grid, amax_in=Aw)
    ref = oracle.gemm_f64(oracle.dequantize(qa["codes"], qa["scales"], qa["tensor_scale"], grid),
                          oracle.dequantize(qb["codes"], qb["scales"], qb["tensor_scale"], grid))
    parity.assert_gemm_close(y0.cpu().numpy()[starts[e] + ms][:, ns], ref)


def test_moe124b_large_layer_full_size(U, oracle):
    """X 65536 x 8192, W 2048 x 8192, dY 65536 x 2048: the benchmark's step
    (E1M2, RHT on every operand, SR on dY, dual quantization), sampled codes
    of all six quantizations and the three GEMMs -- bwd_dw with K = 65536 --
    at 1e-5 against the consumed operands; then fwd_y with RHT off against
    the oracle's own operands."""
    dev = torch.device("cuda")
    d = bench.moe124b_inputs(dev)
    step = bench.Step(U, d["x"], d["w"], d["dy"], U.UFP4_E1M2)
    step.quantize_all()
    step.gemms()
    torch.cuda.synchronize()
    xh, wh, dyh = _f32(d["x"]), _f32(d["w"]), _f32(d["dy"])
    _check_step(oracle, step, xh, wh, dyh, range(41, 53))
    del step
    torch.cuda.empty_cache()
    grid = 1
    qx, qw = U.ufp4_quantize(d["x"], grid), U.ufp4_quantize(d["w"], grid)
    y = U.ufp4_gemm(qx, qw)
    torch.cuda.synchronize()
    _check_rows(oracle, qx, xh, grid, _sample(65536, 8, 61), False, 0, 0, False)
    _gemm_block(oracle, grid, xh, wh, False, False, _sample(65536, NS, 62), _sample(2048, NS, 63), False,
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
