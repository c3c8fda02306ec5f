"""Benchmark of the UFP4 hot path on GB300.

One step = one UFP4 training step of the dense-1.5B-shaped linear layer
(X 8192 x 2048, W 5632 x 2048, dY 8192 x 5632, BF16, seeded synthetic data):
six fused RHT + E1M2 quantizations (X, W, dY, each row-wise and
column-wise; stochastic rounding on dY only) followed by the three training
GEMMs fwd_y = X W^T, bwd_dx = dY W and bwd_dw = dY^T X.

Reported (one JSON line from rank 0):
  value         fused RHT+quantize throughput, GB/s of algorithmic traffic
                (2 B read + 0.5625 B written per element) over the
                quantization launches of the step (tensor-amax pass included
                in the time, not in the bytes);
  gemm          GEMM TFLOP/s (2 M N K logical flops) and fractions of the
                FP8 / FP4 dense peaks;
  roofline      for the dominant kernel by time (the E1M2 GEMM);
  e2e           the same metric through the public API with the inputs
                copied from pinned host memory each step and the three GEMM
                outputs read back;
  cpu_baseline  the CPU oracle on a bounded sample of the same step.
L2 is flushed before every timed step, outside the events: a 256 MiB buffer
is written and then read back, so the timed kernels start with an L2 that
holds none of their data and no dirty lines whose write-back would compete
with their reads.

--impl reference runs the CPU oracle (the reference arm of this tier) on a
bounded sample of the same workload and prints the same line shape.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = dict(name="dense1p5b_linear_train_step", tokens=8192, hidden=2048, ffn=5632)
METRIC = ("fused RHT+quantize GB/s (% HBM peak); FP4 GEMM TFLOPS (% tensor peak)")
Q_BYTES_PER_ELEM = 2.0 + 0.5 + 1.0 / 16.0
FALLBACK = dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
        except (OSError, ValueError):
            d = {}
        # the figures may sit at the top level or one level down
        dicts = [d] + [v for v in d.values() if isinstance(v, dict)] if isinstance(d, dict) else []

        def pick(*keys):
            for dd in dicts:
                for k in keys:
                    if k in dd and isinstance(dd[k], (int, float)) and not isinstance(dd[k], bool) and dd[k] > 0:
                        return float(dd[k])
            return None
        hbm = pick("hbm_gbs", "hbm_GBps", "copy_gbs")
        bf = pick("bf16_tflops", "bf16_tflops_burst")
        bfs = pick("bf16_tflops_sustained")
        if hbm and bf:
            return dict(hbm_gbs=hbm, bf16_tflops=bf, bf16_tflops_sustained=bfs or bf,
                        source="measured")
    return dict(FALLBACK, source="fallback")


def reduce_max(v, world, device="cpu"):
    """Max of a per-rank float over all ranks (one all-reduce; no-op at 1)."""
    if world == 1:
        return float(v)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_rate(units_per_rank, world, steps, max_ms, scale=1e9):
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time (each rank runs its own copy of the workload)."""
    return world * steps * units_per_rank / (max_ms * 1e-3) / scale


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [t.strip() for t in l.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


class L2Flush:
    """Evicts the timed kernels' data from L2: writes a 256 MiB buffer (more
    than the 129 MB L2), then reads it back so the dirty lines are written
    back before the timed region instead of during it."""

    def __init__(self, dev):
        import torch
        self.buf = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)
        self.n = 0

    def __call__(self):
        self.n += 1
        self.buf.fill_(float(self.n & 0xFF))
        self.buf.sum()


# ------------------------------------------------------------- the step
class Step:
    """Buffers and launches of one UFP4 training step (E1M2 + RHT on all
    GEMM operands, SR on dY), all through the libufp4 binding."""

    def __init__(self, U, x, w, dy, grid, dual=True, policy="ufp4"):
        import torch
        self.U, self.torch = U, torch
        self.x, self.w, self.dy = x, w, dy
        self.grid = grid
        T, H = x.shape
        F = w.shape[0]
        dev = x.device
        Q = U.QTensor.empty
        self.qx_r, self.qw_r, self.qdy_r = Q(T, H, grid, dev), Q(F, H, grid, dev), Q(T, F, grid, dev)
        self.qw_c, self.qdy_c, self.qx_c = Q(H, F, grid, dev), Q(F, T, grid, dev), Q(H, T, grid, dev)
        self.y = torch.empty(T, F, dtype=torch.float32, device=dev)
        self.dx = torch.empty(T, H, dtype=torch.float32, device=dev)
        self.dw = torch.empty(F, H, dtype=torch.float32, device=dev)
        self.ws = U.workspace(dev)
        self.counter = 0
        # "nvfp4": the transform only on the bwd_dw operands (dY^T, X^T); the
        # two orientations then differ and are quantized one pass each
        self.policy = policy
        self.dual = dual and policy == "ufp4"
        self.launches_per_step = (3 if self.dual else 6) * 2 + 3
        self.q_elems = 2 * (x.numel() + w.numel() + dy.numel())
        self.flops_each = [2 * T * F * H, 2 * T * H * F, 2 * F * H * T]

    def quantize_all(self):
        U, g = self.U, self.grid
        kw = dict(rht=True, rht_seed=2, ws=self.ws)
        if self.dual:
            # each operand in both orientations from one read per pass
            U.ufp4_quantize_dual(self.x, g, out_row=self.qx_r, out_col=self.qx_c, **kw)
            U.ufp4_quantize_dual(self.w, g, out_row=self.qw_r, out_col=self.qw_c, **kw)
            U.ufp4_quantize_dual(self.dy, g, round=U.UFP4_SR, sr_seed=3, sr_counter_row=self.counter,
                                 sr_counter_col=self.counter, out_row=self.qdy_r, out_col=self.qdy_c, **kw)
            self.counter += 1
            return
        sr = dict(round=U.UFP4_SR, sr_seed=3, sr_counter=self.counter)
        kn = dict(kw, rht=False) if self.policy == "nvfp4" else kw   # fwd_y / bwd_dx operands
        U.ufp4_quantize(self.x, g, out=self.qx_r, **kn)
        U.ufp4_quantize(self.w, g, out=self.qw_r, **kn)
        U.ufp4_quantize(self.dy, g, out=self.qdy_r, **kn, **sr)
        U.ufp4_quantize(self.w, g, colwise=True, out=self.qw_c, **kn)
        U.ufp4_quantize(self.dy, g, colwise=True, out=self.qdy_c, **kw, **sr)
        U.ufp4_quantize(self.x, g, colwise=True, out=self.qx_c, **kw)
        self.counter += 1

    def gemms(self, events=None):
        U = self.U
        pairs = [(self.qx_r, self.qw_r, self.y), (self.qdy_r, self.qw_c, self.dx),
                 (self.qdy_c, self.qx_c, self.dw)]
        for i, (a, b, c) in enumerate(pairs):
            U.ufp4_gemm(a, b, out=c)
            if events is not None:
                events[i + 1].record()



def run_gpu(args):
    import torch
    from fp4_quantized_numerics_gb300 import build, inputs, ufp4 as U

    ws_n, rank, local = dist_env()
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    build.build()
    U.lib()
    dev = torch.device("cuda", local)
    pk = peaks()

    d = inputs.device_dense(seed=rank, tokens=WORKLOAD["tokens"], hidden=WORKLOAD["hidden"],
                            ffn=WORKLOAD["ffn"], device=dev)
    step = Step(U, d["x"], d["w"], d["dy"], U.UFP4_E1M2)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        step.quantize_all()
        step.gemms()
    torch.cuda.synchronize()

    # per-step events: [start, after quantize, after gemm0, gemm1, gemm2]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    if ws_n > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush()
            e = evs[i]
            e[0].record()
            step.quantize_all()
            e[1].record()
            step.gemms(events=[None, e[2], e[3], e[4]])
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if ws_n > 1:
        torch.distributed.barrier()
    q_ms = [e[0].elapsed_time(e[1]) for e in evs]
    g_ms = [[e[1 + j].elapsed_time(e[2 + j]) for j in range(3)] for e in evs]
    step_ms = [e[0].elapsed_time(e[4]) for e in evs]
    tq, tg, tstep = sum(q_ms), sum(sum(g) for g in g_ms), sum(step_ms)

    def allmax(v):
        return reduce_max(v, ws_n, dev)

    tq, tg, tstep = allmax(tq), allmax(tg), allmax(tstep)
    q_bytes = step.q_elems * Q_BYTES_PER_ELEM
    q_gbs = weak_scaling_rate(q_bytes, ws_n, args.steps, tq)
    flops = sum(step.flops_each)
    gemm_tflops = weak_scaling_rate(flops, ws_n, args.steps, tg, 1e12)
    per_gpu_tflops = gemm_tflops / ws_n
    fp8_peak = pk["bf16_tflops"] * 2.0    # nominal dense ratio fp8:bf16 = 4.5 : 2.25
    fp4_peak = pk["bf16_tflops"] * 6.0    # nominal dense ratio fp4:bf16 = 13.5 : 2.25
    gemm_each = [sum(g[j] for g in g_ms) / args.steps for j in range(3)]

    # ---------------------------------------------------- e2e through the API
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, U, step, d, dev, q_bytes)
        e2e["value"] = allmax(e2e["time_s"])
        e2e["value"] = ws_n * e2e["steps"] * q_bytes / e2e["value"] / 1e9
        del e2e["time_s"]

    extra = {}
    if not args.quick:
        extra = side_measurements(U, torch, dev, pk, flush)
        # the same quantize phase with one pass per orientation (six
        # single-orientation calls instead of three dual ones)
        single = Step(U, d["x"], d["w"], d["dy"], U.UFP4_E1M2, dual=False)
        for _ in range(3):
            single.quantize_all()
        tot = 0.0
        for _ in range(20):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(); single.quantize_all(); b.record()
            torch.cuda.synchronize()
            tot += a.elapsed_time(b)
        extra["quantize_step_single_orientation"] = {
            "gbs": round(q_bytes / (tot / 20 * 1e-3) / 1e9, 1), "ms": round(tot / 20, 4),
            "launches": single.launches_per_step - 3}
        del single

    if rank == 0:
        clocks = clk.summary()
        line = {
            "metric": METRIC, "value": round(q_gbs, 2), "unit": "GB/s",
            "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tstep / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp32 quantize / e2m1-plane MMA, f32 accumulate",
            "data": "synthetic (seeded N(0,1)/N(0,0.02)/N(0,1e-3) BF16; 1 outlier column x50)",
            "config": {"workload": WORKLOAD["name"], "X": [WORKLOAD["tokens"], WORKLOAD["hidden"]],
                       "W": [WORKLOAD["ffn"], WORKLOAD["hidden"]],
                       "dY": [WORKLOAD["tokens"], WORKLOAD["ffn"]],
                       "recipe": "UFP4: E1M2, RHT16 on all GEMM operands, SR on dY",
                       "l2": "flushed before every timed step (256 MiB write, then read back)",
                       "parallelism": "replicas" if ws_n > 1 else "single"},
            "quantize": {"gbs": round(q_gbs, 1), "frac_hbm": round(q_gbs / ws_n / pk["hbm_gbs"], 4),
                         "ms_per_step": round(tq / args.steps, 4),
                         "elements_per_step": step.q_elems,
                         "launches_per_step": step.launches_per_step - 3},
            "gemm": {"tflops": round(gemm_tflops, 1), "ms_per_step": round(tg / args.steps, 4),
                     "ms_each": [round(v, 4) for v in gemm_each],
                     "frac_fp8_peak": round(per_gpu_tflops / fp8_peak, 4),
                     "frac_fp4_peak": round(per_gpu_tflops / fp4_peak, 4)},
            "roofline": {"bound": "tensor", "kernel": "k_gemm<E1M2, E planes loaded>",
                         "achieved": round(per_gpu_tflops, 1), "peak": round(fp8_peak, 1),
                         "unit": "TFLOP/s", "frac": round(per_gpu_tflops / fp8_peak, 4),
                         "traffic": traffic_for("k_gemm_e1m2_dense1p5b"),
                         "peak_kind": "dense FP8 = %s bf16 x 2 (%s)" % ("measured" if pk["source"] == "measured" else "fallback", pk["source"])},
            "gpu_launches": step.launches_per_step * args.steps,
            "clocks": clocks,
            "peaks": pk,
        }
        if e2e is not None:
            line["e2e"] = e2e
        line.update(extra)
        if not args.no_cpu_baseline and ws_n >= 1:
            line["cpu_baseline"] = cpu_baseline(args)
        print(json.dumps(line), flush=True)
    if ws_n > 1:
        torch.distributed.destroy_process_group()


def run_e2e(args, U, step, d, dev, q_bytes):
    """The public API end to end: every step copies its inputs from pinned
    host memory to the device, runs the full step and copies its results
    (y, dx, dw) back to pinned host memory, all inside the timed region.
    Steps alternate between two buffer sets and three streams (host-to-device
    copies, compute, device-to-host copies), so the copies of one step
    overlap the compute of its neighbours, as a training loop would."""
    import torch
    hx = d["x"].cpu().pin_memory()
    hw = d["w"].cpu().pin_memory()
    hdy = d["dy"].cpu().pin_memory()
    twin = Step(U, torch.empty_like(step.x), torch.empty_like(step.w), torch.empty_like(step.dy), step.grid)
    sets = [step, twin]
    outs = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (st.y, st.dx, st.dw)] for st in sets]
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in sets]
    ev_cmp = [torch.cuda.Event() for _ in sets]
    ev_out = [torch.cuda.Event() for _ in sets]
    torch.cuda.synchronize()

    def launch(i):
        k = i % 2
        st = sets[k]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_cmp[k])     # step i-2 is done with this set's inputs
            st.x.copy_(hx, non_blocking=True)
            st.w.copy_(hw, non_blocking=True)
            st.dy.copy_(hdy, non_blocking=True)
            ev_in[k].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(ev_in[k])
            if i >= 2:
                s_cmp.wait_event(ev_out[k])    # step i-2's results have left this set
            st.quantize_all()
            st.gemms()
            ev_cmp[k].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[k])
            for h, t in zip(outs[k], (st.y, st.dx, st.dw)):
                h.copy_(t, non_blocking=True)
            ev_out[k].record(s_out)

    n = max(4, min(args.steps, 20))
    for i in range(2):
        launch(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(2, 2 + n):
        launch(i)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    h2d = sum(t.numel() * t.element_size() for t in (hx, hw, hdy))
    d2h = sum(t.numel() * t.element_size() for t in outs[0])
    del twin
    return {"time_s": dt, "steps": n, "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(dt / n * 1e3, 3),
            "overlap": "2 buffer sets, copy-in / compute / copy-out streams"}


def side_measurements(U, torch, dev, pk, flush):
    """Secondary numbers: RHT on/off overhead of the E1M2 quantizer, the
    outlier-heavy 4096 x 4096 quantization, and the E2M1 GEMM."""
    from fp4_quantized_numerics_gb300 import inputs

    def timeit(fn, n=30):
        # median of n timed runs (each after an L2 flush)
        fn(); fn(); fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(n):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(); fn(); b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return sorted(ts)[len(ts) // 2]

    out = {}
    x = inputs.device_normal((8192, 2048), 1.0, 11, dev)
    # the quantizer alone (codes and scales, no E1M2 correction plane)
    q = U.QTensor.empty(8192, 2048, U.UFP4_E1M2, dev, eplane=False)
    amax = torch.ones(1, device=dev)
    ws = U.workspace(dev)
    el = x.numel()
    r = {}
    for rht in (False, True):
        for name, am in (("with_amax_pass", None), ("amax_given", amax)):
            ms = timeit(lambda: U.ufp4_quantize(x, U.UFP4_E1M2, rht=rht, out=q, ws=ws, amax_in=am))
            r["rht_%s_%s" % ("on" if rht else "off", name)] = round(el * Q_BYTES_PER_ELEM / (ms * 1e-3) / 1e9, 1)
    r["rht_overhead_amax_given"] = round(r["rht_off_amax_given"] / r["rht_on_amax_given"] - 1, 4)
    r["frac_hbm_rht_on_amax_given"] = round(r["rht_on_amax_given"] / pk["hbm_gbs"], 4)
    out["quantize_x_8192x2048_gbs"] = r

    # steady state on a large operand (512 MB of BF16): one orientation and
    # both, transform on, E1M2 RTNE
    xl = inputs.device_normal((32768, 8192), 1.0, 15, dev)
    ql = U.QTensor.empty(32768, 8192, U.UFP4_E1M2, dev, eplane=False)
    qlc = U.QTensor.empty(8192, 32768, U.UFP4_E1M2, dev, eplane=False)
    aml = torch.tensor([float(xl.float().abs().max()) * 1.25], device=dev)
    L = {}
    ms = timeit(lambda: U.ufp4_quantize(xl, U.UFP4_E1M2, rht=True, out=ql, ws=ws, amax_in=aml), 10)
    L["single_amax_given"] = round(xl.numel() * Q_BYTES_PER_ELEM / (ms * 1e-3) / 1e9, 1)
    ms = timeit(lambda: U.ufp4_quantize(xl, U.UFP4_E1M2, rht=False, out=ql, ws=ws, amax_in=aml), 10)
    L["single_amax_given_rht_off"] = round(xl.numel() * Q_BYTES_PER_ELEM / (ms * 1e-3) / 1e9, 1)
    L["rht_overhead_amax_given"] = round(L["single_amax_given_rht_off"] / L["single_amax_given"] - 1, 4)
    ms = timeit(lambda: U.ufp4_quantize(xl, U.UFP4_E1M2, rht=True, out=ql, ws=ws), 10)
    L["single_with_amax_pass"] = round(xl.numel() * Q_BYTES_PER_ELEM / (ms * 1e-3) / 1e9, 1)
    ms = timeit(lambda: U.ufp4_quantize_dual(xl, U.UFP4_E1M2, rht=True, amax_row=aml, amax_col=aml, out_row=ql,
                                             out_col=qlc, ws=ws), 10)
    L["dual_amax_given"] = round(2 * xl.numel() * Q_BYTES_PER_ELEM / (ms * 1e-3) / 1e9, 1)
    L["dual_amax_given_dram_gbs"] = round(xl.numel() * (2 + 2 * 0.5625) / (ms * 1e-3) / 1e9, 1)
    ms = timeit(lambda: U.ufp4_quantize_dual(xl, U.UFP4_E1M2, rht=True, out_row=ql, out_col=qlc, ws=ws), 10)
    L["dual_with_amax_pass"] = round(2 * xl.numel() * Q_BYTES_PER_ELEM / (ms * 1e-3) / 1e9, 1)
    L["frac_hbm_single_amax_given"] = round(L["single_amax_given"] / pk["hbm_gbs"], 4)
    # the same with the correction plane written too (+0.5 B/elem, not counted)
    qle = U.QTensor.empty(32768, 8192, U.UFP4_E1M2, dev)
    ms = timeit(lambda: U.ufp4_quantize(xl, U.UFP4_E1M2, rht=True, out=qle, ws=ws, amax_in=aml), 10)
    L["single_amax_given_with_eplane"] = round(xl.numel() * Q_BYTES_PER_ELEM / (ms * 1e-3) / 1e9, 1)
    del qle
    out["quantize_large_32768x8192_e1m2_rht_gbs"] = L
    del xl, ql, qlc

    xo = inputs.device_normal((4096, 4096), 1.0, 12, dev)
    qo = U.QTensor.empty(4096, 4096, U.UFP4_E2M1, dev)
    qo1 = U.QTensor.empty(4096, 4096, U.UFP4_E1M2, dev, eplane=False)
    o = {}
    for g, qq in ((U.UFP4_E2M1, qo), (U.UFP4_E1M2, qo1)):
        ms = timeit(lambda: U.ufp4_quantize(xo, g, rht=True, out=qq, ws=ws))
        o["e2m1" if g == 0 else "e1m2"] = round(xo.numel() * Q_BYTES_PER_ELEM / (ms * 1e-3) / 1e9, 1)
    out["quantize_outlier_4096x4096_rht_gbs"] = o

    # E2M1 GEMM at the fwd_y shape
    a = U.ufp4_quantize(inputs.device_normal((8192, 2048), 1.0, 13, dev), U.UFP4_E2M1)
    b = U.ufp4_quantize(inputs.device_normal((5632, 2048), 0.02, 14, dev), U.UFP4_E2M1)
    c = torch.empty(8192, 5632, dtype=torch.float32, device=dev)
    ms = timeit(lambda: U.ufp4_gemm(a, b, out=c))
    tf = 2 * 8192 * 5632 * 2048 / (ms * 1e-3) / 1e12
    out["gemm_e2m1_fwd_y"] = {"tflops": round(tf, 1), "frac_fp4_peak": round(tf / (pk["bf16_tflops"] * 6), 4),
                              "output_bytes_bound_tflops": round(2 * 2048 / 4 * pk["hbm_gbs"] / 1e3, 1)}
    # E1M2 at the fwd_y shape: correction planes loaded vs expanded on chip
    a = U.ufp4_quantize(inputs.device_normal((8192, 2048), 1.0, 13, dev), U.UFP4_E1M2, rht=True)
    b = U.ufp4_quantize(inputs.device_normal((5632, 2048), 0.02, 14, dev), U.UFP4_E1M2, rht=True)
    e = {}
    for name, (qa, qb) in (("eplanes_loaded", (a, b)),
                           ("expanded_on_chip", tuple(U.QTensor(t.codes, t.scales, t.tensor_scale, t.rows, t.k,
                                                                t.grid) for t in (a, b)))):
        ms = timeit(lambda: U.ufp4_gemm(qa, qb, out=c))
        e[name] = round(2 * 8192 * 5632 * 2048 / (ms * 1e-3) / 1e12, 1)
    out["gemm_e1m2_fwd_y_tflops"] = e
    return out


def traffic_for(key):
    """dram bytes per launch from a committed ncu summary, if its kernel
    source hash still matches the current source (else null)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(key)
    if not ent:
        return None
    src = os.path.join(ROOT, "fp4_quantized_numerics_gb300", "csrc", ent.get("source", ""))
    if not os.path.exists(src):
        return None
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return ent.get("bytes_per_launch") if h == ent.get("sha256_16") else None


# ------------------------------------------------------------ CPU oracle
def cpu_sample(rows_x=2048, rows_dy=2048, gemm_rows=32):
    """The oracle on a bounded sample of the step: RHT + E1M2 row-wise
    quantization of the first rows of X and of dY (SR), and gemm_rows rows of
    fwd_y in fp64.  Returns (quantize GB/s, GEMM GFLOP/s, seconds, desc)."""
    from fp4_quantized_numerics_gb300 import inputs
    from oracle import oracle
    g = np.random.default_rng(0)
    x = inputs.to_bf16_f32(g.standard_normal((rows_x, WORKLOAD["hidden"]), dtype=np.float32))
    dy = inputs.to_bf16_f32(g.standard_normal((rows_dy, WORKLOAD["ffn"]), dtype=np.float32) * np.float32(1e-3))
    w = inputs.to_bf16_f32(g.standard_normal((WORKLOAD["ffn"], WORKLOAD["hidden"]), dtype=np.float32) * np.float32(0.02))
    t0 = time.perf_counter()
    rx = oracle.quantize(x, oracle.E1M2, rht=True, rht_seed=2)
    oracle.quantize(dy, oracle.E1M2, rht=True, rht_seed=2, round_mode=oracle.SR, sr_seed=3)
    tq = time.perf_counter() - t0
    rw = oracle.quantize(w, oracle.E1M2, rht=True, rht_seed=2)
    A = oracle.dequantize(rx["codes"][:gemm_rows], rx["scales"][:gemm_rows], rx["tensor_scale"], oracle.E1M2)
    B = oracle.dequantize(rw["codes"], rw["scales"], rw["tensor_scale"], oracle.E1M2)
    t1 = time.perf_counter()
    oracle.gemm_f64(A, B)
    tg = time.perf_counter() - t1
    el = x.size + dy.size
    flops = 2.0 * gemm_rows * w.shape[0] * w.shape[1]
    desc = ("RHT+E1M2 row-wise quantization of %d x %d of X and %d x %d of dY (SR), "
            "plus %d rows of fwd_y in fp64" % (rows_x, WORKLOAD["hidden"], rows_dy, WORKLOAD["ffn"], gemm_rows))
    return el * Q_BYTES_PER_ELEM / tq / 1e9, flops / tg / 1e9, tq + tg, desc


def cpu_baseline(args):
    gbs, gflops, secs, desc = cpu_sample()
    return {"value": round(gbs, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": desc, "gemm_gflops": round(gflops, 3), "seconds": round(secs, 2),
            "host": host_desc()}


def host_desc():
    try:
        import platform
        return "%s, %d logical cores" % (platform.machine(), os.cpu_count() or 0)
    except Exception:
        return None


def run_reference(args):
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return
    t_all = 0.0
    vals = []
    for i in range(args.warmup + args.steps):
        gbs, gflops, secs, desc = cpu_sample(rows_x=256, rows_dy=256, gemm_rows=4)
        if i >= args.warmup:
            t_all += secs
            vals.append(gbs)
    value = statistics.mean(vals) if vals else 0.0
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "GB/s",
            "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t_all / max(args.steps, 1) * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64/f32 (CPU oracle)",
            "data": "synthetic", "config": {"workload": WORKLOAD["name"]},
            "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_kernel(args):
    """One kernel of the step in isolation, for profiling: `steps` launches
    of the fwd_y GEMM (8192 x 5632 x 2048), of the RHT quantization of X
    (8192 x 2048) in one orientation or both (quant_dual_*; the SR variant
    quantizes dY, 8192 x 5632), after `warmup` launches, the tensor amax
    given.  Prints the mean event time."""
    import torch
    from fp4_quantized_numerics_gb300 import build, inputs, ufp4 as U
    build.build()
    dev = torch.device("cuda", 0)
    T, H, F = WORKLOAD["tokens"], WORKLOAD["hidden"], WORKLOAD["ffn"]
    x = inputs.device_normal((T, H), 1.0, 21, dev)
    kind = args.kernel
    if kind.startswith("gemm"):
        grid = U.UFP4_E2M1 if kind == "gemm_e2m1" else U.UFP4_E1M2
        w = inputs.device_normal((F, H), 0.02, 22, dev)
        a, b = U.ufp4_quantize(x, grid, rht=True), U.ufp4_quantize(w, grid, rht=True)
        c = torch.empty(T, F, dtype=torch.float32, device=dev)
        fn = lambda: U.ufp4_gemm(a, b, out=c)
        work = 2.0 * T * F * H
        unit = "TFLOP/s"
    elif kind.startswith("quant_dual"):
        # both orientations from one read; SR variant on the dY shape
        grid = U.UFP4_E1M2
        sr = kind.startswith("quant_dual_sr")
        src = inputs.device_normal((T, F), 1e-3, 23, dev) if sr else x
        am = torch.tensor([float(src.float().abs().max()) * 1.5], device=dev)
        qr = U.QTensor.empty(src.shape[0], src.shape[1], grid, dev)
        qc = U.QTensor.empty(src.shape[1], src.shape[0], grid, dev)
        kw = dict(round=U.UFP4_SR, sr_seed=3) if sr else {}
        fn = lambda: U.ufp4_quantize_dual(src, grid, rht=True, amax_row=am, amax_col=am, out_row=qr,
                                          out_col=qc, **kw)
        work = 2 * src.numel() * Q_BYTES_PER_ELEM
        unit = "GB/s"
    else:
        grid = U.UFP4_E2M1 if kind.endswith("e2m1") else U.UFP4_E1M2
        col = kind.startswith("quant_col")
        q = U.QTensor.empty(H if col else T, T if col else H, grid, dev)
        am = torch.tensor([float(x.float().abs().max()) * 1.5], device=dev)
        fn = lambda: U.ufp4_quantize(x, grid, rht=True, colwise=col, out=q, amax_in=am)
        work = x.numel() * Q_BYTES_PER_ELEM
        unit = "GB/s"
    flush = L2Flush(dev)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    tot = 0.0
    for _ in range(args.steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(); fn(); e1.record()
        torch.cuda.synchronize()
        tot += e0.elapsed_time(e1)
    ms = tot / args.steps
    rate = work / (ms * 1e-3) / (1e12 if unit == "TFLOP/s" else 1e9)
    print(json.dumps({"kernel": kind, "ms": round(ms, 4), "rate": round(rate, 1), "unit": unit}))



# ------------------------------------------------------------ all workloads
def _ev_time(fn, flush, reps=10):
    import torch
    fn()
    torch.cuda.synchronize()
    tot = 0.0
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(); fn(); b.record()
        torch.cuda.synchronize()
        tot += a.elapsed_time(b)
    return tot / reps


def run_workloads(args):
    """Every synthetic workload at 1 GPU: quantizer GB/s, GEMM TFLOP/s and the
    numerics the pages discuss (alpha, SQNR, bias, prod eta).  One JSON line
    per workload."""
    import torch
    from fp4_quantized_numerics_gb300 import build, inputs, ufp4 as U
    build.build()
    dev = torch.device("cuda", 0)
    pk = peaks()
    flush = L2Flush(dev)
    out = []

    def emit(d):
        print(json.dumps(d), flush=True)
        out.append(d)

    def stats_of(x, grid, rht):
        q = U.ufp4_quantize(x, grid, rht=rht, rht_seed=2)
        st = U.ufp4_stats(x, q, rht=rht, rht_seed=2)
        return {k: round(st[k], 6) for k in ("alpha", "sqnr_db", "mean_bias")}

    # smoke: 256 x 1024 tensor, 256^3 GEMM
    d = inputs.smoke(0)
    x = torch.from_numpy(d["x"]).to(torch.bfloat16).to(dev)
    a = torch.from_numpy(d["a"]).to(torch.bfloat16).to(dev)
    b = torch.from_numpy(d["b"]).to(torch.bfloat16).to(dev)
    r = {"workload": "smoke_256x1024", "numerics": {}}
    for g, gn in ((0, "e2m1"), (1, "e1m2"), (2, "e2m1c")):
        for rht in (False, True):
            r["numerics"]["%s_rht_%s" % (gn, "on" if rht else "off")] = stats_of(x, g, rht)
        qa, qb = U.ufp4_quantize(a, g), U.ufp4_quantize(b, g)
        c = torch.empty(256, 256, device=dev)
        ms = _ev_time(lambda: U.ufp4_gemm(qa, qb, out=c), flush)
        r["gemm_%s_tflops" % gn] = round(2 * 256 ** 3 / (ms * 1e-3) / 1e12, 3)
    for rht in (False, True):   # MXFP4: quantization numerics only (no GEMM)
        r["numerics"]["mxfp4_rht_%s" % ("on" if rht else "off")] = stats_of(x, U.UFP4_MXFP4, rht)
    emit(r)

    # outlier: 4096 x 4096, RHT on/off, both grids
    d = inputs.outlier(0)
    x = torch.from_numpy(d["x"]).to(torch.bfloat16).to(dev)
    r = {"workload": "outlier_4096x4096", "numerics": {}, "quantize_gbs": {}}
    for g, gn in ((0, "e2m1"), (1, "e1m2"), (2, "e2m1c"), (3, "mxfp4")):
        # MXFP4 moves 2 + 0.5 + 1/32 B/elem (one E8M0 byte per 32 elements)
        bpe = 2.53125 if g == U.UFP4_MXFP4 else Q_BYTES_PER_ELEM
        for rht in (False, True):
            key = "%s_rht_%s" % (gn, "on" if rht else "off")
            r["numerics"][key] = stats_of(x, g, rht)
            q = U.QTensor.empty(4096, 4096, g, dev)
            ms = _ev_time(lambda: U.ufp4_quantize(x, g, rht=rht, rht_seed=2, out=q), flush)
            r["quantize_gbs"][key] = round(x.numel() * bpe / (ms * 1e-3) / 1e9, 1)
    n = r["numerics"]
    r["sqnr_ranking"] = {
        "before_rht_e2m1_minus_e1m2_db": round(n["e2m1_rht_off"]["sqnr_db"] - n["e1m2_rht_off"]["sqnr_db"], 3),
        "after_rht_e2m1_minus_e1m2_db": round(n["e2m1_rht_on"]["sqnr_db"] - n["e1m2_rht_on"]["sqnr_db"], 3)}
    emit(r)

    # dense 1.5B training step: UFP4 on both grids, and the NVFP4 policy
    # (E2M1, the transform only on the bwd_dw operands) the pages compare with
    dd = inputs.device_dense(seed=0, device=dev)
    for g, gn, pol in ((1, "e1m2", "ufp4"), (0, "e2m1", "ufp4"), (0, "nvfp4_policy", "nvfp4")):
        st = Step(U, dd["x"], dd["w"], dd["dy"], g, policy=pol)
        mq = _ev_time(st.quantize_all, flush)
        mg = _ev_time(st.gemms, flush)
        emit({"workload": "dense1p5b_step_" + gn, "quantize_ms": round(mq, 4),
              "quantize_gbs": round(st.q_elems * Q_BYTES_PER_ELEM / (mq * 1e-3) / 1e9, 1),
              "gemm_ms": round(mg, 4), "gemm_tflops": round(sum(st.flops_each) / (mg * 1e-3) / 1e12, 1)})
    del dd

    # MoE 7.9B grouped step
    m = inputs.moe(seed=0)
    counts = [int(c) for c in m["counts"]]
    E, H, F = len(counts), 2048, 1408
    tx = torch.from_numpy(m["x"]).to(torch.bfloat16).to(dev)
    tw = torch.from_numpy(m["w"]).to(torch.bfloat16).to(dev)
    tdy = torch.from_numpy(m["dy"]).to(torch.bfloat16).to(dev)
    T = sum(counts)
    starts = np.concatenate([[0], np.cumsum(counts)])
    for g, gn in ((1, "e1m2"), (0, "e2m1")):
        kw = dict(rht=True, rht_seed=2)
        qs = {}

        def quant_all():
            qs["xr"] = U.ufp4_quantize_grouped(tx, g, counts, out=qs.get("xr"), **kw)
            qs["xc"] = U.ufp4_quantize_grouped(tx, g, counts, colwise=True, out=qs.get("xc"), **kw)
            qs["dr"] = U.ufp4_quantize_grouped(tdy, g, counts, round=1, sr_seed=3, out=qs.get("dr"), **kw)
            qs["dc"] = U.ufp4_quantize_grouped(tdy, g, counts, round=1, sr_seed=3, colwise=True,
                                               out=qs.get("dc"), **kw)
            qs["wr"] = U.ufp4_quantize_grouped(tw, g, [F] * E, out=qs.get("wr"), **kw)
            qs["wc"] = U.ufp4_quantize_grouped(tw, g, [F] * E, colwise=True, out=qs.get("wc"), **kw)
        quant_all()
        y = torch.empty(T, F, device=dev)
        dx = torch.empty(T, H, device=dev)
        dw = torch.empty(E * F, H, device=dev)
        xo, ko = U.grouped_offsets(counts, False), U.grouped_offsets(counts, True)
        wo, wk = U.grouped_offsets([F] * E, False), U.grouped_offsets([F] * E, True)
        gy = [dict(M=counts[e], N=F, K=H, a_row=xo[e], a_k=0, b_row=wo[e], b_k=0, a_seg=e, b_seg=e,
                   c=y[starts[e]:starts[e] + counts[e]] if counts[e] else y[:1]) for e in range(E)]
        gx = [dict(M=counts[e], N=H, K=F, a_row=xo[e], a_k=0, b_row=0, b_k=wk[e], a_seg=e, b_seg=e,
                   c=dx[starts[e]:starts[e] + counts[e]] if counts[e] else dx[:1]) for e in range(E)]
        gw = [dict(M=F, N=H, K=(counts[e] + 15) // 16 * 16, a_row=0, a_k=ko[e], b_row=0, b_k=ko[e],
                   a_seg=e, b_seg=e, c=dw[e * F:(e + 1) * F]) for e in range(E)]

        def gemm_all():
            U.ufp4_gemm_grouped(qs["xr"], qs["wr"], gy)
            U.ufp4_gemm_grouped(qs["dr"], qs["wc"], gx)
            U.ufp4_gemm_grouped(qs["dc"], qs["xc"], gw)
        mq = _ev_time(quant_all, flush, 5)
        mg = _ev_time(gemm_all, flush, 5)
        elems = 2 * (tx.numel() + tw.numel() + tdy.numel())
        flops = 3 * 2.0 * T * F * H
        emit({"workload": "moe7p9b_grouped_step_" + gn, "experts": E, "routed_tokens": T,
              "zero_token_experts": int(sum(1 for c in counts if c == 0)),
              "quantize_ms": round(mq, 4), "quantize_gbs": round(elems * Q_BYTES_PER_ELEM / (mq * 1e-3) / 1e9, 1),
              "gemm_ms": round(mg, 4), "gemm_tflops": round(flops / (mg * 1e-3) / 1e12, 1)})
    del tx, tw, tdy, m

    # MoE 124B large layer
    x = inputs.device_normal((65536, 8192), 1.0, 31, dev)
    w = inputs.device_normal((2048, 8192), 0.01, 32, dev)
    dy = inputs.device_normal((65536, 2048), 1e-3, 33, dev)
    for g, gn in ((1, "e1m2"), (0, "e2m1")):
        st = Step(U, x, w, dy, g)
        mq = _ev_time(st.quantize_all, flush, 3)
        mg = _ev_time(st.gemms, flush, 3)
        emit({"workload": "moe124b_layer_" + gn, "quantize_ms": round(mq, 4),
              "quantize_gbs": round(st.q_elems * Q_BYTES_PER_ELEM / (mq * 1e-3) / 1e9, 1),
              "gemm_ms": round(mg, 4), "gemm_tflops": round(sum(st.flops_each) / (mg * 1e-3) / 1e12, 1)})
        del st
    del x, w, dy
    torch.cuda.empty_cache()

    # compounding-attenuation chain: 100 x (4096^3), fresh W_k ~ N(0, 1/64)
    n, steps = 4096, 100
    rows = torch.arange(0, n, n // 64, device=dev)
    for g, gn in ((0, "e2m1"), (1, "e1m2"), (2, "e2m1c")):
        for rht in (False, True):
            X = inputs.device_normal((n, n), 1.0, 50, dev, dtype=torch.float32)
            norm0 = float(X.double().norm())
            ln_prod, sum_delta, ln_alpha = 0.0, 0.0, 0.0
            qx = U.QTensor.empty(n, n, g, dev)
            qw = U.QTensor.empty(n, n, g, dev)
            Y = torch.empty(n, n, device=dev)
            t_gpu = 0.0
            for k in range(steps):
                W = inputs.device_normal((n, n), 1.0 / 64, 1000 + k, dev)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                U.ufp4_quantize(X, g, rht=rht, rht_seed=2, out=qx)
                U.ufp4_quantize(W, g, rht=rht, rht_seed=2, out=qw)
                U.ufp4_gemm(qx, qw, out=Y)
                e1.record()
                torch.cuda.synchronize()
                t_gpu += e0.elapsed_time(e1)
                yref = X[rows].double() @ W.double().t()
                eta = float((Y[rows].double() * yref).sum() / (yref * yref).sum())
                ax = U.ufp4_stats(X, qx, rht=rht, rht_seed=2)["alpha"]
                aw = U.ufp4_stats(W, qw, rht=rht, rht_seed=2)["alpha"]
                ln_prod += float(np.log(eta))
                sum_delta += 1.0 - eta
                ln_alpha += float(np.log(ax * aw))
                X, Y = Y, X
            emit({"workload": "attenuation_chain_4096_x100_%s_rht_%s" % (gn, "on" if rht else "off"),
                  "prod_eta": round(float(np.exp(ln_prod)), 6), "exp_minus_sum_delta": round(float(np.exp(-sum_delta)), 6),
                  "prod_alpha_x_alpha_w": round(float(np.exp(ln_alpha)), 6),
                  "norm_ratio": round(float(X.double().norm()) / norm0, 6),
                  "gpu_ms_per_layer": round(t_gpu / steps, 4),
                  "layer_tflops": round(2.0 * n ** 3 / (t_gpu / steps * 1e-3) / 1e12, 1)})
    return out

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true", help="skip the secondary measurements")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workloads", action="store_true",
                    help="measure every synthetic workload (one JSON line each) instead of the step")
    ap.add_argument("--kernel", default=None,
                    choices=["gemm_e2m1", "gemm_e1m2", "quant_row_e1m2", "quant_col_e1m2", "quant_dual_e1m2",
                             "quant_dual_sr_e1m2",
                             "quant_row_e2m1", "quant_col_e2m1"],
                    help="time one kernel of the step in isolation (profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.kernel:
        run_kernel(args)
    elif args.workloads:
        run_workloads(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
