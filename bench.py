"""Benchmark of the UFP4 hot path on GB300.

Headline (the JSON line's value): one UFP4 training step of the MoE-124B-
shaped large layer -- X 65536 x 8192, W 2048 x 8192, dY 65536 x 2048, BF16,
seeded synthetic data -- six fused RHT + E1M2 quantizations (X, W, dY, each
row-wise and column-wise from one read per pass; stochastic rounding on dY
only) followed by the three training GEMMs fwd_y = X W^T, bwd_dx = dY W and
bwd_dw = dY^T X (K = 65536).

Reported (one JSON line from rank 0):
  value         fused RHT+quantize throughput, GB/s of algorithmic traffic
                (2 B read + 0.5625 B written per element and orientation)
                over the quantization launches of the step (the tensor-amax
                pass is in the time, not in the bytes);
  gemm          GEMM TFLOP/s (2 M N K logical flops) and fractions of the
                dense FP8 / FP4 peaks;
  roofline      the dominant kernel by time (the E1M2 GEMM);
  e2e           the same metric through the public API with the inputs
                copied from pinned host memory each step and the three GEMM
                outputs read back;
  cpu_baseline  the CPU oracle on a bounded sample of the same step;
  quantizer_x   the single- and dual-orientation quantizer on the layer's X
                with the transform on and off (the RHT overhead);
  workloads     every synthetic workload (smoke, outlier, dense-1.5B step,
                MoE-7.9B grouped step, MoE-124B layer and its compounding
                chain) with quantizer GB/s and GEMM TFLOP/s as fractions of
                their rooflines, the numerics the pages discuss, and the
                oracle timed beside each on a stated sample.
L2 is flushed before every timed step, outside the events: a 256 MiB buffer
is written and then read back, so the timed kernels start with an L2 that
holds none of their data and no dirty lines whose write-back would compete
with their reads.

--impl reference runs the CPU oracle (the paper released no code, so the
oracle is the reference arm) on a bounded sample of the same workload and
prints the same line shape.
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

WORKLOAD = dict(name="moe124b_layer_train_step", tokens=65536, hidden=8192, ffn=2048)
DENSE = dict(tokens=8192, hidden=2048, ffn=5632)
METRIC = ("fused RHT+quantize GB/s (% HBM peak); FP4 GEMM TFLOPS (% tensor peak)")
Q_BYTES_PER_ELEM = 2.0 + 0.5 + 1.0 / 16.0
MX_BYTES_PER_ELEM = 2.0 + 0.5 + 1.0 / 32.0     # one E8M0 byte per 32 elements
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


def moe124b_inputs(device, seed=0):
    """The MoE-124B large layer's operands, drawn on the device from seeded
    generators: X 65536 x 8192 N(0,1), W 2048 x 8192 N(0,0.01),
    dY 65536 x 2048 N(0,1e-3), all BF16."""
    from fp4_quantized_numerics_gb300 import inputs
    return dict(x=inputs.device_normal((65536, 8192), 1.0, 31 + 10 * seed, device),
                w=inputs.device_normal((2048, 8192), 0.01, 32 + 10 * seed, device),
                dy=inputs.device_normal((65536, 2048), 1e-3, 33 + 10 * seed, device))


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
        self.launches_per_step = self.count_launches(x.device) + 3
        self.q_elems = 2 * (x.numel() + w.numel() + dy.numel())
        self.flops_each = [2 * T * F * H, 2 * T * H * F, 2 * F * H * T]

    def count_launches(self, dev):
        """Kernels the quantize phase launches, by the library's routing: a
        dual-orientation BF16 call whose tensor fits on chip (at most 14
        128 x 64 tiles per SM) is one cooperative launch that takes its own
        maxima; any other quantization is an amax pass and a quantize pass."""
        import torch
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        n = 0
        for t in (self.x, self.w, self.dy):
            if self.grid == self.U.UFP4_MXFP4:   # no tensor amax: one pass per orientation
                n += 2
                continue
            rows, cols = t.shape
            tiles = -(-rows // 128) * -(-cols // 64)
            if self.dual and t.dtype == torch.bfloat16 and -(-tiles // min(sms, tiles)) <= 14:
                n += 1
            else:
                n += 2 * (1 if self.dual else 2)
        return n

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



def time_steps(step, steps, flush, stream=None):
    """Times `steps` steps on the current stream (L2 flushed before each,
    outside the events).  Returns per-step (quantize ms, [gemm ms x 3])."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    for i in range(steps):
        flush()
        e = evs[i]
        e[0].record()
        step.quantize_all()
        e[1].record()
        step.gemms(events=[None, e[2], e[3], e[4]])
    torch.cuda.synchronize()
    q_ms = [e[0].elapsed_time(e[1]) for e in evs]
    g_ms = [[e[1 + j].elapsed_time(e[2 + j]) for j in range(3)] for e in evs]
    return q_ms, g_ms


def run_gpu(args):
    import torch
    from fp4_quantized_numerics_gb300 import build, ufp4 as U

    ws_n, rank, local = dist_env()
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    build.build()
    U.lib()
    dev = torch.device("cuda", local)
    pk = peaks()

    d = moe124b_inputs(dev, seed=rank)
    step = Step(U, d["x"], d["w"], d["dy"], U.UFP4_E1M2)
    n_launch = step.launches_per_step   # kernels per step (quantize phase + 3 GEMMs)
    flush = L2Flush(dev)

    for _ in range(args.warmup):
        step.quantize_all()
        step.gemms()
    torch.cuda.synchronize()

    if ws_n > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        q_ms, g_ms = time_steps(step, args.steps, flush)
    if ws_n > 1:
        torch.distributed.barrier()
    tq, tg = sum(q_ms), sum(sum(g) for g in g_ms)
    tstep = tq + tg

    def allmax(v):
        return reduce_max(v, ws_n, dev)

    tq, tg, tstep = allmax(tq), allmax(tg), allmax(tstep)
    q_bytes = step.q_elems * Q_BYTES_PER_ELEM
    q_gbs = weak_scaling_rate(q_bytes, ws_n, args.steps, tq)
    flops = sum(step.flops_each)
    gemm_tflops = weak_scaling_rate(flops, ws_n, args.steps, tg, 1e12)
    per_gpu_tflops = gemm_tflops / ws_n
    fp8_sus = pk["bf16_tflops_sustained"] * 2.0   # nominal dense ratio fp8:bf16 = 4.5 : 2.25
    fp8_burst = pk["bf16_tflops"] * 2.0
    fp4_sus = pk["bf16_tflops_sustained"] * 6.0   # nominal dense ratio fp4:bf16 = 13.5 : 2.25
    gemm_each = [sum(g[j] for g in g_ms) / args.steps for j in range(3)]
    launch_ms = tg / (3 * args.steps)             # mean duration of one E1M2 GEMM launch
    flops_launch = step.flops_each[0]             # the three GEMMs have the same M N K
    assert all(f == flops_launch for f in step.flops_each)
    per_launch_tf = flops_launch / (launch_ms * 1e-3) / 1e12

    # ---------------------------------------------------- e2e through the API
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, U, step, d, dev, q_bytes)
        e2e["value"] = allmax(e2e["time_s"])
        e2e["value"] = ws_n * e2e["steps"] * q_bytes / e2e["value"] / 1e9
        del e2e["time_s"]

    extra = {}
    if not args.quick and rank == 0:
        extra["quantizer_x_65536x8192"] = quantizer_on_x(U, torch, dev, pk, flush, d["x"])
    del step, d
    torch.cuda.empty_cache()
    if not args.quick and rank == 0:
        extra["workloads"] = all_workloads(U, torch, dev, pk, flush, with_oracle=not args.no_cpu_baseline)
    if ws_n > 1:
        torch.distributed.barrier()

    if rank == 0:
        clocks = clk.summary()
        line = {
            "metric": METRIC, "value": round(q_gbs, 2), "unit": "GB/s",
            "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tstep / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp32 quantize / e2m1-plane MMA, f32 accumulate",
            "data": "synthetic (seeded N(0,1) / N(0,0.01) / N(0,1e-3) BF16, drawn on the device)",
            "config": {"workload": WORKLOAD["name"], "X": [WORKLOAD["tokens"], WORKLOAD["hidden"]],
                       "W": [WORKLOAD["ffn"], WORKLOAD["hidden"]],
                       "dY": [WORKLOAD["tokens"], WORKLOAD["ffn"]],
                       "recipe": "UFP4: E1M2, RHT16 on all GEMM operands, SR on dY, both orientations per read",
                       "l2": "flushed before every timed step (256 MiB write, then read back)",
                       "parallelism": "replicas" if ws_n > 1 else "single"},
            "quantize": {"gbs": round(q_gbs, 1), "frac_hbm": round(q_gbs / ws_n / pk["hbm_gbs"], 4),
                         "ms_per_step": round(tq / args.steps, 4),
                         "elements_per_step": step_elems(WORKLOAD),
                         "elements_per_s": round(ws_n * step_elems(WORKLOAD) / (tq / args.steps * 1e-3)),
                         "launches_per_step": n_launch - 3},
            "gemm": {"tflops": round(gemm_tflops, 1), "ms_per_step": round(tg / args.steps, 4),
                     "ms_each": [round(v, 4) for v in gemm_each],
                     "frac_fp8_peak_sustained": round(per_gpu_tflops / fp8_sus, 4),
                     "frac_fp8_peak_burst": round(per_gpu_tflops / fp8_burst, 4),
                     "frac_fp4_peak_sustained": round(per_gpu_tflops / fp4_sus, 4)},
            "roofline": {"bound": "tensor", "kernel": "k_gemm<E1M2, E planes loaded>",
                         "achieved": round(per_launch_tf, 1), "peak": round(fp8_sus, 1),
                         "unit": "TFLOP/s", "frac": round(per_launch_tf / fp8_sus, 4),
                         "frac_of_burst_peak": round(per_launch_tf / fp8_burst, 4),
                         "flops_per_launch": flops_launch,
                         "mean_launch_ms": round(launch_ms, 4),
                         "traffic": traffic_for("k_gemm_e1m2_moe124b"),
                         "peak_kind": "dense FP8 = %s sustained bf16 x 2 (timed inside a seconds-long loop of "
                                      "steps)" % pk["source"]},
            "gpu_launches": n_launch * args.steps,
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


def step_elems(wl):
    T, H, F = wl["tokens"], wl["hidden"], wl["ffn"]
    return 2 * (T * H + F * H + T * F)


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


def _timeit(torch, fn, flush, n=20):
    """Median of n timed runs (each after an L2 flush), after 3 untimed."""
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


def quantizer_on_x(U, torch, dev, pk, flush, x):
    """The fused quantizer on the MoE-124B layer's X (65536 x 8192 BF16,
    1 GiB), E1M2 RTNE: one orientation with the tensor amax given, transform
    on and off (the RHT overhead), with the amax pass, with the correction
    plane written; and both orientations from one read."""
    R, C = x.shape
    el = x.numel()
    q = U.QTensor.empty(R, C, U.UFP4_E1M2, dev, eplane=False)
    qc = U.QTensor.empty(C, R, U.UFP4_E1M2, dev, eplane=False)
    am = (x.abs().max().float() * 1.25).reshape(1)   # a valid amax, above the rotated maximum
    ws = U.workspace(dev)
    gbs = lambda ms, n=1: round(n * el * Q_BYTES_PER_ELEM / (ms * 1e-3) / 1e9, 1)
    r = {}
    r["single_amax_given_rht_on"] = gbs(_timeit(torch, lambda: U.ufp4_quantize(
        x, U.UFP4_E1M2, rht=True, out=q, ws=ws, amax_in=am), flush))
    r["single_amax_given_rht_off"] = gbs(_timeit(torch, lambda: U.ufp4_quantize(
        x, U.UFP4_E1M2, rht=False, out=q, ws=ws, amax_in=am), flush))
    r["rht_overhead_amax_given"] = round(r["single_amax_given_rht_off"] / r["single_amax_given_rht_on"] - 1, 4)
    r["frac_hbm_single_amax_given_rht_on"] = round(r["single_amax_given_rht_on"] / pk["hbm_gbs"], 4)
    r["single_with_amax_pass_rht_on"] = gbs(_timeit(torch, lambda: U.ufp4_quantize(
        x, U.UFP4_E1M2, rht=True, out=q, ws=ws), flush))
    r["single_amax_given_rht_off_colwise"] = gbs(_timeit(torch, lambda: U.ufp4_quantize(
        x, U.UFP4_E1M2, rht=False, colwise=True, out=qc, ws=ws, amax_in=am), flush))
    r["single_amax_given_rht_on_colwise"] = gbs(_timeit(torch, lambda: U.ufp4_quantize(
        x, U.UFP4_E1M2, rht=True, colwise=True, out=qc, ws=ws, amax_in=am), flush))
    r["dual_amax_given_rht_on"] = gbs(_timeit(torch, lambda: U.ufp4_quantize_dual(
        x, U.UFP4_E1M2, rht=True, amax_row=am, amax_col=am, out_row=q, out_col=qc, ws=ws), flush), 2)
    r["dual_amax_given_rht_off"] = gbs(_timeit(torch, lambda: U.ufp4_quantize_dual(
        x, U.UFP4_E1M2, rht=False, amax_row=am, amax_col=am, out_row=q, out_col=qc, ws=ws), flush), 2)
    r["dual_with_amax_pass_rht_on"] = gbs(_timeit(torch, lambda: U.ufp4_quantize_dual(
        x, U.UFP4_E1M2, rht=True, out_row=q, out_col=qc, ws=ws), flush), 2)
    del q, qc
    qe = U.QTensor.empty(R, C, U.UFP4_E1M2, dev)
    r["single_amax_given_rht_on_with_eplane"] = gbs(_timeit(torch, lambda: U.ufp4_quantize(
        x, U.UFP4_E1M2, rht=True, out=qe, ws=ws, amax_in=am), flush))
    r["elems_per_s_single_amax_given_rht_on"] = round(r["single_amax_given_rht_on"] * 1e9 / Q_BYTES_PER_ELEM)
    r["elems_per_s_single_with_amax_pass_rht_on"] = round(r["single_with_amax_pass_rht_on"] * 1e9 /
                                                          Q_BYTES_PER_ELEM)
    r["note"] = ("GB/s of algorithmic traffic (2.5625 B per element and result; elements/s = GB/s / 2.5625); "
                 "the amax pass's second read and the correction plane's writes are not counted")
    return r


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
def _oracle_quant_rate(fn, elems):
    t0 = time.perf_counter()
    fn()
    dt = time.perf_counter() - t0
    return elems * Q_BYTES_PER_ELEM / dt / 1e9, dt


def _oracle_gemm_rate(a, b):
    from oracle import oracle
    t0 = time.perf_counter()
    oracle.gemm_f64(a, b)
    dt = time.perf_counter() - t0
    return 2.0 * a.shape[0] * b.shape[0] * a.shape[1] / dt / 1e9, dt


def cpu_sample(rows_x=8192, rows_dy=16384, gemm_rows=16, seed=0):
    """The oracle on a bounded sample of the MoE-124B step: RHT + E1M2
    row-wise quantization of rows_x rows of X (65536 x 8192 in full) and of
    rows_dy rows of dY (SR), and gemm_rows rows of fwd_y in fp64 against the
    whole quantized W.  Returns (quantize GB/s, GEMM GFLOP/s, seconds, desc,
    extrapolated seconds of the full step)."""
    from fp4_quantized_numerics_gb300 import inputs
    from oracle import oracle
    T, H, F = WORKLOAD["tokens"], WORKLOAD["hidden"], WORKLOAD["ffn"]
    g = inputs.rng(seed)
    x = inputs.to_bf16_f32(g.standard_normal((rows_x, H), dtype=np.float32))
    dy = inputs.to_bf16_f32(g.standard_normal((rows_dy, F), dtype=np.float32) * np.float32(1e-3))
    w = inputs.to_bf16_f32(g.standard_normal((F, H), dtype=np.float32) * np.float32(0.01))
    t0 = time.perf_counter()
    rx = oracle.quantize(x, oracle.E1M2, rht=True, rht_seed=2)
    oracle.quantize(dy, oracle.E1M2, rht=True, rht_seed=2, round_mode=oracle.SR, sr_seed=3)
    tq = time.perf_counter() - t0
    rw = oracle.quantize(w, oracle.E1M2, rht=True, rht_seed=2)
    A = oracle.dequantize(rx["codes"][:gemm_rows], rx["scales"][:gemm_rows], rx["tensor_scale"], oracle.E1M2)
    B = oracle.dequantize(rw["codes"], rw["scales"], rw["tensor_scale"], oracle.E1M2)
    gflops, tg = _oracle_gemm_rate(A, B)
    el = x.size + dy.size
    qgbs = el * Q_BYTES_PER_ELEM / tq / 1e9
    full = step_elems(WORKLOAD) * Q_BYTES_PER_ELEM / (qgbs * 1e9) + 3 * 2.0 * T * H * F / (gflops * 1e9)
    desc = ("RHT+E1M2 row-wise quantization of %d x %d of X and %d x %d of dY (SR), "
            "plus %d rows of fwd_y in fp64 (K = %d)" % (rows_x, H, rows_dy, F, gemm_rows, H))
    return qgbs, gflops, tq + tg, desc, full


def cpu_baseline(args):
    gbs, gflops, secs, desc, full = cpu_sample()
    return {"value": round(gbs, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": desc, "gemm_gflops": round(gflops, 3), "seconds": round(secs, 2),
            "full_step_seconds_extrapolated": round(full, 1), "host": host_desc()}


def host_desc():
    try:
        import platform
        model = ""
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
            for l in out.splitlines():
                if l.startswith("Model name"):
                    model = l.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
        return "%s %s, %d logical cores (the oracle uses 1)" % (platform.machine(), model, os.cpu_count() or 0)
    except Exception:
        return None


def run_reference(args):
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return
    t_all = 0.0
    vals = []
    for i in range(args.warmup + args.steps):
        gbs, gflops, secs, desc, _ = cpu_sample(rows_x=256, rows_dy=512, gemm_rows=4, seed=i)
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
                             "sample": desc, "host": host_desc()},
            "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_kernel(args):
    """One kernel of a step in isolation, for profiling: `steps` launches of
    the fwd_y GEMM (T x F x H; gemm_e1m2_dx / _dw: the bwd_dx and bwd_dw
    products of the same layer), of the RHT quantization of X (T x H) in one
    orientation or both (quant_dual_*; the SR variant quantizes dY, T x F),
    after `warmup` launches, the tensor amax given (quant_resident_e1m2: W,
    F x H, both ways with its maxima, the on-chip single pass; quant_grouped_dual_e1m2:
    the MoE-7.9B X both ways, its amax pass included).  --shape dense: T, H,
    F = 8192, 2048, 5632; moe124b: 65536, 8192, 2048.  Prints the mean event
    time."""
    import torch
    from fp4_quantized_numerics_gb300 import build, inputs, ufp4 as U
    build.build()
    dev = torch.device("cuda", 0)
    kind = args.kernel
    if kind == "quant_grouped_dual_e1m2":
        # the MoE-7.9B layer's X (64 experts, 16384 tokens x top-6, Dirichlet
        # routing) in both orientations, amax pass included; --shape unused
        counts = [int(c) for c in inputs.moe_counts(0)]
        x = inputs.device_normal((sum(counts), 2048), 1.0, 21, dev)
        qr = U.QTensor.empty(U.grouped_rows(counts), 2048, U.UFP4_E1M2, dev)
        qc = U.QTensor.empty(2048, U.grouped_kpad(counts), U.UFP4_E1M2, dev)
        qr.tensor_scale = torch.empty(len(counts), device=dev)
        qc.tensor_scale = torch.empty(len(counts), device=dev)
        fn = lambda: U.ufp4_quantize_grouped_dual(x, U.UFP4_E1M2, counts, rht=True, out_row=qr, out_col=qc)
        work = 2 * x.numel() * Q_BYTES_PER_ELEM
        unit = "GB/s"
        return _run_kernel_timing(args, kind, fn, work, unit, dev)
    wl = WORKLOAD if args.shape == "moe124b" else DENSE
    T, H, F = wl["tokens"], wl["hidden"], wl["ffn"]
    x = inputs.device_normal((T, H), 1.0, 21, dev)
    if kind.startswith("gemm"):
        grid = {"gemm_e2m1": U.UFP4_E2M1, "gemm_mxfp4": U.UFP4_MXFP4}.get(kind, U.UFP4_E1M2)
        if kind == "gemm_e1m2_dx":     # dX = dY W: M = T, N = H, K = F
            a_src = inputs.device_normal((T, F), 1e-3, 23, dev)
            b_src = inputs.device_normal((H, F), 0.02, 22, dev)
        elif kind == "gemm_e1m2_dw":   # dW = dY^T X: M = F, N = H, K = T
            a_src = inputs.device_normal((F, T), 1e-3, 23, dev)
            b_src = inputs.device_normal((H, T), 1.0, 21, dev)
        else:                          # Y = X W^T: M = T, N = F, K = H
            a_src, b_src = x, inputs.device_normal((F, H), 0.02, 22, dev)
        a, b = U.ufp4_quantize(a_src, grid, rht=True), U.ufp4_quantize(b_src, grid, rht=True)
        del a_src, b_src
        c = torch.empty(a.rows, b.rows, dtype=torch.float32, device=dev)
        fn = lambda: U.ufp4_gemm(a, b, out=c)
        work = 2.0 * T * F * H
        unit = "TFLOP/s"
    elif kind == "quant_resident_e1m2":
        # W (F x H) both ways with both tensor maxima computed: a tensor that
        # fits on chip takes the single pass (one cooperative launch)
        src = inputs.device_normal((F, H), 0.02, 22, dev)
        qr = U.QTensor.empty(F, H, U.UFP4_E1M2, dev)
        qc = U.QTensor.empty(H, F, U.UFP4_E1M2, dev)
        fn = lambda: U.ufp4_quantize_dual(src, U.UFP4_E1M2, rht=True, out_row=qr, out_col=qc)
        work = 2 * src.numel() * Q_BYTES_PER_ELEM
        unit = "GB/s"
    elif kind.startswith("quant_dual") or kind == "amax_dual_e1m2":
        # both orientations from one read; SR variant on the dY shape; the
        # amax variant computes the tensor maxima (its amax pass is profiled)
        grid = U.UFP4_E1M2
        sr = kind.startswith("quant_dual_sr")
        src = inputs.device_normal((T, F), 1e-3, 23, dev) if sr else x
        am = None if kind == "amax_dual_e1m2" else (src.abs().max().float() * 1.5).reshape(1)
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
        am = (x.abs().max().float() * 1.5).reshape(1)
        fn = lambda: U.ufp4_quantize(x, grid, rht=True, colwise=col, out=q, amax_in=am)
        work = x.numel() * Q_BYTES_PER_ELEM
        unit = "GB/s"
    return _run_kernel_timing(args, kind, fn, work, unit, dev)


def _run_kernel_timing(args, kind, fn, work, unit, dev):
    import torch
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



def run_all_kernels(args):
    """Every public call of the library once per timing, on the dense-1.5B
    shapes (X 8192 x 2048, W 5632 x 2048, dY 8192 x 5632) and the MoE-7.9B
    grouped X: medians of `steps` event-timed runs (L2 flushed, after 3
    untimed) with each call's algorithmic bytes or FLOPs, so that an ncu
    launch list of this command covers every kernel.  Prints one JSON line."""
    import torch
    from fp4_quantized_numerics_gb300 import build, inputs, ufp4 as U
    build.build()
    dev = torch.device("cuda", 0)
    flush = L2Flush(dev)
    T, H, F = DENSE["tokens"], DENSE["hidden"], DENSE["ffn"]
    x = inputs.device_normal((T, H), 1.0, 31, dev)
    w = inputs.device_normal((F, H), 0.02, 32, dev)
    dy = inputs.device_normal((T, F), 1e-3, 33, dev)
    x32 = x.float()
    E1, E2, MX = U.UFP4_E1M2, U.UFP4_E2M1, U.UFP4_MXFP4
    qx, qw = U.ufp4_quantize(x, E1, rht=True), U.ufp4_quantize(w, E1, rht=True)
    qx2, qw2 = U.ufp4_quantize(x, E2, rht=True), U.ufp4_quantize(w, E2, rht=True)
    qxn = U.QTensor.empty(T, H, E1, dev, eplane=False)
    U.ufp4_quantize(x, E1, rht=True, out=qxn)
    qwn = U.QTensor.empty(F, H, E1, dev, eplane=False)
    U.ufp4_quantize(w, E1, rht=True, out=qwn)
    qxm, qwm = U.ufp4_quantize(x, MX), U.ufp4_quantize(w, MX)
    c = torch.empty(T, F, dtype=torch.float32, device=dev)
    deq = torch.empty(T, H, dtype=torch.float32, device=dev)
    counts = [int(v) for v in inputs.moe_counts(0)]
    xg = inputs.device_normal((sum(counts), H), 1.0, 34, dev)
    gr, gc = U.ufp4_quantize_grouped_dual(xg, E1, counts, rht=True)
    wg = inputs.device_normal((len(counts) * 1408, H), 0.02, 35, dev)
    gw = U.ufp4_quantize_grouped(wg, E1, [1408] * len(counts), rht=True)
    yg = torch.empty(sum(counts), 1408, dtype=torch.float32, device=dev)
    xo, wo = U.grouped_offsets(counts, False), U.grouped_offsets([1408] * len(counts), False)
    starts = np.concatenate([[0], np.cumsum(counts)])
    groups = [dict(M=counts[e], N=1408, K=H, a_row=xo[e], a_k=0, b_row=wo[e], b_k=0, a_seg=e, b_seg=e,
                   c=yg[starts[e]:starts[e] + counts[e]] if counts[e] else yg[:1]) for e in range(len(counts))]
    qb, gb = Q_BYTES_PER_ELEM, 2.0 * T * F * H
    nx, ng = x.numel(), xg.numel()
    calls = [
        ("quantize row E1M2 RHT (amax pass + pass)", lambda: U.ufp4_quantize(x, E1, rht=True, out=qx), nx * qb, "B"),
        ("quantize col E1M2 RHT", lambda: U.ufp4_quantize(x, E1, rht=True, colwise=True), nx * qb, "B"),
        ("quantize row E2M1 RHT", lambda: U.ufp4_quantize(x, E2, rht=True, out=qx2), nx * qb, "B"),
        ("quantize row E1M2 SR (dY)", lambda: U.ufp4_quantize(dy, E1, rht=True, round=U.UFP4_SR, sr_seed=3),
         dy.numel() * qb, "B"),
        ("quantize row E1M2 RHT, FP32 input", lambda: U.ufp4_quantize(x32, E1, rht=True), nx * 4.5625, "B"),
        ("quantize dual E1M2 RHT X (on-chip single pass)", lambda: U.ufp4_quantize_dual(x, E1, rht=True),
         2 * nx * qb, "B"),
        ("quantize dual E1M2 RHT SR dY (two passes)",
         lambda: U.ufp4_quantize_dual(dy, E1, rht=True, round=U.UFP4_SR, sr_seed=3), 2 * dy.numel() * qb, "B"),
        ("quantize MXFP4 row", lambda: U.ufp4_quantize(x, MX), nx * MX_BYTES_PER_ELEM, "B"),
        ("quantize MXFP4 col", lambda: U.ufp4_quantize(x, MX, colwise=True), nx * MX_BYTES_PER_ELEM, "B"),
        ("dequantize E1M2 + inverse RHT", lambda: U.ufp4_dequantize(qx, inverse_rht=True, out=deq),
         nx * (0.5625 + 4), "B"),
        ("stats E1M2 RHT", lambda: U.ufp4_stats(x, qx, rht=True), nx * (2 + 0.5625), "B"),
        ("quantize + stats E1M2 RHT (one read)", lambda: U.ufp4_quantize_stats(x, E1, rht=True), nx * qb, "B"),
        ("quantize grouped row E1M2 RHT (MoE-7.9B X)", lambda: U.ufp4_quantize_grouped(xg, E1, counts, rht=True),
         ng * qb, "B"),
        ("quantize grouped col E1M2 RHT", lambda: U.ufp4_quantize_grouped(xg, E1, counts, rht=True, colwise=True),
         ng * qb, "B"),
        ("quantize grouped dual E1M2 RHT",
         lambda: U.ufp4_quantize_grouped_dual(xg, E1, counts, rht=True, out_row=gr, out_col=gc), 2 * ng * qb, "B"),
        ("GEMM E1M2 planes loaded, fwd_y", lambda: U.ufp4_gemm(qx, qw, out=c), gb, "F"),
        ("GEMM E1M2 planes expanded on chip", lambda: U.ufp4_gemm(qxn, qwn, out=c), gb, "F"),
        ("GEMM E2M1", lambda: U.ufp4_gemm(qx2, qw2, out=c), gb, "F"),
        ("GEMM MXFP4", lambda: U.ufp4_gemm(qxm, qwm, out=c), gb, "F"),
        ("GEMM E1M2 + output amax", lambda: U.ufp4_gemm_amax(qx, qw, out=c), gb, "F"),
        ("grouped GEMM E1M2 fwd_y (MoE-7.9B)", lambda: U.ufp4_gemm_grouped(gr, gw, groups),
         2.0 * sum(counts) * 1408 * H, "F"),
    ]
    out = []
    for name, fn, work, kind in calls:
        ms = _timeit(torch, fn, flush, max(args.steps, 1))
        rate = work / (ms * 1e-3) / (1e12 if kind == "F" else 1e9)
        out.append({"call": name, "ms": round(ms, 4), "rate": round(rate, 1),
                    "unit": "TFLOP/s" if kind == "F" else "GB/s"})
    print(json.dumps({"kernel": "all", "calls": out}))


# ------------------------------------------------------------ all workloads
def _ev_time(fn, flush, reps=20):
    import torch
    return _timeit(torch, fn, flush, reps)


def _fracs(pk, q_gbs=None, tflops=None, grid=None, gemm_bytes=None, gemm_flops=None):
    """Roofline fractions: the quantizer against HBM, a GEMM against the
    dense tensor peak of its grid's MMA (E1M2: FP8, as the recipe's target
    states; E2M1: FP4) and, for E2M1, against max(flop time, byte time)."""
    out = {}
    if q_gbs is not None:
        out["quantize_frac_hbm"] = round(q_gbs / pk["hbm_gbs"], 4)
    if tflops is not None:
        fp8, fp4 = 2.0 * pk["bf16_tflops"], 6.0 * pk["bf16_tflops"]
        if grid == 1:
            out["gemm_frac_fp8_dense"] = round(tflops / fp8, 4)
        else:
            out["gemm_frac_fp4_dense"] = round(tflops / fp4, 4)
            if gemm_bytes and gemm_flops:
                # the fastest the GEMM could run: tensor time or HBM time, whichever is longer
                t_min = max(gemm_flops / (fp4 * 1e12), gemm_bytes / (pk["hbm_gbs"] * 1e9))
                t_run = gemm_flops / (tflops * 1e12)
                out["gemm_combined_roofline_tflops"] = round(gemm_flops / t_min / 1e12, 1)
                out["gemm_frac_combined_roofline"] = round(t_min / t_run, 4)
    return out


def _gemm_bytes(M, N, K, mx=False):
    """Algorithmic bytes of one GEMM: both quantized operands (0.5 B codes +
    1/16 B scale per element; MXFP4 1/32 B) and the fp32 output."""
    return (M + N) * K * (0.53125 if mx else 0.5625) + 4.0 * M * N


def all_workloads(U, torch, dev, pk, flush, with_oracle=True):
    """Every synthetic workload at 1 GPU: quantizer GB/s and GEMM TFLOP/s
    with their roofline fractions, the numerics the pages discuss (alpha,
    SQNR, mean bias, prod eta), and the CPU oracle timed beside each on the
    stated sample (1 core; full-workload time extrapolated from the sample's
    rate)."""
    from fp4_quantized_numerics_gb300 import inputs
    out = {}
    o = None
    if with_oracle:
        from oracle import oracle as o

    def oracle_q(x, elems_full, desc, **kw):
        if o is None:
            return None
        gbs, dt = _oracle_quant_rate(lambda: o.quantize(x, **kw), x.size)
        return {"quantize_gbs": round(gbs, 5), "seconds": round(dt, 2), "cores": 1, "sample": desc,
                "full_quantize_seconds_extrapolated": round(elems_full * Q_BYTES_PER_ELEM / (gbs * 1e9), 1)}

    def stats_of(x, grid, rht):
        q = U.ufp4_quantize(x, grid, rht=rht, rht_seed=2)
        st = U.ufp4_stats(x, q, rht=rht, rht_seed=2)
        return {k: round(st[k], 6) for k in ("alpha", "sqnr_db", "mean_bias")}

    # ---- smoke: 256 x 1024 tensor, 256^3 GEMM (launch-bound; reported)
    d = inputs.smoke(0)
    x = torch.from_numpy(d["x"]).to(torch.bfloat16).to(dev)
    a = torch.from_numpy(d["a"]).to(torch.bfloat16).to(dev)
    b = torch.from_numpy(d["b"]).to(torch.bfloat16).to(dev)
    r = {"config": "BF16 256 x 1024 N(0,1); GEMM 256^3", "numerics": {}}
    q = U.QTensor.empty(256, 1024, U.UFP4_E1M2, dev)
    ms = _ev_time(lambda: U.ufp4_quantize(x, U.UFP4_E1M2, rht=True, rht_seed=2, out=q), flush)
    r["quantize_e1m2_rht_gbs"] = round(x.numel() * Q_BYTES_PER_ELEM / (ms * 1e-3) / 1e9, 2)
    r["quantize_e1m2_rht_elems_per_s"] = round(x.numel() / (ms * 1e-3))
    r.update(_fracs(pk, q_gbs=r["quantize_e1m2_rht_gbs"]))
    for g, gn in ((0, "e2m1"), (1, "e1m2"), (2, "e2m1c"), (3, "mxfp4")):
        for rht in (False, True):
            r["numerics"]["%s_rht_%s" % (gn, "on" if rht else "off")] = stats_of(x, g, rht)
        qa, qb = U.ufp4_quantize(a, g), U.ufp4_quantize(b, g)
        c = torch.empty(256, 256, device=dev)
        ms = _ev_time(lambda: U.ufp4_gemm(qa, qb, out=c), flush)
        r["gemm_%s_tflops" % gn] = round(2 * 256 ** 3 / (ms * 1e-3) / 1e12, 3)
    r["note"] = "0.67 MB of input: launch latency, not HBM, bounds it"
    if o is not None:
        r["oracle"] = oracle_q(d["x"], d["x"].size, "the whole 256 x 1024 tensor, RHT + E1M2",
                               grid=1, rht=True, rht_seed=2)
        qa, qb = o.quantize(d["a"], 1), o.quantize(d["b"], 1)
        gf, dt = _oracle_gemm_rate(o.dequantize(qa["codes"], qa["scales"], qa["tensor_scale"], 1),
                                   o.dequantize(qb["codes"], qb["scales"], qb["tensor_scale"], 1))
        r["oracle"]["gemm_gflops"] = round(gf, 3)
    out["smoke_256x1024"] = r

    # ---- outlier: 4096 x 4096, RHT on/off, every grid
    d = inputs.outlier(0)
    x = torch.from_numpy(d["x"]).to(torch.bfloat16).to(dev)
    r = {"config": "BF16 4096 x 4096 N(0,1) + column offsets N(0,0.5), 4 columns x100", "numerics": {},
         "quantize_gbs": {}, "quantize_elems_per_s": {}}
    for g, gn in ((0, "e2m1"), (1, "e1m2"), (2, "e2m1c"), (3, "mxfp4")):
        bpe = MX_BYTES_PER_ELEM if g == U.UFP4_MXFP4 else Q_BYTES_PER_ELEM
        for rht in (False, True):
            key = "%s_rht_%s" % (gn, "on" if rht else "off")
            r["numerics"][key] = stats_of(x, g, rht)
            qq = U.QTensor.empty(4096, 4096, g, dev, eplane=False)
            ms = _ev_time(lambda: U.ufp4_quantize(x, g, rht=rht, rht_seed=2, out=qq), flush)
            r["quantize_gbs"][key] = round(x.numel() * bpe / (ms * 1e-3) / 1e9, 1)
            r["quantize_elems_per_s"][key] = round(x.numel() / (ms * 1e-3))
    r["quantize_frac_hbm"] = {k: round(v / pk["hbm_gbs"], 4) for k, v in r["quantize_gbs"].items()}
    n = r["numerics"]
    r["sqnr_ranking"] = {
        "before_rht_e2m1_minus_e1m2_db": round(n["e2m1_rht_off"]["sqnr_db"] - n["e1m2_rht_off"]["sqnr_db"], 3),
        "after_rht_e2m1_minus_e1m2_db": round(n["e2m1_rht_on"]["sqnr_db"] - n["e1m2_rht_on"]["sqnr_db"], 3)}
    r["note"] = "43 MB of input (amax pass + quantization pass per call): the whole call's time"
    if o is not None:
        r["oracle"] = oracle_q(d["x"][:512], d["x"].size, "512 of the 4096 rows, RHT + E1M2",
                               grid=1, rht=True, rht_seed=2)
    out["outlier_4096x4096"] = r

    # ---- dense 1.5B training step: UFP4 on both grids, and the NVFP4 policy
    T, H, F = DENSE["tokens"], DENSE["hidden"], DENSE["ffn"]
    dd = inputs.device_dense(seed=0, device=dev)
    r = {"config": "X 8192 x 2048 (1 column x50), W 5632 x 2048, dY 8192 x 5632; 3 GEMMs of 189 GFLOP"}
    for g, gn, pol in ((1, "e1m2", "ufp4"), (0, "e2m1", "ufp4"), (0, "nvfp4_policy", "nvfp4"),
                       (3, "mxfp4", "ufp4")):
        # MXFP4 has no two-orientation pass: six single-orientation passes
        st = Step(U, dd["x"], dd["w"], dd["dy"], g, policy=pol, dual=g != U.UFP4_MXFP4)
        mq = _ev_time(st.quantize_all, flush)
        mg = _ev_time(st.gemms, flush)
        bpe = MX_BYTES_PER_ELEM if g == U.UFP4_MXFP4 else Q_BYTES_PER_ELEM
        qg = st.q_elems * bpe / (mq * 1e-3) / 1e9
        tf = sum(st.flops_each) / (mg * 1e-3) / 1e12
        e = {"quantize_ms": round(mq, 4), "quantize_gbs": round(qg, 1),
             "quantize_elems_per_s": round(st.q_elems / (mq * 1e-3)), "gemm_ms": round(mg, 4),
             "gemm_tflops": round(tf, 1)}
        e.update(_fracs(pk, qg, tf, g, 3 * _gemm_bytes(T, F, H, mx=g == U.UFP4_MXFP4), sum(st.flops_each)))
        r[gn] = e
        del st
    del dd
    if o is not None:
        g = inputs.rng(0)
        xs = inputs.to_bf16_f32(g.standard_normal((1024, H), dtype=np.float32))
        dys = inputs.to_bf16_f32(g.standard_normal((1024, F), dtype=np.float32) * np.float32(1e-3))
        full = 2 * (T * H + F * H + T * F)
        r["oracle"] = oracle_q(xs, full, "1024 rows of X, RHT + E1M2 (and the GEMM: 8 rows of fwd_y)",
                               grid=1, rht=True, rht_seed=2)
        ws_ = inputs.to_bf16_f32(g.standard_normal((F, H), dtype=np.float32) * np.float32(0.02))
        qa, qb = o.quantize(xs[:8], 1, rht=True, rht_seed=2), o.quantize(ws_, 1, rht=True, rht_seed=2)
        gf, _ = _oracle_gemm_rate(o.dequantize(qa["codes"], qa["scales"], qa["tensor_scale"], 1),
                                  o.dequantize(qb["codes"], qb["scales"], qb["tensor_scale"], 1))
        r["oracle"]["gemm_gflops"] = round(gf, 3)
        r["oracle"]["full_gemm_seconds_extrapolated"] = round(3 * 2.0 * T * H * F / (gf * 1e9), 1)
        del dys
    out["dense1p5b_step"] = r

    # ---- MoE 7.9B grouped step
    m = inputs.moe(seed=0)
    counts = [int(c) for c in m["counts"]]
    E, H, F = len(counts), 2048, 1408
    tx = torch.from_numpy(m["x"]).to(torch.bfloat16).to(dev)
    tw = torch.from_numpy(m["w"]).to(torch.bfloat16).to(dev)
    tdy = torch.from_numpy(m["dy"]).to(torch.bfloat16).to(dev)
    T = sum(counts)
    starts = np.concatenate([[0], np.cumsum(counts)])
    r = {"config": "64 experts, 16384 tokens x top-6 = %d routed rows (Dirichlet(1) routing, %d empty experts); "
                   "per expert X_e [T_e x 2048], W_e [1408 x 2048], dY_e [T_e x 1408]"
                   % (T, sum(1 for c in counts if c == 0))}
    for g, gn in ((1, "e1m2"), (0, "e2m1")):
        kw = dict(rht=True, rht_seed=2)
        qs = {}

        def quant_all():
            # every operand in both orientations from one read per pass
            qs["xr"], qs["xc"] = U.ufp4_quantize_grouped_dual(tx, g, counts, out_row=qs.get("xr"),
                                                              out_col=qs.get("xc"), **kw)
            qs["dr"], qs["dc"] = U.ufp4_quantize_grouped_dual(tdy, g, counts, round=1, sr_seed=3,
                                                              out_row=qs.get("dr"), out_col=qs.get("dc"), **kw)
            qs["wr"], qs["wc"] = U.ufp4_quantize_grouped_dual(tw, g, [F] * E, out_row=qs.get("wr"),
                                                              out_col=qs.get("wc"), **kw)

        def quant_all_single():
            U.ufp4_quantize_grouped(tx, g, counts, out=qs["xr"], **kw)
            U.ufp4_quantize_grouped(tx, g, counts, colwise=True, out=qs["xc"], **kw)
            U.ufp4_quantize_grouped(tdy, g, counts, round=1, sr_seed=3, out=qs["dr"], **kw)
            U.ufp4_quantize_grouped(tdy, g, counts, round=1, sr_seed=3, colwise=True, out=qs["dc"], **kw)
            U.ufp4_quantize_grouped(tw, g, [F] * E, out=qs["wr"], **kw)
            U.ufp4_quantize_grouped(tw, g, [F] * E, colwise=True, out=qs["wc"], **kw)
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
        mq = _ev_time(quant_all, flush)
        mq1 = _ev_time(quant_all_single, flush)
        mg = _ev_time(gemm_all, flush)
        elems = 2 * (tx.numel() + tw.numel() + tdy.numel())
        flops = 3 * 2.0 * T * F * H
        qg = elems * Q_BYTES_PER_ELEM / (mq * 1e-3) / 1e9
        tf = flops / (mg * 1e-3) / 1e12
        e = {"quantize_ms": round(mq, 4), "quantize_gbs": round(qg, 1),
             "quantize_elems_per_s": round(elems / (mq * 1e-3)), "gemm_ms": round(mg, 4),
             "gemm_tflops": round(tf, 1),
             "quantize_ms_six_single_orientation_calls": round(mq1, 4)}
        e.update(_fracs(pk, qg, tf, g, 3 * sum(_gemm_bytes(c, F, H) for c in counts), flops))
        r[gn] = e
        del qs, y, dx, dw
    if o is not None:
        seg = m["x"][:4096]
        full = 2 * (tx.numel() + tw.numel() + tdy.numel())
        r["oracle"] = oracle_q(seg, full, "4096 routed rows of X (the first segments), RHT + E1M2",
                               grid=1, rht=True, rht_seed=2)
    del tx, tw, tdy, m
    torch.cuda.empty_cache()
    out["moe7p9b_grouped_step"] = r

    # ---- MoE 124B large layer on the E2M1 grid (the E1M2 step is the headline)
    d = moe124b_inputs(dev)
    T, H, F = WORKLOAD["tokens"], WORKLOAD["hidden"], WORKLOAD["ffn"]
    st = Step(U, d["x"], d["w"], d["dy"], U.UFP4_E2M1)
    mq = _ev_time(st.quantize_all, flush)
    mg = _ev_time(st.gemms, flush)
    qg = st.q_elems * Q_BYTES_PER_ELEM / (mq * 1e-3) / 1e9
    tf = sum(st.flops_each) / (mg * 1e-3) / 1e12
    e = {"quantize_ms": round(mq, 4), "quantize_gbs": round(qg, 1),
         "quantize_elems_per_s": round(st.q_elems / (mq * 1e-3)), "gemm_ms": round(mg, 4),
         "gemm_tflops": round(tf, 1)}
    e.update(_fracs(pk, qg, tf, 0, 3 * _gemm_bytes(T, F, H), sum(st.flops_each)))
    out["moe124b_layer_e2m1"] = dict(config="the headline layer on the E2M1 grid (UFP4 recipe otherwise)", **e)
    del st, d
    torch.cuda.empty_cache()

    # ---- compounding-attenuation chain: 100 x (4096^3), fresh W_k ~ N(0, 1/64)
    n, steps = 4096, 100
    rows = torch.arange(0, n, n // 64, device=dev)
    r = {"config": "100 sequential 4096^3 GEMMs, X_0 N(0,1), W_k N(0,1/64) BF16, each output re-quantized "
                   "from fp32 with its tensor amax taken from the GEMM epilogue (ufp4_gemm_amax); eta on 64 "
                   "sampled rows against the fp64 product"}
    for g, gn in ((0, "e2m1"), (1, "e1m2"), (2, "e2m1c")):
        for rht in (False, True):
            X = inputs.device_normal((n, n), 1.0, 50, dev, dtype=torch.float32)
            norm0 = float(X.double().norm())
            ln_prod, sum_delta, ln_alpha = 0.0, 0.0, 0.0
            qx = U.QTensor.empty(n, n, g, dev)
            qw = U.QTensor.empty(n, n, g, dev)
            Y = torch.empty(n, n, device=dev)
            amax = torch.empty(1, device=dev)
            t_gpu = 0.0
            for k in range(steps):
                W = inputs.device_normal((n, n), 1.0 / 64, 1000 + k, dev)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                # each output's amax comes from the GEMM epilogue that wrote it
                U.ufp4_quantize(X, g, rht=rht, rht_seed=2, out=qx, amax_in=amax if k > 0 else None)
                U.ufp4_quantize(W, g, rht=rht, rht_seed=2, out=qw)
                U.ufp4_gemm_amax(qx, qw, rht=rht, rht_seed=2, out=Y, amax=amax)
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
            r["%s_rht_%s" % (gn, "on" if rht else "off")] = {
                "prod_eta": round(float(np.exp(ln_prod)), 6),
                "exp_minus_sum_delta": round(float(np.exp(-sum_delta)), 6),
                "prod_alpha_x_alpha_w": round(float(np.exp(ln_alpha)), 6),
                "norm_ratio": round(float(X.double().norm()) / norm0, 6),
                "gpu_ms_per_layer": round(t_gpu / steps, 4),
                "layer_tflops": round(2.0 * n ** 3 / (t_gpu / steps * 1e-3) / 1e12, 1)}
            del X, Y, qx, qw
    if o is not None:
        Xh = inputs.rng(50).standard_normal((512, n), dtype=np.float32)
        r["oracle"] = oracle_q(Xh, steps * 2 * n * n, "512 rows of an fp32 4096-wide X, RHT + E1M2",
                               grid=1, rht=True, rht_seed=2)
    out["attenuation_chain_4096_x100"] = r
    torch.cuda.empty_cache()
    return out


def build_parser():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true",
                    help="skip the secondary measurements (the quantizer on X and the five workloads)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shape", default="dense", choices=["dense", "moe124b"],
                    help="layer shape of --kernel")
    ap.add_argument("--kernel", default=None,
                    choices=["gemm_e2m1", "gemm_e1m2", "gemm_e1m2_dx", "gemm_e1m2_dw", "gemm_mxfp4",
                             "quant_row_e1m2", "quant_col_e1m2", "quant_dual_e1m2",
                             "quant_dual_sr_e1m2", "amax_dual_e1m2",
                             "quant_row_e2m1", "quant_col_e2m1", "quant_grouped_dual_e1m2", "quant_resident_e1m2",
                             "all"],
                    help="time one kernel of the step in isolation (profiling); all: every public call once")
    return ap


def main():
    ap = build_parser()
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.kernel == "all":
        run_all_kernels(args)
    elif args.kernel:
        run_kernel(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
