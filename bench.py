"""Benchmark of the FP4 block-scaled quantize-and-multiply hot path on GB300.

One step = one refresh step (current amax, D = 1) of a linear layer's forward
and backward pass through the FP4 path on the 8B MLP down_proj shapes:
  amax(X), amax(W), amax(dY);
  producers: X row + transposed (T=448), W 2D 16x16 row + transposed,
             dY row + transposed with Philox stochastic rounding (seed 42);
  UE5M3 scale remap onto the tensor core's E4M3 scale path (both copies);
  GEMMs: fprop Y = X W^T (8192 x 4096 x 14336, BF16 out),
         dgrad dX = dY W (8192 x 14336 x 4096, BF16 out),
         wgrad dW = dY^T X (4096 x 14336 x 8192, FP32 out).
Inputs are seeded synthetic tensors with the workload's distributions,
resident in HBM when the timed region starts; L2 is flushed (a read of a
clean buffer twice its size) before every timed step.  Step times are the
median over the timed steps.

`value` is the step's roofline-normalised throughput: the time the step's
kernels would take at the roofline (quantizer and amax bytes at the measured
HBM bandwidth, GEMM flops at the FP4 dense peak) divided by the measured step
time, in % of one GB300, summed over GPUs (each rank runs its own replica).

`--impl reference` times the CPU oracle (test infrastructure) on a bounded
sample of the same workload, extrapolated to a full step.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

M_TOK, K_FF, N_MODEL = 8192, 14336, 4096
WORKLOAD = "8B MLP down_proj fwd+bwd (refresh step), UE5M3-b16"
FMT_NAMES = {0: "UE5M3-b16", 1: "NVFP4-b16", 2: "MXFP4-b32", 3: "UE5M3-b32",
             4: "NVFP4-CTA-local (tensor scale per 128-row stripe)"}
CTA = 4  # CTA-local NVFP4: current stripe maxima, 1D weight copies
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense FP4 / BF16 tensor ratio on GB300
UNIT = "% of one GB300 roofline (step ideal time / step time, summed over GPUs)"
L2_FLUSH_BYTES = 2 * 129 * 1000 * 1000  # twice the L2
SLEEP_CYCLES = 100_000  # ~50 us of device-side wait before a timed region


def flush_l2(buf):
    """Evict L2 by reading a clean buffer twice its size (a read leaves no
    dirty lines whose write-back would land in the next timed kernel)."""
    torch.amax(buf)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, source="fallback")


def work_model(fmt):
    """Algorithmic bytes / flops of one step (what the method must move)."""
    B = 32 if fmt in (2, 3) else 16
    per_copy = 0.5 + 1.0 / B
    ex, ew, edy = M_TOK * K_FF, N_MODEL * K_FF, M_TOK * N_MODEL
    amax_bytes = 2.0 * (ex + ew + edy)
    quant_bytes = {
        "X": ex * (2 + 2 * per_copy) + 8,
        "W": ew * (2 + 2 * per_copy) + 8,
        "dY": edy * (2 + 2 * per_copy) + 8,
    }
    gemms = {
        "fprop": (M_TOK, N_MODEL, K_FF, 2),
        "dgrad": (M_TOK, K_FF, N_MODEL, 2),
        "wgrad": (N_MODEL, K_FF, M_TOK, 4),
    }
    flops = {k: 2.0 * m * n * k_ for k, (m, n, k_, _) in gemms.items()}
    return amax_bytes, quant_bytes, gemms, flops


class Clocks:
    """nvidia-smi sampler running during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.lines = index, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def reduce_max(v, world):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ GPU arm

class Layer:
    """All device buffers of one step, allocated once; `step()` enqueues the
    whole hot path on the current stream through the C ABI."""

    def __init__(self, fmt, seed, device, host=None):
        import fp4_block_scaled_quantize_gb300 as fq
        from fp4_block_scaled_quantize_gb300 import inputs
        self.fq = fq
        if host is None:
            d = inputs.down_proj_8b(seed=seed)
            host = {k: v.pin_memory() for k, v in d.items()}
        self.host = host
        self.X, self.W, self.dY = (self.host[k].to(device) for k in ("X", "W", "dY"))
        self.fmt = fmt
        mma = fq.FP4_SF_MMA
        self.px = fq.params(format=fmt, T=448.0, sf_layout=mma)
        # (the stripe contract has no 2D tiles: W gets two 1D copies)
        self.pw = fq.params(format=fmt, T=448.0, block2d=(fmt != CTA), sf_layout=mma)
        self.pdy = fq.params(format=fmt, T=448.0, round_row=fq.FP4_ROUND_SR,
                             round_col=fq.FP4_ROUND_SR, sr_seed=42, sf_layout=mma)
        f32 = dict(dtype=torch.float32, device=device)
        if fmt == CTA:
            # stripe maxima: per 128-row stripe (row-wise copy) and per
            # 128-column stripe (transposed copy) of each operand
            self.amax = {k: (torch.zeros(fq.n_stripes(t.shape[0]), **f32),
                             torch.zeros(fq.n_stripes(t.shape[1]), **f32))
                         for k, t in (("X", self.X), ("W", self.W), ("dY", self.dY))}
        else:
            # one amax per operand (no rotation: the transposed copy uses it too)
            self.amax = {k: (a, a) for k, a in ((k, torch.zeros(1, **f32))
                                                for k in ("X", "W", "dY"))}
        self.refresh_amax()
        self.xr, self.xc = fq.quantize_transpose(self.X, *self.amax["X"], self.px)
        self.wr, self.wc = fq.quantize_transpose(self.W, *self.amax["W"], self.pw)
        self.dyr, self.dyc = fq.quantize_transpose(self.dY, *self.amax["dY"], self.pdy)
        self.Y = torch.empty((M_TOK, N_MODEL), dtype=torch.bfloat16, device=device)
        self.dX = torch.empty((M_TOK, K_FF), dtype=torch.bfloat16, device=device)
        self.dW = torch.empty((N_MODEL, K_FF), dtype=torch.float32, device=device)

    def refresh_amax(self):
        fq = self.fq
        if self.fmt == CTA:
            for k, t in (("X", self.X), ("W", self.W), ("dY", self.dY)):
                fq._check(fq.fp4_amax_stripes(t, *self.amax[k]), "amax stripes")
            return
        fq._check(fq.fp4_amax_many([self.X, self.W, self.dY],
                                   [self.amax[k][0] for k in ("X", "W", "dY")]), "amax")

    def _qt(self, x, key, p, r, c):
        fq = self.fq
        a_r, a_c = self.amax[key]
        fq._check(fq.fp4_quantize_transpose(x, a_r, a_c, p, r.q, r.sf, r.s_dec, r.row_shift,
                                            c.q, c.sf, c.s_dec, c.row_shift), "qt " + key)

    def step(self, events=None):
        fq = self.fq
        ev = events if events is not None else {}

        def mark(name):
            if name in ev:
                ev[name].record()

        mark("amax")
        self.refresh_amax()
        mark("quant_X")
        self._qt(self.X, "X", self.px, self.xr, self.xc)
        mark("quant_W")
        self._qt(self.W, "W", self.pw, self.wr, self.wc)
        mark("quant_dY")
        self._qt(self.dY, "dY", self.pdy, self.dyr, self.dyc)
        mark("fprop")
        fq.gemm(self.xr, self.wr, out=self.Y)
        mark("dgrad")
        fq.gemm(self.dyr, self.wc, out=self.dX)
        mark("wgrad")
        fq.gemm(self.dyc, self.xc, out=self.dW)
        mark("end")


def measure_layer(layer, args, world, flush):
    """Warm-up, one CUDA graph of the whole step, the timed steps (median,
    L2 flushed before each) and a per-kernel breakdown of the same step
    launched kernel by kernel between events on the launching stream."""
    fq = layer.fq
    names = ["amax", "quant_X", "quant_W", "quant_dY", "fprop", "dgrad", "wgrad", "end"]
    for _ in range(args.warmup):
        layer.step()
    st = fq.fp4_status_sync()
    if st != fq.FP4_OK:
        raise RuntimeError("device status after warm-up: " + fq.STATUS_NAMES[st])
    torch.cuda.synchronize()
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            layer.step()
        graph.replay()
        torch.cuda.synchronize()
    barrier(world)
    step_ms = []
    for _ in range(args.steps):
        flush_l2(flush)
        s_ev = torch.cuda.Event(enable_timing=True)
        e_ev = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        # a short device-side wait lets the host enqueue the step before the
        # start event fires, so host launch latency stays out of the step
        torch.cuda._sleep(SLEEP_CYCLES)
        s_ev.record()
        if graph is not None:
            graph.replay()
        else:
            layer.step()
        e_ev.record()
        torch.cuda.synchronize()
        step_ms.append(s_ev.elapsed_time(e_ev))
    barrier(world)
    per_kernel = {n: [] for n in names[:-1]}
    for _ in range(min(args.steps, 50)):
        flush_l2(flush)
        ev = {n: torch.cuda.Event(enable_timing=True) for n in names}
        torch.cuda.synchronize()
        torch.cuda._sleep(4 * SLEEP_CYCLES)
        layer.step(ev)
        torch.cuda.synchronize()
        for a_, b_ in zip(names, names[1:]):
            per_kernel[a_].append(ev[a_].elapsed_time(ev[b_]))
    st = fq.fp4_status_sync()
    if st != fq.FP4_OK:
        raise RuntimeError("device status after timed steps: " + fq.STATUS_NAMES[st])
    return {"step_ms": reduce_max(statistics.median(step_ms), world),
            "kernel_ms": {k: statistics.median(v) for k, v in per_kernel.items()},
            "graph": graph}


def summarize_layer(fmt, m, pk, world):
    """Step value, producer GB/s and GEMM TFLOP/s of one measured layer."""
    amax_b, qbytes, gemms, flops = work_model(fmt)
    hbm = pk["hbm_gbs"] * 1e9
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16
    ideal = amax_b / hbm + sum(qbytes.values()) / hbm + sum(flops.values()) / (fp4_peak * 1e12)
    avg = m["kernel_ms"]
    q_ms = avg["quant_X"] + avg["quant_W"] + avg["quant_dY"]
    g_ms = avg["fprop"] + avg["dgrad"] + avg["wgrad"]
    quant_gbs = sum(qbytes.values()) / (q_ms * 1e-3) / 1e9
    gemm_tflops = sum(flops.values()) / (g_ms * 1e-3) / 1e12
    per_producer = {}
    for k in ("X", "W", "dY"):
        ms = avg["quant_" + k]
        gbs = qbytes[k] / (ms * 1e-3) / 1e9
        per_producer[k] = {"ms": round(ms, 4), "gbs": round(gbs, 1),
                           "frac": round(gbs / pk["hbm_gbs"], 4)}
    per_gemm = {}
    B = 32 if fmt in (2, 3) else 16
    for k in ("fprop", "dgrad", "wgrad"):
        tf = flops[k] / (avg[k] * 1e-3) / 1e12
        # applicable roofline: the larger of the math time and the time to
        # move the operands and the output (FP32 outputs are not free)
        Mg, Ng, Kg, ob = gemms[k]
        gbytes = (Mg + Ng) * Kg * (0.5 + 1.0 / B) + Mg * Ng * ob
        t_roof = max(flops[k] / (fp4_peak * 1e12), gbytes / hbm)
        per_gemm[k] = {"ms": round(avg[k], 4), "tflops": round(tf, 1),
                       "frac": round(tf / fp4_peak, 4),
                       "roofline_us": round(t_roof * 1e6, 1),
                       "frac_of_applicable_roofline": round(t_roof / (avg[k] * 1e-3), 4)}
    return {
        "ideal_s": ideal,
        "value": 100.0 * ideal / (m["step_ms"] * 1e-3) * world,
        "quantize": {"gbs": round(quant_gbs, 1), "frac": round(quant_gbs / pk["hbm_gbs"], 4),
                     "ms": round(q_ms, 4), "per_producer": per_producer,
                     "note": "UE5M3 producers include the scale remap launch"
                             if fmt in (0, 3) else "one launch per producer"},
        "amax": {"gbs": round(amax_b / (avg["amax"] * 1e-3) / 1e9, 1),
                 "ms": round(avg["amax"], 4)},
        "gemm": {"tflops": round(gemm_tflops, 1), "frac": round(gemm_tflops / fp4_peak, 4),
                 "ms": {k: round(avg[k], 4) for k in ("fprop", "dgrad", "wgrad")},
                 "per_gemm": per_gemm},
    }


def run_gpu(args, world, rank, local):
    import fp4_block_scaled_quantize_gb300 as fq
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pk = peaks()
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16
    layer = Layer(args.format, seed=args.seed + rank, device=dev)
    amax_b, qbytes, gemms, flops = work_model(args.format)
    flush = torch.zeros(L2_FLUSH_BYTES // 2, dtype=torch.bfloat16, device=dev)

    with Clocks(local) as clk:
        m = measure_layer(layer, args, world, flush)
    graph = m["graph"]
    ms_step = m["step_ms"]
    summ = summarize_layer(args.format, m, pk, world)
    ideal, value, avg = summ["ideal_s"], summ["value"], m["kernel_ms"]
    dominant = max(("fprop", "dgrad", "wgrad"), key=lambda k: avg[k])
    dom_tflops = flops[dominant] / (avg[dominant] * 1e-3) / 1e12
    traffic = load_traffic(dominant)

    # end to end through the C ABI with host buffers: H2D inputs, step, D2H outputs
    fused = run_fused_producer(layer, flush)
    reencode = run_reencode(layer, flush, pk["hbm_gbs"])
    linear = run_linear(layer, flush)
    feed = run_gemm_feed(layer, flush)
    e2e = run_e2e(layer, args, world, ideal, graph)
    out_dtypes = run_out_dtypes(layer, flush, flops, fp4_peak)
    host = layer.host
    graphed = graph is not None
    del layer, graph, m
    torch.cuda.empty_cache()
    per_format = run_per_format(args, world, host, dev, flush, pk)
    fp8_vs_fp4 = run_fp8_vs_fp4(host, dev, flush, pk,
                                dict(per_format, **{FMT_NAMES[args.format]: summ}))
    exact = run_exact_path(host, dev, flush, pk, dict(per_format, **{FMT_NAMES[args.format]: summ}))
    del host
    configs = run_configs(dev, flush, pk)
    ceiling = run_mma_ceiling(dom_tflops)
    ceiling["gemm_feed"] = feed

    clocks = clk.summary()
    out = {
        "metric": "quantize GB/s and FP4 block-scaled GEMM TFLOP/s, each as % of GB300 roofline",
        "value": round(value, 3),
        "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e2m1 payload x fp32 accumulate (u8 codes)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "format": FMT_NAMES[args.format],
                   "X": [M_TOK, K_FF], "W": [N_MODEL, K_FF], "dY": [M_TOK, N_MODEL],
                   "amax": "current (D=1 refresh step)",
                   "l2": "flushed before each step (read of a clean 258 MB buffer)",
                   "timing": "median of the timed steps",
                   "launch": "CUDA graph of the whole step" if graphed else "eager",
                   "parallelism": f"replicas x{world}"},
        "quantize": summ["quantize"],
        "amax": summ["amax"],
        "gemm": summ["gemm"],
        "roofline": {"kernel": "k_gemm (" + dominant + ")", "bound": "tensor",
                     "achieved": round(dom_tflops, 1), "peak": round(fp4_peak, 1),
                     "unit": "TFLOP/s", "frac": round(dom_tflops / fp4_peak, 4),
                     "traffic": traffic,
                     "peak_source": f"{pk['source']} bf16 burst x {FP4_OVER_BF16:g} (nominal "
                                    "FP4/BF16 dense ratio)"},
        "clocks": clocks,
        "gpu_launches": layer_launches(args.format) * args.steps,
        "e2e": e2e,
        "gemm_out_dtypes": out_dtypes,
        "per_format": per_format,
        "fp8_vs_fp4": fp8_vs_fp4,
        "ue5m3_exact_path": exact,
        "tensor_pipe_ceiling": ceiling,
        "configs": configs,
        "epilogue_fused_producer": fused,
        "mxfp4_to_fp8": reencode,
        "linear_layer": linear,
    }
    if rank == 0:
        out["cpu_baseline"] = cpu_baseline(args, ideal)
        print(json.dumps(out))


def layer_launches(fmt):
    """Kernel launches of one step: amax (zeroing + one batched launch; the
    stripe contract: one stripe-maxima launch per operand), producers x3,
    GEMMs x3, one remap per UE5M3 producer."""
    return (3 if fmt == CTA else 2) + 3 + 3 + (3 if fmt in (0, 3) else 0)


def median_ms(fn, flush, reps=20):
    """Median device time of fn() over `reps` runs, each after an L2 flush:
    fn is captured once as a CUDA graph, and events on the launching stream
    bracket each replay."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    g.replay()
    torch.cuda.synchronize()
    evs = []
    for _ in range(reps):
        flush_l2(flush)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def run_out_dtypes(layer, flush, flops, fp4_peak):
    """The three GEMMs of the step with the other output type: fprop and dgrad
    to binary32, wgrad to BF16 (the step itself writes BF16, BF16, binary32)."""
    fq = layer.fq
    dev = layer.X.device
    y32 = torch.empty((M_TOK, N_MODEL), dtype=torch.float32, device=dev)
    dx32 = torch.empty((M_TOK, K_FF), dtype=torch.float32, device=dev)
    dw16 = torch.empty((N_MODEL, K_FF), dtype=torch.bfloat16, device=dev)
    runs = {"fprop_f32": ("fprop", lambda: fq.gemm(layer.xr, layer.wr, out=y32)),
            "dgrad_f32": ("dgrad", lambda: fq.gemm(layer.dyr, layer.wc, out=dx32)),
            "wgrad_bf16": ("wgrad", lambda: fq.gemm(layer.dyc, layer.xc, out=dw16))}
    out = {}
    for key, (g, fn) in runs.items():
        ms = median_ms(fn, flush)
        tf = flops[g] / (ms * 1e-3) / 1e12
        out[key] = {"ms": round(ms, 4), "tflops": round(tf, 1), "frac": round(tf / fp4_peak, 4)}
    fq._check(fq.fp4_status_sync(), "out dtypes")
    return out


def run_per_format(args, world, host, dev, flush, pk):
    """The same step under the comparison formats (NVFP4-b16, MXFP4-b32) and
    the UE5M3-b32 control, measured exactly as the headline format."""
    out = {}
    for fmt in (0, 1, 2, 3, CTA):
        if fmt == args.format:
            continue
        layer = Layer(fmt, seed=0, device=dev, host=host)
        m = measure_layer(layer, args, world, flush)
        summ = summarize_layer(fmt, m, pk, world)
        out[FMT_NAMES[fmt]] = {"value": round(summ["value"], 3), "unit": UNIT,
                               "ms_per_step": round(m["step_ms"], 4),
                               "launches_per_step": layer_launches(fmt),
                               "quantize": summ["quantize"], "amax": summ["amax"],
                               "gemm": summ["gemm"]}
        del layer, m
        torch.cuda.empty_cache()
    return out


def run_fp8_vs_fp4(host, dev, flush, pk, per_format):
    """The step's three GEMMs in FP8 on the re-encoded MXFP4 copies
    (fp4_mxfp4_to_fp8 for row-wise operands, fp4_mxfp4_to_fp8_transpose for
    the transposed ones) against the same GEMMs in FP4 (MXFP4-b32 and
    UE5M3-b16, from the step measurements).  FP8 peak: the measured BF16
    burst x 2 (nominal FP8 / BF16 dense ratio)."""
    import fp4_block_scaled_quantize_gb300 as fq
    X, W, dY = (host[k].to(dev) for k in ("X", "W", "dY"))
    p = fq.params(format=fq.FP4_FMT_MXFP4_B32, sf_layout=fq.FP4_SF_PLAIN)
    fp8 = {}
    for name, x in (("X", X), ("W", W), ("dY", dY)):
        (a,) = fq.amax_many([x])
        c = fq.quantize(x, a, p)
        sf = c.sf.view(x.shape[0], x.shape[1] // 32)
        fp8[name] = fq.mxfp4_to_fp8(c.q, sf)
        fp8[name + "t"] = fq.mxfp4_to_fp8_transpose(c.q, sf)
        del c, sf
    del X, W, dY
    torch.cuda.empty_cache()
    gemms = {"fprop": ("X", "W", torch.bfloat16), "dgrad": ("dY", "Wt", torch.bfloat16),
             "wgrad": ("dYt", "Xt", torch.float32)}
    fp8_peak = pk["bf16_tflops"] * 2.0
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16
    out = {"operands": "MXFP4-b32 copies of the step's X, W, dY re-encoded to E4M3-b128",
           "fp8_peak_tflops": round(fp8_peak, 1),
           "fp8_peak_source": f"{pk['source']} bf16 burst x 2 (nominal FP8/BF16 dense ratio)"}
    for g, (a, b, dt) in gemms.items():
        qa, sa = fp8[a]
        qb, sb = fp8[b]
        D = torch.empty((qa.shape[0], qb.shape[0]), dtype=dt, device=dev)
        ms = median_ms(lambda: fq.fp8_gemm(qa, sa, qb, sb, out=D), flush)
        flop = 2.0 * qa.shape[0] * qb.shape[0] * qa.shape[1]
        tf = flop / (ms * 1e-3) / 1e12
        row = {"shape": [qa.shape[0], qb.shape[0], qa.shape[1]], "fp8_ms": round(ms, 4),
               "fp8_tflops": round(tf, 1), "fp8_frac_of_fp8_peak": round(tf / fp8_peak, 4)}
        for fmt_name in ("MXFP4-b32", "UE5M3-b16"):
            pf = per_format.get(fmt_name)
            if pf is not None:
                g4 = pf["gemm"]["per_gemm"][g]
                row[fmt_name + "_ms"] = g4["ms"]
                row[fmt_name + "_tflops"] = g4["tflops"]
        out[g] = row
        del D
    fq._check(fq.fp4_status_sync(), "fp8 gemm")
    out["note"] = "FP4 figures are the step's GEMMs (frac of FP4 peak " + \
                  f"{round(fp4_peak, 1)} TFLOP/s in per_format)"
    return out


def run_exact_path(host, dev, flush, pk, per_format):
    """The exact path for UE5M3 copies outside the E4M3 scale window on the
    step's fprop: plain-layout UE5M3-b16 copies of X and W, fp4_dequantize of
    each (0.5 + 1/16 B read, 2 B written per element) and fp4_gemm_bf16 on
    the BF16 tensor cores (peak: the measured BF16 burst), against the FP4
    fprop of the step."""
    import fp4_block_scaled_quantize_gb300 as fq
    X, W = (host[k].to(dev) for k in ("X", "W"))
    p = fq.params(format=fq.FP4_FMT_UE5M3_B16, sf_layout=fq.FP4_SF_PLAIN)
    cx = fq.quantize(X, fq.amax_many([X])[0], p)
    cw = fq.quantize(W, fq.amax_many([W])[0], p)
    del X, W
    torch.cuda.empty_cache()
    yx = torch.empty((M_TOK, K_FF), dtype=torch.bfloat16, device=dev)
    yw = torch.empty((N_MODEL, K_FF), dtype=torch.bfloat16, device=dev)
    D = torch.empty((M_TOK, N_MODEL), dtype=torch.bfloat16, device=dev)
    deq_x = lambda: fq._check(fq.fp4_dequantize(cx.q, cx.sf, cx.format, M_TOK, K_FF, yx), "deq")
    deq_w = lambda: fq._check(fq.fp4_dequantize(cw.q, cw.sf, cw.format, N_MODEL, K_FF, yw), "deq")
    mm = lambda: fq.gemm_bf16(yx, yw, cx.s_dec, cw.s_dec, out=D)
    deq_x()
    deq_w()
    mm()
    fq._check(fq.fp4_status_sync(), "exact path")
    out = {"operands": "plain-layout UE5M3-b16 copies of the step's X and W",
           "bf16_peak_tflops": round(pk["bf16_tflops"], 1),
           "bf16_peak_source": f"{pk['source']} bf16 burst"}
    nb = M_TOK * K_FF * (0.5 + 1 / 16 + 2)
    ms = graph_ms(deq_x, flush)
    gbs = nb / (ms * 1e-3) / 1e9
    out["dequantize_X"] = {"shape": [M_TOK, K_FF], "bytes_per_launch": int(nb), "ms": round(ms, 4),
                           "gbs": round(gbs, 1), "frac": round(gbs / pk["hbm_gbs"], 4)}
    ms_w = graph_ms(deq_w, flush)
    ms_g = median_ms(mm, flush)
    flop = 2.0 * M_TOK * N_MODEL * K_FF
    tf = flop / (ms_g * 1e-3) / 1e12
    out["gemm_bf16_fprop"] = {"shape": [M_TOK, N_MODEL, K_FF], "ms": round(ms_g, 4),
                              "tflops": round(tf, 1), "frac": round(tf / pk["bf16_tflops"], 4)}
    out["exact_fprop_ms"] = round(ms + ms_w + ms_g, 4)
    pf = per_format.get("UE5M3-b16")
    if pf is not None:
        out["fp4_fprop_ms"] = pf["gemm"]["per_gemm"]["fprop"]["ms"]
    return out


def run_mma_ceiling(dominant_tflops):
    """What the tensor pipe sustains on this device for the GEMMs' MMA forms
    (fp4_mma_loop: back-to-back M128 N256 MMAs on resident operands, no
    copies or hand-offs), beside the dominant GEMM's rate.  Context for the
    roofline, whose peak stays the measured BF16 burst x the nominal ratio."""
    import fp4_block_scaled_quantize_gb300 as fq
    out = {"what": "tcgen05.mma M128 N256 back to back on operands resident in shared memory "
                   "(fp4_mma_loop), median of 5 launches"}
    for name, kind in (("fp4", fq.FP4_MMA_FP4), ("fp8", fq.FP4_MMA_FP8), ("bf16", fq.FP4_MMA_BF16)):
        out[name + "_tflops"] = round(fq.mma_loop_tflops(kind), 1)
    out["dominant_gemm_frac_of_fp4_loop"] = round(dominant_tflops / out["fp4_tflops"], 4)
    return out


def run_gemm_feed(layer, flush, reps=5):
    """Each GEMM of the step against its own copies into shared memory
    (gemm_copies: the same tiles, boxes, scale tiles and ring, no MMA and no
    output), both L2-flushed, median of `reps`: the share of the GEMM's time
    that filling its shared memory takes, and the fill rate per SM it implies
    (each CTA takes in 128 rows of A and of B and its scale tiles per K256
    stage)."""
    fq = layer.fq
    sms = torch.cuda.get_device_properties(layer.X.device).multi_processor_count
    stage = 2 * 16384 + 3 * (2 if layer.fmt == 2 else 4) * 512

    def med(fn):
        ts = []
        for _ in range(reps + 1):
            flush_l2(flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        ts = sorted(ts[1:])
        return ts[len(ts) // 2]

    out = {"what": "GEMM vs its own copies alone (fp4_gemm_copies), L2 flushed, median of %d" % reps,
           "stage_bytes_per_cta": stage}
    for k, a, b, D in (("fprop", layer.xr, layer.wr, layer.Y), ("dgrad", layer.dyr, layer.wc, layer.dX),
                       ("wgrad", layer.dyc, layer.xc, layer.dW)):
        t_g = med(lambda: fq.gemm(a, b, out=D))
        t_c = med(lambda: fq.gemm_copies(a, b))
        tiles = -(-a.rows // 256) * -(-b.rows // 256)
        nbytes = tiles * -(-a.k // 256) * 2 * stage
        out[k] = {"gemm_us": round(t_g * 1e3, 1), "copies_us": round(t_c * 1e3, 1),
                  "copies_share": round(t_c / t_g, 3),
                  "fill_gbs_per_sm": round(nbytes / sms / (t_c * 1e-3) / 1e9, 1)}
    layer.fq._check(fq.fp4_status_sync(), "gemm_copies")
    return out


# ------------------------------------------------------------ other configs

SWEEP_SIZES = (2048, 4096, 8192, 16384)
HAD32_SIGNS = 0x5A5AF00F  # fixed sign vector of the 32-point rotation


def _qt(fq, x, a_r, a_c, p, r, c):
    fq._check(fq.fp4_quantize_transpose(x, a_r, a_c, p, r.q, r.sf, r.s_dec, r.row_shift,
                                        c.q, c.sf, c.s_dec, c.row_shift), "quantize_transpose")


def _q(fq, x, a, p, r):
    fq._check(fq.fp4_quantize(x, a, p, r.q, r.sf, r.s_dec, r.row_shift), "quantize")


def producer_bytes(fmt, elems, copies):
    """Algorithmic bytes of a producer: 2 B read per element, per copy 0.5 B
    of payload and 1/B of scale bytes, 4 B of s_dec."""
    B = 32 if fmt in (2, 3) else 16
    return elems * (2.0 + copies * (0.5 + 1.0 / B)) + 4 * copies


def _rate(nbytes=None, flop=None, ms=None, pk=None):
    if flop is not None:
        tf = flop / (ms * 1e-3) / 1e12
        peak = pk["bf16_tflops"] * FP4_OVER_BF16
        return {"ms": round(ms, 4), "tflops": round(tf, 1), "frac": round(tf / peak, 4)}
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"ms": round(ms, 4), "gbs": round(gbs, 1), "frac": round(gbs / pk["hbm_gbs"], 4)}


def config_tiny(fq, dev, flush):
    """Tiny UE5M3-b16 layer (X, W 256 x 256, seed 0): fresh amax of both, the
    X producer (row + transposed), the 2D W producer (row + transposed) and
    Y = X W^T.  Launch-bound: latency only."""
    from fp4_block_scaled_quantize_gb300 import inputs
    d = inputs.tiny(seed=0)
    X, W = d["X"].to(dev), d["W"].to(dev)
    mma = fq.FP4_SF_MMA
    px = fq.params(format=0, T=448.0, sf_layout=mma)
    pw = fq.params(format=0, T=448.0, block2d=True, sf_layout=mma)
    ax = torch.zeros(1, dtype=torch.float32, device=dev)
    aw = torch.zeros(1, dtype=torch.float32, device=dev)
    fq._check(fq.fp4_amax_many([X, W], [ax, aw]), "amax")
    xr, xc = fq.quantize_transpose(X, ax, ax, px)
    wr, wc = fq.quantize_transpose(W, aw, aw, pw)
    Y = torch.empty((256, 256), dtype=torch.float32, device=dev)

    def step():
        fq._check(fq.fp4_amax_many([X, W], [ax, aw]), "amax")
        _qt(fq, X, ax, ax, px, xr, xc)
        _qt(fq, W, aw, aw, pw, wr, wc)
        fq.gemm(xr, wr, out=Y)

    dev_ms = median_ms(step, flush, reps=50)
    step()
    torch.cuda.synchronize()
    host = []
    for _ in range(50):
        t0 = time.perf_counter()
        step()
        torch.cuda.synchronize()
        host.append(time.perf_counter() - t0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    replay = []
    for _ in range(50):
        t0 = time.perf_counter()
        g.replay()
        torch.cuda.synchronize()
        replay.append(time.perf_counter() - t0)
    fq._check(fq.fp4_status_sync(), "tiny")
    return {"shape": "X [256, 256], W [256, 256], Y = X W^T (binary32)", "format": "UE5M3-b16",
            "launches": 2 + 2 + 2 + 1,
            "device_us": round(dev_ms * 1e3, 2),
            "host_eager_us": round(statistics.median(host) * 1e6, 1),
            "host_graph_replay_us": round(statistics.median(replay) * 1e6, 1),
            "note": "launch-bound; latency only, no roofline claim"}


def config_forward(fq, dev, flush, pk):
    """Forward layer: X [8192, 4096] N(0,1) with 1% of channels scaled by
    LogNormal(0,1), W [4096, 4096] N(0, 0.02) with 2D tiles; row-wise
    producers, fprop M=8192 N=4096 K=4096, UE5M3-b16 and NVFP4-b16, RNE."""
    from fp4_block_scaled_quantize_gb300 import inputs
    d = inputs.forward_layer(seed=0)
    X, W = d["X"].to(dev), d["W"].to(dev)
    M, K, N = X.shape[0], X.shape[1], W.shape[0]
    out = {"shapes": {"X": [M, K], "W": [N, K]}}
    ax, aw = fq.amax_many([X, W])
    Y16 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    Y32 = torch.empty((M, N), dtype=torch.float32, device=dev)
    for fmt in (0, 1):
        mma = fq.FP4_SF_MMA
        px = fq.params(format=fmt, T=448.0, sf_layout=mma)
        pw = fq.params(format=fmt, T=448.0, block2d=True, sf_layout=mma)
        xr, wr = fq.quantize(X, ax, px), fq.quantize(W, aw, pw)
        flop = 2.0 * M * N * K
        out[FMT_NAMES[fmt]] = {
            "quant_X_row": _rate(producer_bytes(fmt, M * K, 1),
                                 ms=median_ms(lambda: _q(fq, X, ax, px, xr), flush), pk=pk),
            "quant_W_2d_row": _rate(producer_bytes(fmt, N * K, 1),
                                    ms=median_ms(lambda: _q(fq, W, aw, pw, wr), flush), pk=pk),
            "fprop_bf16": _rate(flop=flop, ms=median_ms(lambda: fq.gemm(xr, wr, out=Y16), flush),
                                pk=pk),
            "fprop_f32": _rate(flop=flop, ms=median_ms(lambda: fq.gemm(xr, wr, out=Y32), flush),
                               pk=pk),
        }
        del xr, wr
    out["amax_ms"] = round(median_ms(lambda: fq.amax_many([X, W]), flush), 4)
    fq._check(fq.fp4_status_sync(), "forward config")
    return out


def config_backward_sr(fq, dev, flush, pk):
    """Backward with SR: dY [8192, 4096] Student-t(3) * 1e-4 quantised with a
    stale held amax (half the true one), UE5M3-b16 T=2048, Philox SR seed 42
    on both copies; X [8192, 4096] (N(0,1), 0.1% x50) row + transposed, RNE,
    T=448, fresh amax; W [4096, 4096] 2D; dgrad dX = dY W, wgrad dW = dY^T X."""
    from fp4_block_scaled_quantize_gb300 import inputs
    d = inputs.backward_sr(seed=0)
    dY, X, W = d["dY"].to(dev), d["X"].to(dev), d["W"].to(dev)
    M, N = dY.shape
    K_in = X.shape[1]
    mma = fq.FP4_SF_MMA
    ady, ax, aw = fq.amax_many([dY, X, W])
    ady_held = ady * 0.5
    pdy = fq.params(format=0, T=2048.0, round_row=fq.FP4_ROUND_SR, round_col=fq.FP4_ROUND_SR,
                    sr_seed=42, sf_layout=mma)
    px = fq.params(format=0, T=448.0, sf_layout=mma)
    pw = fq.params(format=0, T=448.0, block2d=True, sf_layout=mma)
    dyr, dyc = fq.quantize_transpose(dY, ady_held, ady_held, pdy)
    xr, xc = fq.quantize_transpose(X, ax, ax, px)
    wr, wc = fq.quantize_transpose(W, aw, aw, pw)
    dX16 = torch.empty((M, K_in), dtype=torch.bfloat16, device=dev)
    dX32 = torch.empty((M, K_in), dtype=torch.float32, device=dev)
    dW32 = torch.empty((N, K_in), dtype=torch.float32, device=dev)
    dW16 = torch.empty((N, K_in), dtype=torch.bfloat16, device=dev)
    f_dgrad = 2.0 * M * K_in * N
    f_wgrad = 2.0 * N * K_in * M
    out = {"shapes": {"dY": [M, N], "X": [M, K_in], "W": [N, K_in]},
           "dgrad": [M, K_in, N], "wgrad": [N, K_in, M],
           "quant_dY_sr_row_col": _rate(producer_bytes(0, M * N, 2), ms=median_ms(
               lambda: _qt(fq, dY, ady_held, ady_held, pdy, dyr, dyc), flush), pk=pk),
           "quant_X_row_col": _rate(producer_bytes(0, M * K_in, 2), ms=median_ms(
               lambda: _qt(fq, X, ax, ax, px, xr, xc), flush), pk=pk),
           "quant_W_2d_row_col": _rate(producer_bytes(0, N * K_in, 2), ms=median_ms(
               lambda: _qt(fq, W, aw, aw, pw, wr, wc), flush), pk=pk),
           "dgrad_bf16": _rate(flop=f_dgrad, ms=median_ms(lambda: fq.gemm(dyr, wc, out=dX16),
                                                          flush), pk=pk),
           "dgrad_f32": _rate(flop=f_dgrad, ms=median_ms(lambda: fq.gemm(dyr, wc, out=dX32),
                                                         flush), pk=pk),
           "wgrad_f32": _rate(flop=f_wgrad, ms=median_ms(lambda: fq.gemm(dyc, xc, out=dW32),
                                                         flush), pk=pk),
           "wgrad_bf16": _rate(flop=f_wgrad, ms=median_ms(lambda: fq.gemm(dyc, xc, out=dW16),
                                                          flush), pk=pk),
           "format": "UE5M3-b16 (dY T=2048 SR, X and W T=448 RNE)"}
    fq._check(fq.fp4_status_sync(), "backward config")
    return out


def config_sweep(fq, dev, flush, pk):
    """GEMM sweep: (M, N, K) in {2048, 4096, 8192, 16384}^3 plus
    (8192, 14336, 4096) and (14336, 8192, 4096); A [M, K] and B [N, K] are
    N(0,1) with 1% of entries x50 (seeds 7 and 8, drawn on the device),
    quantised row-wise to UE5M3-b16; BF16 output.  Then the three producer
    variants on a [8192, 8192] operand pair: MXFP4-b32 with the fixed-sign
    32-point rotation on the transposed (wgrad) copies, UE5M3-b16 with H16,
    UE5M3-b16 without rotation, each with its wgrad GEMM on those copies."""
    from fp4_block_scaled_quantize_gb300 import inputs
    mma = fq.FP4_SF_MMA
    p = fq.params(format=0, T=448.0, sf_layout=mma)
    cache = {}

    def operand(role, rows, k):
        key = (role, rows, k)
        if key not in cache:
            x = inputs.sweep_operand(rows, k, seed=7 if role == "A" else 8, device=dev)
            (a,) = fq.amax_many([x])
            cache[key] = fq.quantize(x, a, p)
            del x
        return cache[key]

    shapes = [(m, n, k) for m in SWEEP_SIZES for n in SWEEP_SIZES for k in SWEEP_SIZES]
    shapes += [(8192, 14336, 4096), (14336, 8192, 4096)]
    tflops = {}
    fracs = []
    for m, n, k in shapes:
        A, B = operand("A", m, k), operand("B", n, k)
        D = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        ms = median_ms(lambda: fq.gemm(A, B, out=D), flush, reps=10)
        r = _rate(flop=2.0 * m * n * k, ms=ms, pk=pk)
        tflops[f"{m}x{n}x{k}"] = r["tflops"]
        fracs.append(r["frac"])
        del D
    fq._check(fq.fp4_status_sync(), "sweep")
    cache.clear()
    torch.cuda.empty_cache()
    variants = {}
    R = 8192
    xa = inputs.sweep_operand(R, R, seed=7, device=dev)
    xb = inputs.sweep_operand(R, R, seed=8, device=dev)
    for name, fmt, had, signs in (("MXFP4-b32 + H32", 2, 32, HAD32_SIGNS),
                                  ("UE5M3-b16 + H16", 0, 16, 0),
                                  ("UE5M3-b16", 0, 0, 0)):
        pv = fq.params(format=fmt, T=448.0, hadamard_n=had, hadamard_signs=signs, sf_layout=mma)
        copies = []
        for x in (xa, xb):
            ar, ac = fq.amax(x, had, signs)
            r_, c_ = fq.quantize_transpose(x, ar, ac, pv)
            copies.append((x, ar, ac, r_, c_))
        x, ar, ac, r_, c_ = copies[0]
        amax_ms = median_ms(lambda: fq.amax(x, had, signs), flush)
        q_ms = median_ms(lambda: _qt(fq, x, ar, ac, pv, r_, c_), flush)
        D = torch.empty((R, R), dtype=torch.float32, device=dev)
        ca, cb = copies[0][4], copies[1][4]
        g_ms = median_ms(lambda: fq.gemm(ca, cb, out=D), flush)
        variants[name] = {"amax_view": _rate(2.0 * R * R, ms=amax_ms, pk=pk),
                          "producer_row_col": _rate(producer_bytes(fmt, R * R, 2), ms=q_ms, pk=pk),
                          "wgrad_gemm_f32": _rate(flop=2.0 * R ** 3, ms=g_ms, pk=pk)}
        del copies, D
    fq._check(fq.fp4_status_sync(), "sweep variants")
    fs = sorted(fracs)
    return {"format": "UE5M3-b16", "out": "bf16", "shapes": len(shapes),
            "inputs": "N(0,1), 1% of entries x50, drawn on the device (seeds 7, 8)",
            "tflops": tflops,
            "frac": {"min": fs[0], "median": fs[len(fs) // 2], "max": fs[-1]},
            "producer_variants": {"shape": [R, R], "variants": variants}}


def run_configs(dev, flush, pk):
    import fp4_block_scaled_quantize_gb300 as fq
    out = {"tiny_256": config_tiny(fq, dev, flush)}
    torch.cuda.empty_cache()
    out["forward_8192x4096"] = config_forward(fq, dev, flush, pk)
    torch.cuda.empty_cache()
    out["backward_sr_8192x4096"] = config_backward_sr(fq, dev, flush, pk)
    torch.cuda.empty_cache()
    out["sweep"] = config_sweep(fq, dev, flush, pk)
    torch.cuda.empty_cache()
    return out


def graph_ms(fn, flush, reps=20):
    """Device time of fn() per call: CUDA graphs of [L2 flush, fn] and of
    [L2 flush] alone, replayed back to back, difference of the two."""
    def cap(with_fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            flush_l2(flush)
            if with_fn:
                fn()
        return g

    def t(g):
        g.replay()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    return t(cap(True)) - t(cap(False))


def run_fused_producer(layer, flush):
    """fprop with the next layer's producer fused into the GEMM epilogue
    (fp4_gemm_quantize: the row-wise FP4 copy of Y is written instead of Y)
    against the unfused pair (BF16 Y written, then read back by
    fp4_quantize).  Held amax of Y from a previous step."""
    fq = layer.fq
    fq.gemm(layer.xr, layer.wr, out=layer.Y)
    amax_y, _ = fq.amax(layer.Y)
    p = fq.params(format=layer.fmt, T=448.0, sf_layout=fq.FP4_SF_MMA)
    ws = fq._want_shift(p, True)
    fused_out = fq._alloc_copy(M_TOK, N_MODEL, p, layer.Y.device, ws)
    plain_out = fq._alloc_copy(M_TOK, N_MODEL, p, layer.Y.device, ws)
    a, b = layer.xr.operand(), layer.wr.operand()

    def fused():
        fq._check(fq.fp4_gemm_quantize(a, b, M_TOK, N_MODEL, K_FF, amax_y, p, fused_out.q,
                                       fused_out.sf, fused_out.s_dec, fused_out.row_shift),
                  "fused")

    def unfused():
        fq.gemm(layer.xr, layer.wr, out=layer.Y)
        fq._check(fq.fp4_quantize(layer.Y, amax_y, p, plain_out.q, plain_out.sf,
                                  plain_out.s_dec, plain_out.row_shift), "unfused")

    t_f = graph_ms(fused, flush)
    t_u = graph_ms(unfused, flush)
    fq._check(fq.fp4_status_sync(), "fused producer")
    return {"gemm": "fprop %d x %d x %d" % (M_TOK, N_MODEL, K_FF),
            "fused_ms": round(t_f, 4), "unfused_ms": round(t_u, 4),
            "hbm_bytes_avoided": 2 * M_TOK * N_MODEL * 2,
            "note": "fused quantises the binary32 product; unfused quantises the stored BF16 Y"}


def run_reencode(layer, flush, hbm_gbs):
    """Direct MXFP4-b32 -> FP8 E4M3-b128 re-encoding (fp4_mxfp4_to_fp8) of X's
    MXFP4 row-wise copy, 8192 x 14336: 0.5 + 1/32 B read and 1 + 4/128 B
    written per element."""
    fq = layer.fq
    p = fq.params(format=fq.FP4_FMT_MXFP4_B32, sf_layout=fq.FP4_SF_PLAIN)
    mx = fq.quantize(layer.X, layer.amax["X"][0], p)
    sf = mx.sf.view(M_TOK, K_FF // 32)
    q8 = torch.empty((M_TOK, K_FF), dtype=torch.uint8, device=layer.X.device)
    s8 = torch.empty((M_TOK, K_FF // 128), dtype=torch.float32, device=layer.X.device)
    q8t = torch.empty((K_FF, M_TOK), dtype=torch.uint8, device=layer.X.device)
    s8t = torch.empty((K_FF, M_TOK // 128), dtype=torch.float32, device=layer.X.device)
    run = lambda: fq._check(fq.fp4_mxfp4_to_fp8(mx.q, sf, M_TOK, K_FF, q8, s8), "reencode")
    run_t = lambda: fq._check(fq.fp4_mxfp4_to_fp8_transpose(mx.q, sf, M_TOK, K_FF, q8t, s8t),
                              "reencode_t")
    run()
    run_t()
    nbytes = M_TOK * K_FF * (0.5 + 1 / 32 + 1 + 4 / 128)
    out = {"shape": [M_TOK, K_FF], "bytes_per_launch": int(nbytes), "bound": "hbm"}
    for key, fn in (("row", run), ("transposed", run_t)):
        ms = graph_ms(fn, flush)
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[key] = {"ms": round(ms, 4), "gbs": round(gbs, 1), "frac": round(gbs / hbm_gbs, 4)}
    return out


def run_linear(layer, flush, steps=10):
    """FP4Linear (the autograd layer over the same entry points) on the same
    shapes: forward + backward of one step, eager, with the amax caches on a
    hold step (D = 50) and on a refresh step."""
    from fp4_block_scaled_quantize_gb300.linear import FP4Linear
    dev = layer.X.device
    lin = FP4Linear(K_FF, N_MODEL, D=50, format=layer.fmt, device=dev)
    with torch.no_grad():
        lin.weight.copy_(layer.W)
    x = layer.X.detach().clone().requires_grad_(True)
    dy = layer.dY

    def one():
        x.grad = None
        lin.weight.grad = None
        lin(x).backward(dy)

    one()                      # step 0: refresh
    lin.next_step()
    one()
    torch.cuda.synchronize()
    out = {}
    for name, step in (("hold_step_ms", 1), ("refresh_step_ms", 50)):
        tot = 0.0
        for _ in range(steps):
            lin.step = step
            flush_l2(flush)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record()
            one()
            b.record()
            torch.cuda.synchronize()
            tot += a.elapsed_time(b)
        out[name] = round(tot / steps, 4)
    layer.fq._check(layer.fq.fp4_status_sync(), "linear")
    out["shape"] = "x [%d, %d], W [%d, %d]" % (M_TOK, K_FF, N_MODEL, K_FF)
    out["launch"] = "eager autograd (Python dispatch included)"
    return out


def run_e2e(layer, args, world, ideal, graph=None):
    """Same step with host inputs and outputs: every step copies X, W, dY from
    pinned host memory and reads Y, dX, dW back into pinned host memory, all
    inside the timed region.  Two device buffer sets alternate so that step
    i's uploads, step i-1's compute and step i-2's downloads overlap (copy
    streams for each direction, events for the hand-offs)."""
    fq = layer.fq
    dev = layer.X.device
    sets = [layer, Layer(layer.fmt, 0, dev, host=layer.host)]
    graphs = [graph, None]
    if graph is not None:
        torch.cuda.synchronize()
        sets[1].step()
        torch.cuda.synchronize()
        graphs[1] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graphs[1]):
            sets[1].step()
    host_out = [{k: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                 for k, t in (("Y", L.Y), ("dX", L.dX), ("dW", L.dW))} for L in sets]
    h2d = sum(t.numel() * t.element_size() for t in layer.host.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    steps = max(2, min(args.steps, 60))  # amortises the pipeline's fill and drain
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    inputs_free = [ev(), ev()]   # compute on this set finished reading its inputs
    outputs_free = [ev(), ev()]  # downloads from this set finished
    for e_ in inputs_free + outputs_free:
        e_.record(comp)
    torch.cuda.synchronize()
    barrier(world)
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(comp)
    s_in.wait_event(s)
    s_out.wait_event(s)
    for i in range(steps):
        L, out, b = sets[i % 2], host_out[i % 2], i % 2
        landed, computed = ev(), ev()
        with torch.cuda.stream(s_in):
            s_in.wait_event(inputs_free[b])
            L.X.copy_(L.host["X"], non_blocking=True)
            L.W.copy_(L.host["W"], non_blocking=True)
            L.dY.copy_(L.host["dY"], non_blocking=True)
            landed.record(s_in)
        comp.wait_event(landed)
        comp.wait_event(outputs_free[b])
        if graphs[b] is not None:
            graphs[b].replay()
        else:
            L.step()
        computed.record(comp)
        inputs_free[b] = computed
        with torch.cuda.stream(s_out):
            s_out.wait_event(computed)
            out["Y"].copy_(L.Y, non_blocking=True)
            out["dX"].copy_(L.dX, non_blocking=True)
            out["dW"].copy_(L.dW, non_blocking=True)
            done = ev()
            done.record(s_out)
            outputs_free[b] = done
    comp.wait_stream(s_in)
    comp.wait_stream(s_out)
    e.record(comp)
    torch.cuda.synchronize()
    ms = reduce_max(s.elapsed_time(e) / steps, world)
    fq._check(fq.fp4_status_sync(), "e2e")
    return {"value": round(100.0 * ideal / (ms * 1e-3) * world, 3),
            "unit": UNIT, "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "overlap": "uploads, compute and downloads of consecutive steps overlap "
                       "(two device buffer sets, one copy stream per direction)"}


def gemm_source_digest():
    """Short digest of the GEMM kernel source: a traffic figure measured on
    another version of the kernel is stale."""
    import hashlib
    h = hashlib.sha256()
    for name in ("gemm.cu", "gemm2.cu", "tcgen05.cuh", "qout.cuh"):
        with open(os.path.join(ROOT, "fp4_block_scaled_quantize_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(kernel):
    """DRAM read+write bytes per launch of one GEMM direction from the
    committed ncu summary (its `traffic_per_launch` line), or None when the
    summary is absent or was taken on another version of the kernel."""
    import re
    path = os.path.join(ROOT, "profiles", "k_gemm_down_proj_8b_ue5m3.md")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            if line.startswith("traffic_per_launch"):
                fields = dict(re.findall(r"(\w+)=(\w+)", line))
                if fields.get("source") != gemm_source_digest() or kernel not in fields:
                    return None
                return int(fields[kernel])
    return None


# ------------------------------------------------------------ CPU oracle arm

def oracle_step_seconds(args, sample_rows=64, sample_outputs=24, threads=None):
    """Time the oracle on a bounded sample of one step and extrapolate.
    Returns (seconds per full step, threads used, description)."""
    import numpy as np

    import oracle as orc
    from fp4_block_scaled_quantize_gb300 import inputs
    fmt = {0: orc.UE5M3, 1: orc.NVFP4, 2: orc.MXFP4, 3: orc.UE5M3_B32}[args.format]
    R = sample_rows
    g = inputs.down_proj_8b(seed=args.seed, M=R * 2, K=K_FF, N=N_MODEL)
    threads = threads or min(16, os.cpu_count() or 1)
    t_quant = 0.0
    elems_done = 0
    for name, x in (("X", g["X"][:R]), ("W", g["W"][:R]), ("dY", g["dY"][:R])):
        x32 = x.float().numpy()
        t0 = time.perf_counter()
        a = orc.amax(x32)
        orc.quantize_transpose(x32, a, a, fmt, block2d=(name == "W"), sr_row=(name == "dY"),
                               sr_col=(name == "dY"), seed=42, threads=threads)
        t_quant += time.perf_counter() - t0
        elems_done += x32.size
    total_elems = M_TOK * K_FF + N_MODEL * K_FF + M_TOK * N_MODEL
    quant_s = t_quant / elems_done * total_elems
    gemm_s = 0.0
    gemm_desc = []
    for name, (M, N, K) in (("fprop", (M_TOK, N_MODEL, K_FF)), ("dgrad", (M_TOK, K_FF, N_MODEL)),
                            ("wgrad", (N_MODEL, K_FF, M_TOK))):
        rng = np.random.default_rng(1)
        a = orc.quantize(rng.standard_normal((4, K)).astype(np.float32), 4.0, fmt)
        b = orc.quantize(rng.standard_normal((4, K)).astype(np.float32), 4.0, fmt)
        mi = np.arange(sample_outputs) % 4
        ni = (np.arange(sample_outputs) // 4) % 4
        t0 = time.perf_counter()
        orc.gemm_model(a["q"], a["sf"], b["q"], b["sf"], fmt, K, a["s_dec"], b["s_dec"], mi, ni,
                       threads=threads)
        dt = time.perf_counter() - t0
        gemm_s += dt / sample_outputs * M * N
        gemm_desc.append(f"{name} {sample_outputs} outputs")
    desc = (f"amax+producers on {R} rows of each of X, W, dY; probe-matched GEMM model on "
            + ", ".join(gemm_desc) + "; extrapolated to the full step")
    return quant_s + gemm_s, threads, desc


def cpu_baseline(args, ideal):
    """The oracle on all host cores (up to 16 threads) and on one thread."""
    secs, threads, desc = oracle_step_seconds(args, sample_rows=256, sample_outputs=128)
    secs1, _, _ = oracle_step_seconds(args, sample_rows=32, sample_outputs=16, threads=1)
    return {"value": 100.0 * ideal / secs, "unit": UNIT, "cores": threads,
            "kind": "oracle", "sample": desc, "seconds_per_step_extrapolated": round(secs, 1),
            "host_cpus": os.cpu_count(),
            "single_thread": {"value": 100.0 * ideal / secs1, "cores": 1,
                              "seconds_per_step_extrapolated": round(secs1, 1),
                              "sample": "32 rows of each producer, 16 outputs per GEMM"}}


def run_reference(args, world, rank):
    if rank != 0:
        return
    pk = peaks()
    amax_b, qbytes, gemms, flops = work_model(args.format)
    ideal = (amax_b / (pk["hbm_gbs"] * 1e9) + sum(qbytes.values()) / (pk["hbm_gbs"] * 1e9)
             + sum(flops.values()) / (pk["bf16_tflops"] * FP4_OVER_BF16 * 1e12))
    for _ in range(args.warmup):
        oracle_step_seconds(args, sample_rows=32, sample_outputs=4)
    # each step is a bounded sample; the whole run stays within a time budget
    times, t_start = [], time.time()
    for _ in range(args.steps):
        s, threads, desc = oracle_step_seconds(args, sample_rows=32, sample_outputs=8)
        times.append(s)
        if time.time() - t_start > 90.0:
            break
    secs = statistics.median(times)
    value = 100.0 * ideal / secs
    out = {"impl": "reference",
           "metric": "quantize GB/s and FP4 block-scaled GEMM TFLOP/s, each as % of GB300 roofline",
           "value": value, "unit": UNIT, "n_gpus": world,
           "steps": len(times), "steps_requested": args.steps, "warmup": args.warmup,
           "ms_per_step": secs * 1e3, "ms_per_step_extrapolated": True,
           "timing": "each step times the oracle on a bounded sample of the step (rows of each "
                     "producer, sampled GEMM outputs) and extrapolates to the full step; median "
                     "over steps",
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "e2m1 payload x exact accumulate (u8 codes)", "data": "synthetic",
           "config": {"workload": WORKLOAD, "format": FMT_NAMES[args.format],
                      "X": [M_TOK, K_FF], "W": [N_MODEL, K_FF], "dY": [M_TOK, N_MODEL]},
           "cpu_baseline": {"value": value, "unit": UNIT, "kind": "oracle",
                            "cores": threads, "sample": desc},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def run_profile(args, local):
    """Set up the step's buffers, then launch one kernel kind three times
    (the workload of an ncu capture; prints nothing else)."""
    torch.cuda.set_device(local)
    layer = Layer(args.format, seed=args.seed, device=torch.device("cuda", local))
    fq = layer.fq
    ops = {
        "amax": layer.refresh_amax,
        "quant_X": lambda: layer._qt(layer.X, "X", layer.px, layer.xr, layer.xc),
        "quant_W": lambda: layer._qt(layer.W, "W", layer.pw, layer.wr, layer.wc),
        "quant_dY": lambda: layer._qt(layer.dY, "dY", layer.pdy, layer.dyr, layer.dyc),
        "fprop": lambda: fq.gemm(layer.xr, layer.wr, out=layer.Y),
        "dgrad": lambda: fq.gemm(layer.dyr, layer.wc, out=layer.dX),
        "wgrad": lambda: fq.gemm(layer.dyc, layer.xc, out=layer.dW),
    }
    if args.profile == "amax_stripes":
        ar = torch.empty(fq.n_stripes(M_TOK), dtype=torch.float32, device=layer.X.device)
        ac = torch.empty(fq.n_stripes(K_FF), dtype=torch.float32, device=layer.X.device)
        ops["amax_stripes"] = lambda: fq._check(fq.fp4_amax_stripes(layer.X, ar, ac), "stripes")
    if args.profile.startswith("fp8_"):
        # the step's operands as FP8 copies (MXFP4-b32 re-encoded), one GEMM
        p = fq.params(format=fq.FP4_FMT_MXFP4_B32, sf_layout=fq.FP4_SF_PLAIN)
        f8 = {}
        for name, x in (("X", layer.X), ("W", layer.W), ("dY", layer.dY)):
            c = fq.quantize(x, layer.amax[name][0], p)
            sf = c.sf.view(x.shape[0], x.shape[1] // 32)
            f8[name] = fq.mxfp4_to_fp8(c.q, sf)
            f8[name + "t"] = fq.mxfp4_to_fp8_transpose(c.q, sf)
        a, b, dt = {"fp8_fprop": ("X", "W", torch.bfloat16), "fp8_dgrad": ("dY", "Wt", torch.bfloat16),
                    "fp8_wgrad": ("dYt", "Xt", torch.float32)}[args.profile]
        D = torch.empty((f8[a][0].shape[0], f8[b][0].shape[0]), dtype=dt, device=layer.X.device)
        ops[args.profile] = lambda: fq.fp8_gemm(*f8[a], *f8[b], out=D)
    if args.profile in ("reencode", "reencode_t"):
        p = fq.params(format=fq.FP4_FMT_MXFP4_B32, sf_layout=fq.FP4_SF_PLAIN)
        mx = fq.quantize(layer.X, layer.amax["X"][0], p)
        sf = mx.sf.view(M_TOK, K_FF // 32)
        q8 = torch.empty((M_TOK, K_FF), dtype=torch.uint8, device=layer.X.device)
        s8 = torch.empty((M_TOK, K_FF // 128), dtype=torch.float32, device=layer.X.device)
        ops["reencode"] = lambda: fq._check(fq.fp4_mxfp4_to_fp8(mx.q, sf, M_TOK, K_FF, q8, s8),
                                            "reencode")
        q8t = torch.empty((K_FF, M_TOK), dtype=torch.uint8, device=layer.X.device)
        s8t = torch.empty((K_FF, M_TOK // 128), dtype=torch.float32, device=layer.X.device)
        ops["reencode_t"] = lambda: fq._check(
            fq.fp4_mxfp4_to_fp8_transpose(mx.q, sf, M_TOK, K_FF, q8t, s8t), "reencode_t")
    if args.profile in ("dequantize", "gemm_bf16"):
        p = fq.params(format=fq.FP4_FMT_UE5M3_B16, sf_layout=fq.FP4_SF_PLAIN)
        cx = fq.quantize(layer.X, layer.amax["X"][0], p)
        cw = fq.quantize(layer.W, layer.amax["W"][0], p)
        yx, yw = fq.dequantize(cx), fq.dequantize(cw)
        ops["dequantize"] = lambda: fq._check(
            fq.fp4_dequantize(cx.q, cx.sf, cx.format, M_TOK, K_FF, yx), "dequantize")
        ops["gemm_bf16"] = lambda: fq.gemm_bf16(yx, yw, cx.s_dec, cw.s_dec, out=layer.Y)
    torch.cuda.synchronize()
    for _ in range(3):
        ops[args.profile]()
    torch.cuda.synchronize()
    fq._check(fq.fp4_status_sync(), "profile")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--format", type=int, default=0, choices=[0, 1, 2, 3])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the timed steps kernel by kernel instead of as a CUDA graph")
    ap.add_argument("--profile", default=None,
                    choices=["amax", "quant_X", "quant_W", "quant_dY", "fprop", "dgrad", "wgrad",
                             "reencode", "reencode_t", "fp8_fprop", "fp8_dgrad", "fp8_wgrad",
                             "amax_stripes", "dequantize", "gemm_bf16"],
                    help="run only this kernel (3 launches after set-up) for an ncu capture")
    args = ap.parse_args()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one process per GPU: relaunch this command under torchrun
        port = os.environ.get("MASTER_PORT", "29500")
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
               f"--nproc-per-node={args.gpus}", "--master-addr=127.0.0.1",
               f"--master-port={port}", os.path.abspath(__file__)] + sys.argv[1:]
        sys.exit(subprocess.call(cmd))
    world, rank, local = dist_init()
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    if args.profile:
        run_profile(args, local)
    elif args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_gpu(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
