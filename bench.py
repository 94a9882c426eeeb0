"""Benchmark of the FP8 linear-layer hot path on GB300.

One step = one forward + backward pass of an MXFP8 transformer MLP block (8192 tokens,
hidden 4096, ffn 16384), everything through the library's C ABI:
    quantize X, W1, W2 (row + column copies, one grouped launch) -> fc1 GEMM whose epilogue
    applies GeLU, keeps its input h in FP8 and writes the MXFP8 copies of the activation ->
    fc2 GEMM -> quantize dY -> fc2 dgrad (epilogue: dGeLU and the MXFP8 copies of dh) + fc2
    wgrad -> fc1 dgrad + wgrad.
`--unfused` runs the same step with the GEMMs storing h and da in bf16 and the standalone
GeLU / dGeLU quantize kernels in between.
Metric: GEMM TFLOP/s of the whole step (quantize time included), plus the quantize kernels'
algorithmic HBM GB/s. Inputs are seeded synthetic bf16 tensors resident in HBM (about 2 GB
touched per step, far above the 129 MB L2). `e2e` repeats the step with the inputs copied
from pinned host memory and every result (y, dX, dW1, dW2) copied back inside the timed region,
uploads and downloads on their own streams overlapping the neighbouring steps' compute.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload mlp|mxfp8_fprop|blockwise_fwd_bwd|delayed_step|tensorwise_256]

`--workload` times one of the smaller configurations instead (MXFP8 quantize + fprop;
blockwise quantize + fprop, dgrad and wgrad at 4096^3; a delayed-scaling step with its amax
history; a 256^3 tensorwise step replayed as a CUDA graph), with the same JSON contract.

`--impl reference` times the CPU oracle (a deliberately slow, plain implementation) on a
bounded sample of the same workload and reports the same metric.
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

import numpy as np  # noqa: E402

METRIC = "FP8 linear fwd+bwd TFLOPS (incl. quantize) vs FP8 peak; quantize HBM GB/s"
TOKENS, HIDDEN, FFN = 8192, 4096, 16384
GEMM_FLOPS = 6 * 2.0 * TOKENS * HIDDEN * FFN          # fc1, fc2 fwd; dgrad + wgrad of both
WORKLOAD = "mxfp8_mlp_fwd_bwd tokens=8192 hidden=4096 ffn=16384"
KERNELS_PER_STEP = 8                                  # 2 quantize, 6 GEMMs (2 fused)
KERNELS_PER_STEP_UNFUSED = 10                         # plus standalone gelu and dgelu
E2E_SETS = 3                                          # buffer sets the end-to-end leg rotates
DELAYED_STEPS = 64                                    # distinct inputs of the delayed-scaling config
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP8_OVER_BF16 = 2.0                                   # nominal dense fp8 / bf16 rate
# DRAM bytes (read + write) per launch of the plain-store MXFP8 GEMM: the average over the
# step's four such launches in one capture of `ncu --metrics dram__bytes_read.sum,
# dram__bytes_write.sum,gpu__time_duration.sum --clock-control none -k regex:gemm_tn_kernel
# -s 4 -c 4 python bench.py --profile gemm_mx_mlp --steps 2` (480.0, 340.9, 476.4 and 345.6
# MB for fc2 fprop, fc2 wgrad, fc1 dgrad and fc1 wgrad). Reset to None whenever that kernel
# changes.
GEMM_TRAFFIC_BYTES = 410.7e6


def peaks():
    """(hbm GB/s, fp8 TFLOP/s, source). Measured peaks if the file exists, else fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        hbm = float(d.get("hbm_gbs"))
        bf16 = float(d.get("bf16_tflops"))
        return hbm, bf16 * FP8_OVER_BF16, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS * FP8_OVER_BF16, "fallback"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle samples every 50 ms while the timed region runs. start()
    returns once the first sample has arrived (nvidia-smi takes a while to start), and only
    the samples taken after that count."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.mark = 0

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
            return
        t_end = time.monotonic() + 5.0
        while not self.lines and time.monotonic() < t_end and self.proc.poll() is None:
            time.sleep(0.01)
        self.mark = len(self.lines)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines[self.mark:]:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- GPU step

class MlpStep:
    """Preallocated device buffers and the step itself (device-resident inputs)."""

    def __init__(self, torch, F, dev, fused=True):
        self.torch, self.F, self.dev, self.fused = torch, F, dev, fused
        from workloads import bf16_bits_normal
        self.rec = F.Recipe(kind="mxfp8")
        M, H, Fd = TOKENS, HIDDEN, FFN
        host = {
            "x": bf16_bits_normal(M, H, seed=0, stream=0),
            "w1": bf16_bits_normal(Fd, H, seed=0, stream=1, sigma=0.02),
            "w2": bf16_bits_normal(H, Fd, seed=0, stream=3, sigma=0.02),
            "dy": bf16_bits_normal(M, H, seed=0, stream=2, sigma=1e-3),
        }
        # pinned host copies (for the end-to-end leg) and device copies
        self.h = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).pin_memory()
                  for k, v in host.items()}
        self.d = {k: v.to(dev) for k, v in self.h.items()}
        e = F.empty_qtensor
        self.xq = e(self.rec, M, H, "activation", device=dev)
        self.w1q = e(self.rec, Fd, H, "weight", device=dev)
        self.w2q = e(self.rec, H, Fd, "weight", device=dev)
        self.dyq = e(self.rec, M, H, "grad", device=dev)
        self.aq = e(self.rec, M, Fd, "activation", device=dev)
        self.hq = e(self.rec, M, Fd, "activation", want_col=False, device=dev)
        self.dhq = e(self.rec, M, Fd, "grad", device=dev)
        bf = torch.bfloat16
        if not fused:
            self.hbuf = torch.empty((M, Fd), dtype=bf, device=dev)
            self.da = torch.empty((M, Fd), dtype=bf, device=dev)
        shapes = {"y": (M, H), "dx": (M, H), "dw1": (Fd, H), "dw2": (H, Fd)}
        # E2E_SETS sets of device inputs / outputs and pinned host outputs, so the end-to-end
        # leg can copy the data of the steps around the one that computes
        self.out_sets = [{k: torch.empty(v, dtype=bf, device=dev) for k, v in shapes.items()}
                         for _ in range(E2E_SETS)]
        self.outs = self.out_sets[0]
        self.d_sets = [self.d] + [{k: torch.empty_like(v) for k, v in self.d.items()}
                                  for _ in range(E2E_SETS - 1)]
        self.h_out = [{k: torch.empty(v, dtype=bf).pin_memory() for k, v in shapes.items()}
                      for _ in range(E2E_SETS)]
        # algorithmic bytes of the quantize kernels per step
        mx = lambda r, c, copies: r * c * (2 + copies + copies / 32.0)  # noqa: E731
        self.quant_bytes = mx(M, H, 2) + mx(Fd, H, 2) + mx(H, Fd, 2) + mx(M, H, 2)
        if not fused:
            self.quant_bytes += (M * Fd * (2 + 3 + 3 / 32.0)                # gelu: h in, a x2 + h
                                 + M * Fd * (2 + 1 + 1 / 32.0 + 2 + 2 / 32.0))  # dgelu
        self.kernels_per_step = KERNELS_PER_STEP if fused else KERNELS_PER_STEP_UNFUSED
        self.stream = torch.cuda.current_stream(dev)
        self.events = []

    def _timed(self, kind, fn, name):
        if self.events is None:
            return fn()
        s = self.torch.cuda.Event(enable_timing=True)
        e = self.torch.cuda.Event(enable_timing=True)
        s.record(self.stream)
        r = fn()
        e.record(self.stream)
        self.events.append((kind, name, s, e))
        return r

    def run(self, src=None, outs=None):
        F, rec, T = self.F, self.rec, self._timed
        d = src or self.d
        o = outs or self.outs
        # X, W1 and W2 in one launch (fp8_quantize_group)
        T("quant", lambda: F.quantize_group(rec, [d["x"], d["w1"], d["w2"]],
                                            ["activation", "weight", "weight"],
                                            outs=[self.xq, self.w1q, self.w2q]), "quantize_x_w1_w2")
        if self.fused:
            T("gemm_fused", lambda: F.linear_fwd_gelu(rec, self.xq, self.w1q, a_q=self.aq,
                                                      h_q=self.hq), "fc1_fprop_gelu")
        else:
            T("gemm", lambda: F.linear_fwd(rec, self.xq, self.w1q, y=self.hbuf), "fc1_fprop")
            T("quant", lambda: F.gelu_quantize(rec, self.hbuf, a_q=self.aq, h_q=self.hq),
              "gelu_quantize")
        T("gemm", lambda: F.linear_fwd(rec, self.aq, self.w2q, y=o["y"]), "fc2_fprop")
        T("quant", lambda: F.quantize(rec, d["dy"], "grad", out=self.dyq), "quantize_dy")
        if self.fused:
            T("gemm_fused", lambda: F.linear_dgrad_dgelu(rec, self.dyq, self.w2q, self.hq,
                                                         dh_q=self.dhq), "fc2_dgrad_dgelu")
        else:
            T("gemm", lambda: F.linear_bwd(rec, self.dyq, self.aq, self.w2q, want_dw=False,
                                           dx=self.da), "fc2_dgrad")
        T("gemm", lambda: F.linear_bwd(rec, self.dyq, self.aq, self.w2q, want_dx=False,
                                       dw=o["dw2"]), "fc2_wgrad")
        if not self.fused:
            T("quant", lambda: F.dgelu_quantize(rec, self.da, self.hq, dh_q=self.dhq),
              "dgelu_quantize")
        T("gemm", lambda: F.linear_bwd(rec, self.dhq, self.xq, self.w1q, want_dw=False,
                                       dx=o["dx"]), "fc1_dgrad")
        T("gemm", lambda: F.linear_bwd(rec, self.dhq, self.xq, self.w1q, want_dx=False,
                                       dw=o["dw1"]), "fc1_wgrad")

    def run_e2e(self, steps):
        """`steps` steps whose inputs are copied from pinned host memory and whose results
        (y, dX, dW1, dW2) are copied back to pinned host memory, pipelined the way a training
        loop overlaps its data movement: step i's inputs are uploaded on one stream while the
        steps before it compute, and its results are downloaded on a third stream while the
        steps after it compute (E2E_SETS buffer sets rotate, so a copy has more than one step's
        compute to hide behind). Returns the elapsed ms from the first upload to the last
        download, measured on the compute stream."""
        torch = self.torch
        comp = self.stream
        s_in, s_out = torch.cuda.Stream(self.dev), torch.cuda.Stream(self.dev)
        ev_in = [torch.cuda.Event() for _ in range(E2E_SETS)]
        ev_comp = [torch.cuda.Event() for _ in range(E2E_SETS)]
        ev_out = [torch.cuda.Event() for _ in range(E2E_SETS)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(comp)
        s_in.wait_stream(comp)
        s_out.wait_stream(comp)
        for i in range(steps):
            b = i % E2E_SETS
            if i >= E2E_SETS:
                s_in.wait_event(ev_comp[b])               # the set's last step is done with them
            with torch.cuda.stream(s_in):
                for k, v in self.h.items():
                    self.d_sets[b][k].copy_(v, non_blocking=True)
                ev_in[b].record(s_in)
            comp.wait_event(ev_in[b])
            if i >= E2E_SETS:
                comp.wait_event(ev_out[b])                # the set's last results are downloaded
            with torch.cuda.stream(comp):
                self.run(self.d_sets[b], self.out_sets[b])
                ev_comp[b].record(comp)
            s_out.wait_event(ev_comp[b])
            with torch.cuda.stream(s_out):
                for k, v in self.out_sets[b].items():
                    self.h_out[b][k].copy_(v, non_blocking=True)
                ev_out[b].record(s_out)
        comp.wait_stream(s_in)
        comp.wait_stream(s_out)
        t1.record(comp)
        t1.synchronize()
        return t0.elapsed_time(t1)

    def h2d_bytes(self):
        return sum(v.numel() * 2 for v in self.h.values())

    def d2h_bytes(self):
        return sum(v.numel() * 2 for v in self.outs.values())

    def kernel_stats(self):
        """Per-kind lists of launch times (ms) and the mean time of each named launch."""
        ms = {"gemm": [], "gemm_fused": [], "quant": []}
        by_name = {}
        for kind, name, s, e in self.events:
            t = s.elapsed_time(e)
            ms[kind].append(t)
            by_name.setdefault(name, []).append(t)
        return ms, {k: round(statistics.mean(v), 4) for k, v in by_name.items()}


def max_over_ranks(value, dist=None, device=None):
    """The slowest rank's figure (timings are taken as the max over ranks)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world, ms_total, steps):
    """All ranks' GEMM flops (each rank runs its own replica step) over the slowest time."""
    return world * GEMM_FLOPS / (ms_total / steps * 1e-3) / 1e12


def _event_ms(torch, stream, fn, reps, warm=5):
    """Mean device time (ms) of fn over `reps` back-to-back calls on `stream` (CUDA events,
    after `warm` untimed calls)."""
    for _ in range(warm):
        fn(0)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for i in range(reps):
        fn(i)
    e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) / reps


def measure_gemm_4096(torch, F, dev, fp8_peak, reps=30):
    """The MXFP8 GEMM 4096 x 4096 x 4096 alone (fprop of seeded X N(0,1), W N(0,0.02)): mean of
    `reps` back-to-back launches timed with CUDA events."""
    from workloads import bf16_bits_normal
    rec = F.Recipe(kind="mxfp8")
    n = 4096
    to_dev = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(dev)  # noqa: E731
    xq = F.quantize(rec, to_dev(bf16_bits_normal(n, n, seed=0, stream=0)), "activation")
    wq = F.quantize(rec, to_dev(bf16_bits_normal(n, n, seed=0, stream=1, sigma=0.02)), "weight")
    y = torch.empty((n, n), dtype=torch.bfloat16, device=dev)
    ms = _event_ms(torch, torch.cuda.current_stream(dev),
                   lambda i: F.linear_fwd(rec, xq, wq, y=y), reps)
    tf = 2.0 * n ** 3 / (ms * 1e-3) / 1e12
    return {"kernel": "gemm_tn_kernel<G_MX> (CTA pair)", "M": n, "N": n, "K": n,
            "launches": reps, "avg_launch_ms": round(ms, 4), "tflops": round(tf, 1),
            "peak": fp8_peak, "frac": round(tf / fp8_peak, 4), "target_frac": 0.60,
            "operands": "16 MB FP8 each, L2-resident across launches (compute-bound)"}


def measure_quantize_by_recipe(torch, F, dev, hbm, reps=20):
    """Every recipe's quantize of an 8192 x 4096 tensor (row + column copies) alone: mean of
    `reps` launches, the input rotating over enough distinct buffers (> 2 x L2) that each
    launch reads it from DRAM. GB/s are algorithmic bytes (bf16 or fp32 read, one byte per
    code written, the scales) over the CUDA-event time."""
    R, C = 8192, 4096
    n_in = 5                                             # 5 x 64 MiB bf16 > 2 x 129 MB L2
    g = torch.Generator(device=dev).manual_seed(0)
    xs = [torch.randn((R, C), device=dev, generator=g).to(torch.bfloat16) for _ in range(n_in)]
    stream = torch.cuda.current_stream(dev)
    cases = [("tensorwise", "activation", 4.0), ("delayed", "activation", 4.0),
             ("mxfp8", "activation", 4.0 + 2 / 32.0),
             ("blockwise_1x128", "activation", 4.0 + 2 * 4 / 128.0),
             ("blockwise_128x128", "weight", 4.0 + 2 * 4 / (128.0 * 128.0))]
    out = {}
    for name, role, per_elt in cases:
        rec = F.Recipe(kind=name.split("_")[0])
        q = F.empty_qtensor(rec, R, C, role, device=dev)
        ws = torch.empty(max(16, F.workspace_bytes(rec, R, C)), dtype=torch.uint8, device=dev)
        ms = _event_ms(torch, stream,
                       lambda i: F.quantize(rec, xs[i % n_in], role, out=q, workspace=ws), reps)
        gbs = R * C * per_elt / (ms * 1e-3) / 1e9
        out[name] = {"ms": round(ms, 4), "gbs": round(gbs, 1), "frac": round(gbs / hbm, 4),
                     "bytes_per_elt": round(per_elt, 5)}
    del xs
    # fp32 master weight -> MXFP8 row + column copies: 4 B in, 2 x (1 + 1/32) B out
    w32 = [torch.randn((R, C), device=dev, generator=g) * 0.02 for _ in range(3)]  # 3 x 128 MiB
    rec = F.Recipe(kind="mxfp8")
    q = F.empty_qtensor(rec, R, C, "weight", device=dev)
    ms = _event_ms(torch, stream, lambda i: F.quantize_master(rec, w32[i % 3], out=q), reps)
    per_elt = 4.0 + 2 + 2 / 32.0
    gbs = R * C * per_elt / (ms * 1e-3) / 1e9
    out["master_mxfp8"] = {"ms": round(ms, 4), "gbs": round(gbs, 1), "frac": round(gbs / hbm, 4),
                           "bytes_per_elt": per_elt}
    return {"shape": [R, C], "copies": "row + column", "launches": reps, "peak_gbs": hbm,
            "target_frac": 0.70, "recipes": out}


def measure_sustained(torch, st, ms_step, local, seconds=3.0):
    """The step back to back for about `seconds` (long enough to reach the power cap), with its
    own clock samples: the figure a long training run sees, next to the short timed region."""
    n = max(10, int(seconds * 1e3 / max(ms_step, 1e-3)))
    st.events = None
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(st.stream)
    for _ in range(n):
        st.run()
    t1.record(st.stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1)
    return {"steps": n, "seconds": round(ms / 1e3, 2), "ms_per_step": round(ms / n, 4),
            "tflops": round(GEMM_FLOPS / (ms / n * 1e-3) / 1e12, 1), "clocks": clk}


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from scaled_quantize_fp8_gb300 import build as B
    B.build()
    import scaled_quantize_fp8_gb300 as F

    st = MlpStep(torch, F, dev, fused=not args.unfused)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # ---- device-resident leg: the step back to back with nothing between its kernels (an
    # event between two kernels would stop the next one's prologue from overlapping the
    # previous one's tail)
    st.events = None
    for _ in range(args.warmup):
        st.run()
    barrier()
    clocks = ClockSampler(local)
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(st.stream)
    for _ in range(args.steps):
        st.run()
    t1.record(st.stream)
    barrier()
    clk = clocks.stop()
    ms_total = max_over_ranks(t0.elapsed_time(t1), dist if world > 1 else None, dev)
    # ---- per-kernel times (roofline, kernels_ms): further steps with an event pair around
    # every launch, on the same stream
    st.events = []
    for _ in range(max(1, min(args.steps, 20))):
        st.run()
    barrier()
    ks, per_kernel = st.kernel_stats()

    # ---- end-to-end leg (host buffers, copies inside the timed region)
    st.events = None
    st.run_e2e(max(2, args.warmup))
    barrier()
    ms_e2e = max_over_ranks(st.run_e2e(args.steps), dist if world > 1 else None, dev)
    barrier()

    ms_step = ms_total / args.steps
    hbm, fp8_peak, src = peaks()
    # ---- the two named performance targets (4096^3 MXFP8 GEMM, quantize bandwidth per
    # recipe) and the power-capped figure, measured apart from the timed region above
    gemm4096 = measure_gemm_4096(torch, F, dev, fp8_peak)
    quant_recipes = measure_quantize_by_recipe(torch, F, dev, hbm)
    sustained = measure_sustained(torch, st, ms_step, local)
    barrier()
    value = whole_job_tflops(world, ms_total, args.steps)
    e2e_value = whole_job_tflops(world, ms_e2e, args.steps)
    # the roofline kernel: the plain-store MXFP8 GEMM (four of the six GEMM launches when the
    # MLP epilogues are fused, all six otherwise); every GEMM of the step has the same flops
    gemm_ms = statistics.mean(ks["gemm"])
    gemm_flops_launch = GEMM_FLOPS / 6
    achieved = gemm_flops_launch / (gemm_ms * 1e-3) / 1e12
    fused_ms = statistics.mean(ks["gemm_fused"]) if ks["gemm_fused"] else None
    quant_ms_step = sum(ks["quant"]) / max(1, min(args.steps, 20))
    quant_gbs = st.quant_bytes / (quant_ms_step * 1e-3) / 1e9

    if rank == 0:
        cpu = cpu_baseline()
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 (fp32 accumulate)", "data": "synthetic",
            "config": {"workload": WORKLOAD, "recipe": "mxfp8",
                       "mlp_epilogues": "fused" if st.fused else "unfused",
                       "parallelism": "replicas" if world > 1 else "single",
                       "l2": "inputs larger than L2 (~2 GB touched per step)",
                       "gemm_flops_per_step": GEMM_FLOPS},
            "roofline": {"bound": "tensor", "kernel": "gemm_tn_kernel<G_MX> (bf16 store)",
                         "achieved": round(achieved, 1), "peak": fp8_peak, "unit": "TFLOP/s",
                         "frac": round(achieved / fp8_peak, 4),
                         "traffic": GEMM_TRAFFIC_BYTES if st.fused else None,
                         "traffic_source": "ncu dram bytes read + write per launch"
                         if GEMM_TRAFFIC_BYTES else "not captured for this kernel version",
                         "peak_source": f"{src}: bf16 x {FP8_OVER_BF16} (nominal fp8/bf16)",
                         "avg_launch_ms": round(gemm_ms, 4)},
            "fused_gemm": None if fused_ms is None else {
                "kernel": "gemm_mlp_kernel (GeLU / dGeLU + MXFP8 epilogue)",
                "avg_launch_ms": round(fused_ms, 4),
                "tflops": round(gemm_flops_launch / (fused_ms * 1e-3) / 1e12, 1)},
            "quantize": {"gbs": round(quant_gbs, 1), "peak_gbs": hbm,
                         "frac": round(quant_gbs / hbm, 4), "ms_per_step": round(quant_ms_step, 4),
                         "algorithmic_bytes_per_step": st.quant_bytes, "peak_source": src},
            "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": st.h2d_bytes(), "d2h_bytes_per_step": st.d2h_bytes(),
                    "copies": "pinned host, own streams, overlapped with the neighbouring "
                              f"steps ({E2E_SETS} buffer sets)"},
            "kernels_ms": per_kernel,
            "gemm_4096_mxfp8": gemm4096,
            "quantize_by_recipe": quant_recipes,
            "sustained": sustained,
            "gpu_launches": st.kernels_per_step * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- other configs

CONFIGS = {
    "tensorwise_256": "tensorwise quantize X, W 256x256 (N(0,1)) + fprop 256^3, one CUDA graph "
                      "a step",
    "mxfp8_fprop": "mxfp8 quantize X 8192x4096 (0.1% outliers x50) + W 4096x4096 + fprop",
    "blockwise_fwd_bwd": "blockwise quantize X, W (one grouped launch), dY 4096x4096 + fprop + "
                         "dgrad + wgrad",
    "delayed_step": "delayed quantize X_t 8192x4096 (log-uniform sigma) + fprop (W 4096x4096) "
                    "+ amax history update (length 1024)",
}


class ConfigStep:
    """One step of a smaller configuration of the layer (device-resident buffers)."""

    def __init__(self, torch, F, dev, name):
        from workloads import STREAM_STEP0, bf16_bits_normal, sigma_schedule
        self.torch, self.F, self.dev, self.name = torch, F, dev, name
        bf = torch.bfloat16

        def host(bits):
            return torch.from_numpy(bits.view(np.int16)).view(bf).pin_memory()

        e = F.empty_qtensor
        self.events = None
        if name == "tensorwise_256":
            self.rec = F.Recipe(kind="tensorwise")
            n = 256
            self.h = {"x": host(bf16_bits_normal(n, n, seed=0, stream=0)),
                      "w": host(bf16_bits_normal(n, n, seed=0, stream=1))}
            self.q = {"x": e(self.rec, n, n, "activation", device=dev),
                      "w": e(self.rec, n, n, "weight", device=dev)}
            self.ws = torch.empty(F.workspace_bytes(self.rec, n, n), dtype=torch.uint8,
                                  device=dev)
            self.outs = {"y": torch.empty((n, n), dtype=bf, device=dev)}
            self.flops = 2.0 * n ** 3
            self.quant_bytes = 2 * n * n * 4.0
            self.launches = 5                    # amax + cast for X and W, GEMM
        elif name == "mxfp8_fprop":
            self.rec = F.Recipe(kind="mxfp8")
            M, N, K = 8192, 4096, 4096
            self.h = {"x": host(bf16_bits_normal(M, K, seed=0, stream=0, outlier_p=1e-3,
                                                 outlier_factor=50.0)),
                      "w": host(bf16_bits_normal(N, K, seed=0, stream=1, sigma=0.02))}
            self.q = {"x": e(self.rec, M, K, "activation", device=dev),
                      "w": e(self.rec, N, K, "weight", device=dev)}
            self.outs = {"y": torch.empty((M, N), dtype=bf, device=dev)}
            self.flops = 2.0 * M * N * K
            self.quant_bytes = (M * K + N * K) * (2 + 2 + 2 / 32.0)
            self.launches = 2                    # X and W in one grouped launch, GEMM
        elif name == "blockwise_fwd_bwd":
            self.rec = F.Recipe(kind="blockwise")
            n = 4096
            self.h = {"x": host(bf16_bits_normal(n, n, seed=0, stream=0)),
                      "w": host(bf16_bits_normal(n, n, seed=0, stream=1, sigma=0.02)),
                      "dy": host(bf16_bits_normal(n, n, seed=0, stream=2, sigma=1e-3))}
            self.q = {"x": e(self.rec, n, n, "activation", device=dev),
                      "w": e(self.rec, n, n, "weight", device=dev),
                      "dy": e(self.rec, n, n, "grad", device=dev)}
            self.outs = {k: torch.empty((n, n), dtype=bf, device=dev) for k in ("y", "dx", "dw")}
            self.flops = 3 * 2.0 * n ** 3
            self.quant_bytes = 2 * n * n * (2 + 2 + 2 * 4 / 128.0) + n * n * (2 + 2)
            self.launches = 5                    # X and W grouped, dY, three GEMMs
        else:
            self.rec = F.Recipe(kind="delayed", amax_history_len=1024)
            M, N, K = 8192, 4096, 4096
            sig = sigma_schedule(DELAYED_STEPS)
            # 64 distinct inputs of drifting scale (x_t ~ N(0, sigma_t), 64 MB each), drawn on
            # the device from one seeded generator per step (a host draw takes seconds per
            # tensor); the timed steps walk through them in order
            def draw(t):
                gt = torch.Generator(device=dev).manual_seed(STREAM_STEP0 + t)
                return (torch.randn((M, K), device=dev, generator=gt) * float(sig[t])).to(bf)
            self.xs = [draw(t) for t in range(DELAYED_STEPS)]
            self.xs_host = [x.cpu().pin_memory() for x in self.xs]
            self.h = {"x": self.xs_host[0]}
            self.state = F.DelayedState(self.rec, device=dev)
            wstate = F.DelayedState(self.rec, device=dev, role="weight")
            wd = torch.from_numpy(bf16_bits_normal(N, K, seed=0, stream=1, sigma=0.02)
                                  .view(np.int16)).view(bf).to(dev)
            self.wq = F.quantize(self.rec, wd, "weight",
                                 out=wstate.bind(e(self.rec, N, K, "weight", device=dev)))
            self.q = {"x": self.state.bind(e(self.rec, M, K, "activation", device=dev))}
            self.ws = torch.empty(F.workspace_bytes(self.rec, M, K), dtype=torch.uint8, device=dev)
            self.outs = {"y": torch.empty((M, N), dtype=bf, device=dev)}
            self.flops = 2.0 * M * N * K
            self.quant_bytes = M * K * 4.0
            self.launches = 4                    # cast, amax finalize, GEMM, history update
            self.t = 0
        self.d = {k: v.to(dev) for k, v in self.h.items()}
        self.stream = torch.cuda.current_stream(dev)

    def _t(self, kind, fn, name):
        if self.events is None:
            return fn()
        s, e = self.torch.cuda.Event(enable_timing=True), self.torch.cuda.Event(enable_timing=True)
        s.record(self.stream)
        fn()
        e.record(self.stream)
        self.events.append((kind, name, s, e))

    def run(self, d=None, o=None):
        F, rec, T, q = self.F, self.rec, self._t, self.q
        resident = d is None
        d = self.d if resident else d
        o = self.outs if o is None else o
        if self.name == "tensorwise_256":
            T("quant", lambda: F.quantize(rec, d["x"], "activation", out=q["x"],
                                          workspace=self.ws), "quantize_x")
            T("quant", lambda: F.quantize(rec, d["w"], "weight", out=q["w"], workspace=self.ws),
              "quantize_w")
            T("gemm", lambda: F.linear_fwd(rec, q["x"], q["w"], y=o["y"]), "fprop")
        elif self.name == "mxfp8_fprop":
            T("quant", lambda: F.quantize_group(rec, [d["x"], d["w"]], ["activation", "weight"],
                                                outs=[q["x"], q["w"]]), "quantize_x_w")
            T("gemm", lambda: F.linear_fwd(rec, q["x"], q["w"], y=o["y"]), "fprop")
        elif self.name == "blockwise_fwd_bwd":
            T("quant", lambda: F.quantize_group(rec, [d["x"], d["w"]], ["activation", "weight"],
                                                outs=[q["x"], q["w"]]), "quantize_x_w")
            T("gemm", lambda: F.linear_fwd(rec, q["x"], q["w"], y=o["y"]), "fprop")
            T("quant", lambda: F.quantize(rec, d["dy"], "grad", out=q["dy"]), "quantize_dy")
            T("gemm", lambda: F.linear_bwd(rec, q["dy"], q["x"], q["w"], want_dw=False,
                                           dx=o["dx"]), "dgrad")
            T("gemm", lambda: F.linear_bwd(rec, q["dy"], q["x"], q["w"], want_dx=False,
                                           dw=o["dw"]), "wgrad")
        else:
            x = self.xs[self.t % DELAYED_STEPS] if resident else d["x"]
            self.t += 1
            T("quant", lambda: F.quantize(rec, x, "activation", out=q["x"], workspace=self.ws),
              "quantize_x")
            T("gemm", lambda: F.linear_fwd(rec, q["x"], self.wq, y=o["y"]), "fprop")
            T("other", lambda: F.amax_update(rec, self.state, q["x"].amax), "amax_update")

    def run_e2e(self, steps):
        """`steps` steps whose inputs are copied from pinned host memory and whose outputs are
        copied back to pinned host memory, pipelined like the MLP step's: uploads on one
        stream, the step on the compute stream, downloads on a third, two buffer sets
        alternating. Returns the elapsed ms from the first upload to the last download."""
        torch = self.torch
        comp = self.stream
        if not hasattr(self, "d_sets"):
            self.d_sets = [self.d, {k: torch.empty_like(v) for k, v in self.d.items()}]
            self.o_sets = [self.outs, {k: torch.empty_like(v) for k, v in self.outs.items()}]
            self.h_out = [{k: torch.empty(v.shape, dtype=v.dtype).pin_memory()
                           for k, v in self.outs.items()} for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(self.dev), torch.cuda.Stream(self.dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(comp)
        s_in.wait_stream(comp)
        s_out.wait_stream(comp)
        for i in range(steps):
            b = i % 2
            src = ({"x": self.xs_host[i % DELAYED_STEPS]} if self.name == "delayed_step"
                   else self.h)
            if i >= 2:
                s_in.wait_event(ev_comp[b])               # step i-2 is done with these inputs
            with torch.cuda.stream(s_in):
                for k, v in src.items():
                    self.d_sets[b][k].copy_(v, non_blocking=True)
                ev_in[b].record(s_in)
            comp.wait_event(ev_in[b])
            if i >= 2:
                comp.wait_event(ev_out[b])                # step i-2's outputs are downloaded
            with torch.cuda.stream(comp):
                self.run(self.d_sets[b], self.o_sets[b])
                ev_comp[b].record(comp)
            s_out.wait_event(ev_comp[b])
            with torch.cuda.stream(s_out):
                for k, v in self.o_sets[b].items():
                    self.h_out[b][k].copy_(v, non_blocking=True)
                ev_out[b].record(s_out)
        comp.wait_stream(s_in)
        comp.wait_stream(s_out)
        t1.record(comp)
        t1.synchronize()
        return t0.elapsed_time(t1)

    def h2d_bytes(self):
        return sum(v.numel() * 2 for v in self.h.values())

    def d2h_bytes(self):
        return sum(v.numel() * 2 for v in self.outs.values())


_CFG_SETUP = {}


def cpu_baseline_config(name, m_sample=1024):
    """The oracle on a bounded sample of a configuration's step: quantisation and GEMM rows of
    m_sample of the activation rows (scaled up), weight quantisation of m_sample of its rows
    (scaled up)."""
    from oracle import fp8_oracle as O
    from workloads import bf16_bits_normal
    if name == "tensorwise_256":                 # small enough for the whole step
        x = bf16_bits_normal(256, 256, seed=0, stream=0)
        w = bf16_bits_normal(256, 256, seed=0, stream=1)
        reps = 20
        t0 = time.perf_counter()
        for _ in range(reps):
            qx, qw = O.quantize_tensorwise(x), O.quantize_tensorwise(w)
            O.f64_to_bf16(O.gemm_tn_f64(O.dequant_tensor(qx["row"], qx["scale_inv"]),
                                        O.dequant_tensor(qw["row"], qw["scale_inv"])))
        step_s = (time.perf_counter() - t0) / reps
        cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
        return {"value": round(2.0 * 256 ** 3 / step_s / 1e12, 6), "unit": "TFLOP/s",
                "cores": cores, "kind": "oracle", "step_seconds_estimate": round(step_s, 5),
                "sample": f"the whole oracle step, mean of {reps}"}
    n_rows = {"mxfp8_fprop": 8192, "blockwise_fwd_bwd": 4096, "delayed_step": 8192}[name]
    K = 4096
    if name == "blockwise_fwd_bwd":                # whole 128-row blocks of the column copies
        m_sample = max(128, m_sample // 128 * 128)
    xs = bf16_bits_normal(m_sample, K, seed=0, stream=0)
    ws = bf16_bits_normal(m_sample, K, seed=0, stream=1, sigma=0.02)
    if name not in _CFG_SETUP:                    # untimed: the full weight's quantised copies
        wfull = bf16_bits_normal(4096, K, seed=0, stream=1, sigma=0.02)
        if name == "mxfp8_fprop":
            qw = O.quantize_mxfp8(wfull, want_col=False)
            _CFG_SETUP[name] = dict(wr=O.dequant_mx(qw["row"], qw["row_scale"]))
        elif name == "blockwise_fwd_bwd":
            qw = O.quantize_blockwise_128x128(wfull)
            _CFG_SETUP[name] = dict(wr=O.dequant_128x128(qw["row"], qw["row_scale_inv"]),
                                    wc=O.dequant_128x128(qw["col"], qw["col_scale_inv"]))
        else:
            qw = O.DelayedScaling(1024).quantize(wfull)
            _CFG_SETUP[name] = dict(wr=O.dequant_tensor(qw["row"], qw["scale_inv"]))
    S = _CFG_SETUP[name]
    t0 = time.perf_counter()
    if name == "mxfp8_fprop":
        O.quantize_mxfp8(ws)
        t_w = time.perf_counter() - t0
        t0 = time.perf_counter()
        qx = O.quantize_mxfp8(xs)
        O.f64_to_bf16(O.gemm_tn_f64(O.dequant_mx(qx["row"], qx["row_scale"]), S["wr"]))
        t_x = time.perf_counter() - t0
        flops = 2.0 * 8192 * 4096 * K
    elif name == "blockwise_fwd_bwd":
        O.quantize_blockwise_128x128(bf16_bits_normal(128, K, seed=0, stream=1, sigma=0.02))
        t_w = (time.perf_counter() - t0) * m_sample / 128.0      # per m_sample weight rows
        wr, wc = S["wr"], S["wc"]
        t0 = time.perf_counter()
        qx = O.quantize_blockwise_1x128(xs)
        qd = O.quantize_blockwise_1x128(bf16_bits_normal(m_sample, K, seed=0, stream=2,
                                                         sigma=1e-3))
        O.gemm_tn_f64(O.dequant_1x128(qx["row"], qx["row_scale_inv"]), wr)
        O.gemm_tn_f64(O.dequant_1x128(qd["row"], qd["row_scale_inv"]), wc)
        # wgrad: each sampled token row adds its outer product to every dW element
        O.gemm_tn_f64(O.dequant_1x128(qd["col"], qd["col_scale_inv"]),
                      O.dequant_1x128(qx["col"], qx["col_scale_inv"]))
        t_x = time.perf_counter() - t0
        flops = 3 * 2.0 * 4096 ** 3
    else:
        t_w = 0.0
        d = O.DelayedScaling(1024)
        t0 = time.perf_counter()
        q = d.quantize(xs)
        O.f64_to_bf16(O.gemm_tn_f64(O.dequant_tensor(q["row"], q["scale_inv"]), S["wr"]))
        d.update(q["amax"])
        t_x = time.perf_counter() - t0
        flops = 2.0 * 8192 * 4096 * K
    step_s = t_w * (4096 / m_sample) + t_x * (n_rows / m_sample)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(flops / step_s / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle", "step_seconds_estimate": round(step_s, 2),
            "sample": f"oracle step on {m_sample} of {n_rows} activation rows and {m_sample} "
                      f"weight rows, scaled by {n_rows // m_sample}"}


def run_config(args):
    """`--workload` other than the MLP step: the same JSON contract for that configuration."""
    import torch
    import scaled_quantize_fp8_gb300 as F
    from scaled_quantize_fp8_gb300 import build as B
    B.build()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    st = ConfigStep(torch, F, dev, args.workload)
    for _ in range(args.warmup):
        st.run()
    step = st.run
    if args.workload == "tensorwise_256":
        # launch-bound: one step is one replay of a CUDA graph holding its five kernels
        side = torch.cuda.Stream(dev)
        side.wait_stream(st.stream)
        with torch.cuda.stream(side):
            st.run()
        st.stream.wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            st.run()
        step = graph.replay
        for _ in range(args.warmup):
            step()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local)
    clocks.start()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(st.stream)
    for _ in range(args.steps):
        step()
    t1.record(st.stream)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    ms_total = max_over_ranks(t0.elapsed_time(t1), dist, dev)
    st.events = []
    for _ in range(max(1, min(args.steps, 20))):
        st.run()
    torch.cuda.synchronize(dev)
    ms = {"gemm": [], "quant": [], "other": []}
    per_name = {}
    for kind, name, s, e in st.events:
        ms[kind].append(s.elapsed_time(e))
        per_name.setdefault(name, []).append(s.elapsed_time(e))
    st.events = None
    st.run_e2e(max(2, args.warmup))
    ms_e2e = max_over_ranks(st.run_e2e(args.steps), dist, dev)
    n_pk = max(1, min(args.steps, 20))
    value = world * st.flops / (ms_total / args.steps * 1e-3) / 1e12
    hbm, fp8_peak, src = peaks()
    gemm_ms = statistics.mean(ms["gemm"])
    gemm_flops = st.flops / (3 if args.workload == "blockwise_fwd_bwd" else 1)
    achieved = gemm_flops / (gemm_ms * 1e-3) / 1e12
    quant_ms = sum(ms["quant"]) / n_pk
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_total / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate)",
            "data": "synthetic",
            "config": {"workload": CONFIGS[args.workload], "recipe": st.rec.kind,
                       "parallelism": "replicas" if world > 1 else "single",
                       "l2": ("inputs fit in L2 and are not flushed: a launch-bound "
                              "configuration, timed as graph replays"
                              if args.workload == "tensorwise_256" else
                              "not flushed: each step touches more than L2 (129 MB): "
                              "0.26-0.3 GB of inputs, codes and outputs; the delayed step "
                              f"walks through {DELAYED_STEPS} distinct 64 MB X_t"),
                       "gemm_flops_per_step": st.flops},
            "roofline": {"bound": "tensor", "kernel": f"gemm_tn_kernel ({st.rec.kind})",
                         "achieved": round(achieved, 1), "peak": fp8_peak, "unit": "TFLOP/s",
                         "frac": round(achieved / fp8_peak, 4), "traffic": None,
                         "peak_source": f"{src}: bf16 x {FP8_OVER_BF16} (nominal fp8/bf16)",
                         "avg_launch_ms": round(gemm_ms, 4)},
            "quantize": {"gbs": round(st.quant_bytes / (quant_ms * 1e-3) / 1e9, 1),
                         "peak_gbs": hbm, "ms_per_step": round(quant_ms, 4),
                         "algorithmic_bytes_per_step": st.quant_bytes, "peak_source": src},
            "e2e": {"value": round(world * st.flops / (ms_e2e / args.steps * 1e-3) / 1e12, 2),
                    "unit": "TFLOP/s", "h2d_bytes_per_step": st.h2d_bytes(),
                    "d2h_bytes_per_step": st.d2h_bytes(),
                    "copies": "pinned host, own streams, overlapped with the adjacent steps"},
            "kernels_ms": {k: round(statistics.mean(v), 4) for k, v in per_name.items()},
            "gpu_launches": st.launches * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu_baseline_config(args.workload),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- CPU oracle

_ORACLE_SETUP = {}


def _oracle_setup():
    """Untimed: seeded inputs and the dequantised full weights the sampled GEMMs read."""
    if not _ORACLE_SETUP:
        from oracle import fp8_oracle as O
        from workloads import bf16_bits_normal
        w1 = bf16_bits_normal(FFN, HIDDEN, seed=0, stream=1, sigma=0.02)
        w2 = bf16_bits_normal(HIDDEN, FFN, seed=0, stream=3, sigma=0.02)
        qw1, qw2 = O.quantize_mxfp8(w1), O.quantize_mxfp8(w2)
        dq = lambda q, c: O.dequant_mx(q[c], q[c + "_scale"])  # noqa: E731
        _ORACLE_SETUP.update(
            w1=w1, w2=w2, w1r=dq(qw1, "row"), w1c=dq(qw1, "col"), w2r=dq(qw2, "row"),
            w2c=dq(qw2, "col"),
            x=bf16_bits_normal(TOKENS, HIDDEN, seed=0, stream=0),
            dy=bf16_bits_normal(TOKENS, HIDDEN, seed=0, stream=2, sigma=1e-3))
    return _ORACLE_SETUP


def _oracle_warm(_):
    """Pool worker start-up: import the oracle and the generators (not timed)."""
    from oracle import fp8_oracle  # noqa: F401
    from workloads import bf16_bits_normal  # noqa: F401
    time.sleep(0.5)
    return os.getpid()


def _oracle_quantize_chunk(task):
    """Pool worker: the oracle's MXFP8 quantiser (row + column copies) on one seeded
    rows x 4096 bf16 chunk; returns the wall-clock start and end of the quantisation."""
    seed, rows = task
    from oracle import fp8_oracle as O
    from workloads import bf16_bits_normal
    x = bf16_bits_normal(rows, 4096, seed=seed, stream=0)
    t0 = time.time()
    O.quantize_mxfp8(x)
    return t0, time.time()


def oracle_quantize_rates(rows=512):
    """The oracle's MXFP8 quantize in algorithmic GB/s (2 B read, 2 x (1 + 1/32) B written per
    element) on one core, and on every core of the host with one chunk per core in a spawned
    process pool (wall clock from the first chunk's start to the last one's end)."""
    import multiprocessing as mp
    per_chunk = rows * 4096 * (2 + 2 + 2 / 32.0)
    t0, t1 = _oracle_quantize_chunk((0, rows))
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    with mp.get_context("spawn").Pool(cores) as pool:
        pool.map(_oracle_warm, range(cores), chunksize=1)
        spans = pool.map(_oracle_quantize_chunk, [(i + 1, rows) for i in range(cores)],
                         chunksize=1)
    wall = max(e for _, e in spans) - min(b for b, _ in spans)
    return {"gbs_1_core": round(per_chunk / (t1 - t0) / 1e9, 4),
            "gbs_all_cores": round(cores * per_chunk / wall / 1e9, 4), "cores": cores,
            "sample": f"MXFP8 quantize (row + column copies) of a {rows} x 4096 bf16 chunk, "
                      f"one chunk per core"}


def cpu_baseline(m_sample=128, w_frac=16, quantize_rates=True):
    """The oracle, as it stands, on a bounded sample of the same step: the token-proportional
    work on m_sample of the 8192 tokens (scaled up by 8192/m_sample) plus the per-step weight
    quantisation on 1/w_frac of the weight rows (scaled up by w_frac)."""
    from oracle import fp8_oracle as O
    S = _oracle_setup()
    dq = lambda q, c: O.dequant_mx(q[c], q[c + "_scale"])  # noqa: E731
    x, dy = S["x"][:m_sample], S["dy"][:m_sample]
    t0 = time.perf_counter()
    O.quantize_mxfp8(S["w1"][: FFN // w_frac])
    O.quantize_mxfp8(S["w2"][: HIDDEN // w_frac])
    t_w = (time.perf_counter() - t0) * w_frac
    t0 = time.perf_counter()
    qx = O.quantize_mxfp8(x)
    h = O.f64_to_bf16(O.gemm_tn_f64(dq(qx, "row"), S["w1r"]))
    qh = O.quantize_mxfp8(h, want_col=False)
    qa = O.quantize_mxfp8(O.gelu_bf16(h))
    O.f64_to_bf16(O.gemm_tn_f64(dq(qa, "row"), S["w2r"]))
    qdy = O.quantize_mxfp8(dy)
    da = O.f64_to_bf16(O.gemm_tn_f64(dq(qdy, "row"), S["w2c"]))
    O.gemm_tn_f64(dq(qdy, "col"), dq(qa, "col"))
    qdh = O.quantize_mxfp8(O.dgelu_bf16(da, qh["row"], qh["row_scale"]))
    O.gemm_tn_f64(dq(qdh, "row"), S["w1c"])
    O.gemm_tn_f64(dq(qdh, "col"), dq(qx, "col"))
    t_tok = (time.perf_counter() - t0) * (TOKENS // m_sample)
    step_s = t_w + t_tok
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    out = {"value": round(GEMM_FLOPS / step_s / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
           "kind": "oracle", "step_seconds_estimate": round(step_s, 2),
           "sample": (f"oracle MLP step on {m_sample} of {TOKENS} tokens (x{TOKENS // m_sample})"
                      f" plus weight quantisation of 1/{w_frac} of the rows (x{w_frac}); "
                      "numpy: elementwise work on one core, fp64 matmuls on the BLAS threads")}
    if quantize_rates:
        out["quantize"] = oracle_quantize_rates()
    return out


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and rank != 0:
        return
    vals = []
    if args.workload == "mlp":
        def one():
            return cpu_baseline(m_sample=32, w_frac=64, quantize_rates=False)
        workload = WORKLOAD
    else:
        def one():
            return cpu_baseline_config(args.workload, m_sample=128)
        workload = CONFIGS[args.workload]
    if args.workload == "mlp":
        _oracle_setup()
    for _ in range(min(args.warmup, 1)):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(one())
    elapsed = time.perf_counter() - t0
    v = statistics.median(x["value"] for x in vals)
    c = dict(vals[0])
    c["value"] = v
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(statistics.median(x["step_seconds_estimate"] for x in vals) * 1e3, 1),
        "ms_per_step_kind": "extrapolated: each step times the oracle on a bounded sample of the "
                            "workload and scales the time to the whole step",
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": workload, "recipe": {"mlp": "mxfp8"}.get(
            args.workload, args.workload.split("_")[0]), "parallelism": "single"},
        "cpu_baseline": c, "wall_seconds": round(elapsed, 1),
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_profile_case(args):
    """Launch one kernel kind a few times on its own (for ncu captures; prints no JSON line).
    quant_mx / quant_tensorwise / quant_blockwise: X --rows x --cols bf16 (default 16384 x 8192,
    256 MiB, above L2).
    gemm_mx / gemm_tensorwise / gemm_blockwise: fprop 8192 x 4096 x 4096.
    gemm_wgrad_blockwise: blockwise wgrad 4096 x 4096 x 8192 (1x128 scales on both operands).
    gelu_mx / dgelu_mx: the standalone GeLU / dGeLU + MXFP8 quantize on h 8192 x 16384.
    gemm_gelu_mx / gemm_dgelu_mx: fc1 with the GeLU epilogue (8192 x 16384 x 4096) and fc2's
    dgrad with the dGeLU epilogue (8192 x 16384 x 4096).
    gemm_mx_mlp: the MLP step's four plain-store MXFP8 GEMMs (fc2 fprop, fc2 wgrad, fc1
    dgrad, fc1 wgrad) at full size, in that order.
    quant_group_mx: the MLP step's grouped MXFP8 quantize of X 8192 x 4096, W1 16384 x 4096
    and W2 4096 x 16384 (one launch); quant_group_blockwise: the same three tensors under the
    blockwise recipe (X in 1x128 blocks, W1 and W2 in 128x128 tiles)."""
    import torch
    import scaled_quantize_fp8_gb300 as F
    from scaled_quantize_fp8_gb300 import build as B
    B.build()
    case = args.profile
    parts = case.split("_")
    kind = "mxfp8" if "mx" in parts else parts[-1]
    rec = F.Recipe(kind=kind)
    g = torch.Generator(device="cuda").manual_seed(0)
    if case in ("gemm_gelu_mx", "gemm_dgelu_mx"):
        M, H, Fd = TOKENS, HIDDEN, FFN
        x = torch.randn((M, H), device="cuda", generator=g).to(torch.bfloat16)
        w1 = (torch.randn((Fd, H), device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        w2 = (torch.randn((H, Fd), device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        dy = (torch.randn((M, H), device="cuda", generator=g) * 1e-3).to(torch.bfloat16)
        xq, w1q = F.quantize(rec, x, "activation"), F.quantize(rec, w1, "weight")
        w2q, dyq = F.quantize(rec, w2, "weight"), F.quantize(rec, dy, "grad")
        a_q, h_q = F.linear_fwd_gelu(rec, xq, w1q)
        dh_q = F.linear_dgrad_dgelu(rec, dyq, w2q, h_q)
        for _ in range(args.steps):
            if case == "gemm_gelu_mx":
                F.linear_fwd_gelu(rec, xq, w1q, a_q=a_q, h_q=h_q)
            else:
                F.linear_dgrad_dgelu(rec, dyq, w2q, h_q, dh_q=dh_q)
    elif case == "gemm_mx_mlp":
        M, H, Fd = TOKENS, HIDDEN, FFN
        x = torch.randn((M, H), device="cuda", generator=g).to(torch.bfloat16)
        w1 = (torch.randn((Fd, H), device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        w2 = (torch.randn((H, Fd), device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        a = torch.randn((M, Fd), device="cuda", generator=g).to(torch.bfloat16)
        dy = (torch.randn((M, H), device="cuda", generator=g) * 1e-3).to(torch.bfloat16)
        xq, w1q = F.quantize(rec, x, "activation"), F.quantize(rec, w1, "weight")
        w2q, aq = F.quantize(rec, w2, "weight"), F.quantize(rec, a, "activation")
        dyq, dhq = F.quantize(rec, dy, "grad"), F.quantize(rec, a, "grad")
        y, dx = torch.empty_like(x), torch.empty_like(x)
        dw1, dw2 = torch.empty_like(w1), torch.empty_like(w2)
        for _ in range(args.steps):
            F.linear_fwd(rec, aq, w2q, y=y)                                   # fc2 fprop
            F.linear_bwd(rec, dyq, aq, None, want_dx=False, dw=dw2)           # fc2 wgrad
            F.linear_bwd(rec, dhq, None, w1q, want_dw=False, dx=dx)           # fc1 dgrad
            F.linear_bwd(rec, dhq, xq, None, want_dx=False, dw=dw1)           # fc1 wgrad
    elif case in ("gelu_mx", "dgelu_mx"):
        h = torch.randn((8192, 16384), device="cuda", generator=g).to(torch.bfloat16)
        a_q, h_q, _ = F.gelu_quantize(rec, h)
        for _ in range(args.steps):
            if case == "gelu_mx":
                F.gelu_quantize(rec, h, a_q=a_q, h_q=h_q)
            else:
                F.dgelu_quantize(rec, h, h_q, dh_q=a_q)
    elif case in ("quant_group_mx", "quant_group_blockwise"):
        shapes = ((8192, 4096, 1.0), (16384, 4096, 0.02), (4096, 16384, 0.02))
        xs = [(torch.randn((r, c), device="cuda", generator=g) * sg).to(torch.bfloat16)
              for r, c, sg in shapes]
        roles = ["activation", "weight", "weight"]
        outs = F.quantize_group(rec, xs, roles)
        for _ in range(args.steps):
            F.quantize_group(rec, xs, roles, outs=outs)
    elif case == "gemm_wgrad_blockwise":
        x = torch.randn((8192, 4096), device="cuda", generator=g).to(torch.bfloat16)
        dy = (torch.randn((8192, 4096), device="cuda", generator=g) * 1e-3).to(torch.bfloat16)
        xq, dyq = F.quantize(rec, x, "activation"), F.quantize(rec, dy, "grad")
        dw = torch.empty((4096, 4096), dtype=torch.bfloat16, device="cuda")
        for _ in range(args.steps):
            F.linear_bwd(rec, dyq, xq, None, want_dx=False, dw=dw)
    elif case.startswith("quant"):
        R, C = args.rows, args.cols
        x = torch.randn((R, C), device="cuda", generator=g).to(torch.bfloat16)
        q = F.empty_qtensor(rec, R, C, "activation")
        for _ in range(args.steps):
            F.quantize(rec, x, "activation", out=q)
    else:
        x = torch.randn((8192, 4096), device="cuda", generator=g).to(torch.bfloat16)
        w = (torch.randn((4096, 4096), device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        xq, wq = F.quantize(rec, x, "activation"), F.quantize(rec, w, "weight")
        y = torch.empty((8192, 4096), dtype=torch.bfloat16, device="cuda")
        for _ in range(args.steps):
            F.linear_fwd(rec, xq, wq, y=y)
    torch.cuda.synchronize()
    print(f"profile case {case}: {args.steps} launches done")


def run_profile_suite(args):
    """Every kernel of the library that has no capture of its own, twice each (the second call
    inside an NVTX range "capture"), one case after another, for one ncu capture; prints the
    case order, no JSON line. Tensors are 16384 x
    8192 bf16 (256 MiB, above L2) for the quantizers, 8192 x 16384 for GeLU / dGeLU, and
    8192 x 4096 x 4096 for the GEMMs; each case frees its memory before the next."""
    import torch
    import scaled_quantize_fp8_gb300 as F
    from scaled_quantize_fp8_gb300 import build as B
    B.build()
    g = torch.Generator(device="cuda").manual_seed(0)
    bf = torch.bfloat16
    R, C = 16384, 8192

    def randn(r, c, sigma=1.0, dtype=bf):
        return (torch.randn((r, c), device="cuda", generator=g) * sigma).to(dtype)

    def case(name, fn, prep=None):
        # the second call runs inside an NVTX range named "capture", which an ncu capture
        # selects with --nvtx --nvtx-include capture/
        state = prep() if prep else None
        torch.cuda.synchronize()
        print(f"case {name}", flush=True)
        fn(state)
        torch.cuda.nvtx.range_push("capture")
        fn(state)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        del state
        torch.cuda.empty_cache()

    def quant(kind, role="activation", fmt="e4m3"):
        rec = F.Recipe(kind=kind, format=fmt)

        def prep():
            x = randn(R, C)
            q = F.empty_qtensor(rec, R, C, role)
            if kind == "delayed":
                q.scale.fill_(448.0 / 5.0)
                q.scale_inv.fill_(5.0 / 448.0)
            ws = torch.empty(max(16, F.workspace_bytes(rec, R, C)), dtype=torch.uint8,
                             device="cuda")
            return x, q, ws
        return lambda st: F.quantize(rec, st[0], role, out=st[1], workspace=st[2]), prep

    for kind, role, fmt in (("tensorwise", "activation", "e4m3"),
                            ("delayed", "activation", "e4m3"),
                            ("blockwise", "activation", "e4m3"),
                            ("blockwise", "weight", "e4m3"),
                            ("tensorwise", "grad", "hybrid"),
                            ("blockwise", "grad", "hybrid")):
        fn, prep = quant(kind, role, fmt)
        case(f"quantize {kind} {role} {fmt}", fn, prep)

    rec_d = F.Recipe(kind="delayed", amax_history_len=1024)

    def prep_hist():
        st = F.DelayedState(rec_d)
        return st, torch.full((1,), 3.0, device="cuda")
    case("amax_history_update L=1024", lambda st: F.amax_update(rec_d, st[0], st[1]), prep_hist)

    for kind in ("mxfp8", "tensorwise", "blockwise"):
        rec = F.Recipe(kind=kind)

        def prep_master(rec=rec):
            w = torch.randn((R, C // 2), device="cuda", generator=g) * 0.02
            q = F.empty_qtensor(rec, R, C // 2, "weight")
            ws = torch.empty(max(16, F.workspace_bytes(rec, R, C // 2)), dtype=torch.uint8,
                             device="cuda")
            return w, q, ws
        case(f"quantize_master {kind} fp32 {R}x{C // 2}",
             lambda st, rec=rec: F.quantize_master(rec, st[0], out=st[1], workspace=st[2]),
             prep_master)

    rec = F.Recipe(kind="mxfp8")

    def prep_gelu():
        h = randn(8192, 16384, 2.0)
        a_q, h_q, _ = F.gelu_quantize(rec, h)
        return h, a_q, h_q
    case("gelu_quantize 8192x16384", lambda st: F.gelu_quantize(rec, st[0], a_q=st[1], h_q=st[2]),
         prep_gelu)

    def prep_dgelu():
        h = randn(8192, 16384, 2.0)
        _, h_q, _ = F.gelu_quantize(rec, h)
        da = randn(8192, 16384, 1e-3)
        dh_q, _ = F.dgelu_quantize(rec, da, h_q)
        return da, h_q, dh_q
    case("dgelu_quantize 8192x16384",
         lambda st: F.dgelu_quantize(rec, st[0], st[1], dh_q=st[2]), prep_dgelu)

    rec_t = F.Recipe(kind="tensorwise")

    def prep_gemm_t():
        xq = F.quantize(rec_t, randn(8192, 4096), "activation")
        wq = F.quantize(rec_t, randn(4096, 4096, 0.02), "weight")
        return xq, wq, torch.empty((8192, 4096), dtype=bf, device="cuda")
    case("gemm tensorwise 8192x4096x4096",
         lambda st: F.linear_fwd(rec_t, st[0], st[1], y=st[2]), prep_gemm_t)

    rec_b = F.Recipe(kind="mxfp8", fp8_wgrad=False)

    def prep_gemm_bf16():
        xq = F.quantize(rec_b, randn(8192, 4096), "activation", want_row=False)
        dyq = F.quantize(rec_b, randn(8192, 4096, 1e-3), "grad", want_row=False)
        return xq, dyq, torch.empty((4096, 4096), dtype=bf, device="cuda")
    case("gemm bf16 wgrad 4096x4096x8192",
         lambda st: F.linear_bwd(rec_b, st[1], st[0], None, want_dx=False, dw=st[2]),
         prep_gemm_bf16)
    print("profile suite done", flush=True)


def run_targets(args):
    """The two named performance targets alone (prints one JSON object, not the benchmark
    line): the 4096^3 MXFP8 GEMM and every recipe's quantize at 8192 x 4096."""
    import torch
    import scaled_quantize_fp8_gb300 as F
    from scaled_quantize_fp8_gb300 import build as B
    B.build()
    dev = torch.device("cuda", 0)
    hbm, fp8_peak, _ = peaks()
    print(json.dumps({"gemm_4096_mxfp8": measure_gemm_4096(torch, F, dev, fp8_peak),
                      "quantize_by_recipe": measure_quantize_by_recipe(torch, F, dev, hbm)}),
          flush=True)


def run_kernels(args):
    """Per-recipe kernel timings (prints one JSON object; not the benchmark line): quantize of an
    8192 x 4096 bf16 activation (row + column copies) and the fprop GEMM 8192 x 4096 x 4096 and
    4096^3, each the mean of 20 launches timed with CUDA events after 5 warm-up launches."""
    import torch
    import scaled_quantize_fp8_gb300 as F
    from scaled_quantize_fp8_gb300 import build as B
    B.build()

    def timed(fn, reps=20, warm=5):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            fn()
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / reps

    g = torch.Generator(device="cuda").manual_seed(0)
    M, N, K = 8192, 4096, 4096
    x = torch.randn((M, K), device="cuda", generator=g).to(torch.bfloat16)
    w = (torch.randn((N, K), device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    out = {}
    for kind in ("mxfp8", "tensorwise", "delayed", "blockwise"):
        rec = F.Recipe(kind=kind)
        qx = F.empty_qtensor(rec, M, K, "activation")
        ws = torch.empty(max(1, F.workspace_bytes(rec, M, K)), dtype=torch.uint8, device="cuda")
        ms = timed(lambda: F.quantize(rec, x, "activation", out=qx, workspace=ws))
        per_elt = {"mxfp8": 2 + 2 + 2 / 32.0, "blockwise": 2 + 2 + 2 * 4 / 128.0}.get(kind, 4.0)
        out[f"quantize_{kind}"] = {"ms": round(ms, 4),
                                   "GB/s": round(M * K * per_elt / ms / 1e6, 1)}
        qw = F.quantize(rec, w, "weight")
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        ms = timed(lambda: F.linear_fwd(rec, qx, qw, y=y))
        qx4 = F.quantize(rec, x[:4096].contiguous(), "activation")
        y4 = torch.empty((4096, N), dtype=torch.bfloat16, device="cuda")
        ms4 = timed(lambda: F.linear_fwd(rec, qx4, qw, y=y4))
        out[f"gemm_{kind}"] = {"8192x4096x4096_TFLOP/s": round(2 * M * N * K / ms / 1e9, 1),
                               "4096^3_TFLOP/s": round(2 * 4096 ** 3 / ms4 / 1e9, 1)}
    # blockwise with power-of-two scales: E8M0 scales in the MXFP8 layout, MXFP8 GEMM path
    rec = F.Recipe(kind="blockwise", power_2_scales=True)
    xq2, wq2 = F.quantize(rec, x, "activation"), F.quantize(rec, w, "weight")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ms = timed(lambda: F.linear_fwd(rec, xq2, wq2, y=y))
    out["gemm_blockwise_pow2"] = {"8192x4096x4096_TFLOP/s": round(2 * M * N * K / ms / 1e9, 1)}
    # tensorwise dgrad 8192 x 4096 x 4096 reading W's column copy (K-major) or, with the column
    # copy never written, W's row copy as an MN-major operand; and the quantize without it
    rec = F.Recipe(kind="tensorwise")
    dy = (torch.randn((M, N), device="cuda", generator=g) * 1e-3).to(torch.bfloat16)
    dyq = F.quantize(rec, dy, "grad", want_col=False)
    w_col = F.quantize(rec, w, "weight")
    w_row = F.quantize(rec, w, "weight", want_col=False)
    dx = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    for name, wq in (("col_copy", w_col), ("row_copy_mn_major", w_row)):
        ms = timed(lambda: F.linear_bwd(rec, dyq, None, wq, want_dw=False, dx=dx))
        out[f"gemm_tensorwise_dgrad_{name}"] = {"TFLOP/s": round(2 * M * N * K / ms / 1e9, 1)}
    qx = F.empty_qtensor(rec, M, K, "activation", True, False)
    ws = torch.empty(max(1, F.workspace_bytes(rec, M, K)), dtype=torch.uint8, device="cuda")
    ms = timed(lambda: F.quantize(rec, x, "activation", want_col=False, out=qx, workspace=ws))
    out["quantize_tensorwise_row_only"] = {"ms": round(ms, 4),
                                           "GB/s": round(M * K * 3.0 / ms / 1e6, 1)}
    # fp32 master weight W1 16384 x 4096 -> MXFP8 row + column copies (4 B in, 2.06 B out)
    w32 = torch.randn((16384, 4096), device="cuda", generator=g) * 0.02
    rec = F.Recipe(kind="mxfp8")
    qm = F.empty_qtensor(rec, 16384, 4096, "weight")
    ms = timed(lambda: F.quantize_master(rec, w32, out=qm))
    out["quantize_master_mxfp8_16384x4096"] = {
        "ms": round(ms, 4), "GB/s": round(16384 * 4096 * (4 + 2 + 2 / 32.0) / ms / 1e6, 1)}
    torch.cuda.synchronize()
    print(json.dumps({"kernels": out}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile", default=None,
                    choices=["quant_mx", "quant_group_mx", "quant_group_blockwise",
                             "quant_tensorwise", "quant_blockwise",
                             "gemm_mx",
                             "gemm_tensorwise", "gemm_blockwise", "gelu_mx", "dgelu_mx",
                             "gemm_gelu_mx", "gemm_dgelu_mx", "gemm_mx_mlp",
                             "gemm_wgrad_blockwise", "suite"])
    ap.add_argument("--rows", type=int, default=16384, help="--profile quant_*: tensor rows")
    ap.add_argument("--cols", type=int, default=8192, help="--profile quant_*: tensor columns")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mlp", choices=["mlp"] + sorted(CONFIGS),
                    help="the MXFP8 MLP step (default) or one of the smaller configurations")
    ap.add_argument("--targets", action="store_true",
                    help="the 4096^3 MXFP8 GEMM and per-recipe quantize rates only")
    ap.add_argument("--kernels", action="store_true",
                    help="per-recipe quantize and GEMM timings instead of the benchmark step")
    ap.add_argument("--unfused", action="store_true",
                    help="standalone GeLU / dGeLU kernels instead of the fused GEMM epilogues")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile == "suite":
        run_profile_suite(args)
    elif args.profile:
        run_profile_case(args)
    elif args.targets:
        run_targets(args)
    elif args.kernels:
        run_kernels(args)
    elif args.workload != "mlp" and args.impl != "reference":
        run_config(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
