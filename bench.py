"""Benchmark of the NVFP4 linear layer hot path at Llama-3-8B MLP up-projection
shapes: x bf16[16384,4096], W bf16[14336,4096], dy bf16[16384,14336].

One step = the whole path once: amax + fused row/col quantization of x (RHT on
the columnwise copy) and W, the forward GEMM, amax + quantization of dy
(stochastic rounding, RHT on the columnwise copy), the dgrad and the wgrad
GEMMs (3 x 2*16384*14336*4096 = 5.77 TFLOP).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (plain C, OpenMP) on a bounded sample
of the same workload on the host cores.  With N > 1 (torchrun), every rank
runs an independent replica on its own GPU (the path needs no exchange at one
GPU per replica); the value is the sum over ranks, the time the max.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

M, N, K = 16384, 14336, 4096
GEMM_FLOP = 2.0 * M * N * K
STEP_FLOP = 3 * GEMM_FLOP
METRIC = "NVFP4 linear fwd+dgrad+wgrad TFLOP/s (Llama-3-8B MLP up-proj)"
UNIT = "TFLOP/s"
CONFIG = {"workload": "llama3_8b_mlp_up_fwd_dgrad_wgrad", "M_tokens": M, "N_out": N, "K_in": K,
          "x": "bf16[16384,4096] N(0,1) seed 0", "W": "bf16[14336,4096] N(0,0.02^2) seed 1",
          "dy": "bf16[16384,14336] N(0,1e-4) seed 2", "sr_seed": 1234, "rht_sign_seed": 7,
          "l2": "inputs larger than L2 (each step streams > 1.5 GB through HBM)"}
# fp4 dense / bf16 dense nominal ratio (13.5 / 2.25 PFLOP/s) applied to the measured bf16 peak
FP4_OVER_BF16 = 6.0
# dram__bytes_read.sum + dram__bytes_write.sum per launch from ncu captures of the
# current kernels on this workload (profiles/gemm_pair_nvfp4_llama3_8b_fwd.md: the
# forward GEMM launch; profiles/quantize_nvfp4_llama3_8b.md: the six amax + quantize
# launches of one step).  Set to None whenever those kernels change.
GEMM_TRAFFIC_BYTES = float(104373504 + 426027008)
QUANT_TRAFFIC_BYTES = float(134246144 + 2973696 + 134285568 + 39769600 + 117470208 + 65280
                            + 117523968 + 29878016 + 469813760 + 75520 + 469958144 + 229856512)


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- CPU oracle sample
def oracle_sample(x, w, dy, sign, target_s=10.0):
    """Time the oracle on a bounded sample of one step and extrapolate to the
    whole step: quantization of `rows` rows (amax, row + col as in the step) of
    each tensor scaled by element count, plus one tile x tile output block of
    each GEMM (dequantize + fp64 product) scaled by FLOPs.  A small calibration
    pass sizes the sample to take about `target_s` seconds.
    Returns (TFLOP/s, description, threads, seconds measured)."""
    import numpy as np
    import oracle

    def bits(t):
        import torch
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    def deq(t, n):
        c, s, a = t
        return oracle.nvfp4_dequant(c[:n], s[:n], oracle.nvfp4_g(a))

    def run(rows, tile):
        xb, wb, dyb = bits(x[:rows]), bits(w[:rows]), bits(dy[:rows])
        t0 = time.perf_counter()
        xr = oracle.nvfp4_quantize_rows(xb, A=oracle.amax(xb))
        xc = oracle.nvfp4_quantize_cols(xb, rht_sign=sign)
        wr = oracle.nvfp4_quantize_rows(wb, A=oracle.amax(wb))
        oracle.nvfp4_quantize_cols(wb)
        dr = oracle.nvfp4_quantize_rows(dyb, A=oracle.amax(dyb), sr=(1234, 0))
        dc = oracle.nvfp4_quantize_cols(dyb, rht_sign=sign, sr=(1234, 0))
        t_q = time.perf_counter() - t0
        t0 = time.perf_counter()
        oracle.gemm_tn_f64(deq(xr, tile), deq(wr, tile))        # fwd-shaped tile, contraction K
        oracle.gemm_tn_f64(deq(dr, tile), deq(dr, tile))        # dgrad-shaped tile, contraction N
        oracle.gemm_tn_f64(deq(dc, tile), deq(xc, tile))        # wgrad-shaped tile, contraction rows
        t_g = time.perf_counter() - t0
        return t_q, t_g

    r0, g0 = 64, 64
    tq, tg = run(r0, g0)
    rows = int(min(M, max(r0, r0 * (0.5 * target_s) / max(tq, 1e-3))))
    rows = max(16, rows // 16 * 16)
    tile = int(min(rows, max(g0, g0 * ((0.5 * target_s) / max(tg, 1e-3)) ** (1 / 3))))
    t_q, t_g = run(rows, tile)
    q_scale = (M * K + N * K + M * N) / float(rows * (K + K + N))
    g_flop = 2.0 * tile * tile * (K + N + rows)
    g_scale = STEP_FLOP / g_flop
    t_step = t_q * q_scale + t_g * g_scale
    threads = _env_int("OMP_NUM_THREADS", os.cpu_count() or 1)
    desc = (f"oracle on {rows} rows of x/W/dy (amax, row+col quantize with RHT/SR as in the step) "
            f"extrapolated x{q_scale:.3g} by elements, plus one {tile}x{tile} tile of each GEMM "
            f"(dequantize + fp64) extrapolated x{g_scale:.3g} by FLOPs; measured {t_q + t_g:.2f} s")
    return STEP_FLOP / t_step / 1e12, desc, threads, t_q + t_g


def oracle_single_thread(target_s=6.0):
    """The same bounded oracle sample with one OpenMP thread, in a child
    process (the thread count is fixed when the oracle library loads).
    Returns (TFLOP/s, description) or (None, reason)."""
    env = dict(os.environ, OMP_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-child", str(target_s)],
                           env=env, capture_output=True, text=True, timeout=600)
        d = json.loads(r.stdout.strip().splitlines()[-1])
        return d["value"], d["sample"]
    except Exception as e:  # a reported baseline, never a reason to fail the bench
        return None, f"single-thread oracle run failed: {type(e).__name__}"


def oracle_sweep_rate(Ms):
    """The oracle (every OpenMP thread of this process) on the quantize sweep's
    tensors of M in Ms: per tensor the amax and row + col quantization of the
    three variants (NVFP4 RTN, NVFP4 with RHT and SR, MXFP8), input generation
    not timed.  Returns (GB/s of the sweep's algorithmic bytes, seconds)."""
    import numpy as np
    import torch
    import oracle
    from mxfp8_block_scaled_bf16_gb300 import inputs
    sign = inputs.rht_sign_vector()
    sr = (inputs.SR_SEED, 0)
    tot_b = tot_s = 0.0
    for Mq in Ms:
        xb = inputs.student_t3_outliers(Mq).contiguous().view(torch.int16).numpy().view(np.uint16)
        t0 = time.perf_counter()
        A = oracle.amax(xb)
        oracle.nvfp4_quantize_rows(xb, A=A)
        oracle.nvfp4_quantize_cols(xb)
        oracle.nvfp4_quantize_rows(xb, A=A, sr=sr)
        oracle.nvfp4_quantize_cols(xb, rht_sign=sign, sr=sr)
        oracle.mxfp8_quantize_rows(xb)
        oracle.mxfp8_quantize_cols(xb)
        tot_s += time.perf_counter() - t0
        tot_b += xb.size * (5.125 + 5.125 + 4.0625)
    return tot_b / tot_s / 1e9, tot_s


def _oracle_child(target_s):
    if target_s < 0:  # the quantize sweep's single-thread figure, on its smallest tensor
        from mxfp8_block_scaled_bf16_gb300 import inputs
        Ms = [min(inputs.QUANT_SWEEP_M)]
        v, secs = oracle_sweep_rate(Ms)
        print(json.dumps({"value": v, "sample": f"sweep tensor M={Ms[0]}, measured {secs:.2f} s"}), flush=True)
        return 0
    from mxfp8_block_scaled_bf16_gb300 import inputs
    x, w, dy = inputs.llama_up()
    v, desc, threads, _ = oracle_sample(x, w, dy, inputs.rht_sign_vector(), target_s=target_s)
    print(json.dumps({"value": v, "sample": desc, "threads": threads}), flush=True)
    return 0


# ---------------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from mxfp8_block_scaled_bf16_gb300 import inputs
    x, w, dy = inputs.llama_up()
    sign = inputs.rht_sign_vector()
    vals, secs = [], []
    for i in range(args.warmup + args.steps):
        v, desc, threads, s = oracle_sample(x, w, dy, sign, target_s=4.0)
        if i >= args.warmup:
            vals.append(v)
            secs.append(s)
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": STEP_FLOP / (value * 1e12) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4 (oracle: f32 encode, f64 GEMM)",
            "data": "synthetic", "config": CONFIG, "extrapolated": True,
            "extrapolation": "each step times a bounded sample of the workload and scales it to the whole step "
                             "(quantization by elements, GEMM tiles by FLOPs); ms_per_step is that estimate",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc,
                             "extrapolated": True},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import __graft_entry__
    import mxfp8_block_scaled_bf16_gb300 as nvq
    from mxfp8_block_scaled_bf16_gb300 import inputs

    __graft_entry__.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    x_h, w_h, dy_h = inputs.llama_up()
    sign = inputs.rht_sign_vector()
    sr = (inputs.SR_SEED, 0)
    x, w, dy = x_h.to(dev), w_h.to(dev), dy_h.to(dev)
    alloc = nvq.alloc_qtensor
    cc = nvq.colwise_cols
    fwd_bufs = dict(x_row=alloc(nvq.NVFP4, M, K, device=dev), w_row=alloc(nvq.NVFP4, N, K, device=dev),
                    x_col=alloc(nvq.NVFP4, K, cc(nvq.NVFP4, M), device=dev),
                    w_col=alloc(nvq.NVFP4, K, cc(nvq.NVFP4, N), device=dev))
    bwd_bufs = dict(dy_row=alloc(nvq.NVFP4, M, N, device=dev), dy_col=alloc(nvq.NVFP4, N, cc(nvq.NVFP4, M), device=dev))
    y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    dx = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    dw = torch.empty(N, K, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    gemm_events = []

    def step(record):
        # forward: amax + fused quantize of x (row, col+RHT) and W (row, col), GEMM
        nvq.nvfp4_quantize(x, 3, rht_sign=sign, out_row=fwd_bufs["x_row"], out_col=fwd_bufs["x_col"])
        nvq.nvfp4_quantize(w, 3, out_row=fwd_bufs["w_row"], out_col=fwd_bufs["w_col"])
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)] if record else None
        if record:
            ev[0].record(stream)
        nvq.gemm_tn(fwd_bufs["x_row"], fwd_bufs["w_row"], out=y)
        if record:
            ev[1].record(stream)
        # backward: quantize dy (row + col, SR, RHT on col), dgrad, wgrad
        nvq.nvfp4_linear_bwd_quantize(dy, rht_sign=sign, sr=sr, bufs=bwd_bufs)
        if record:
            ev[2].record(stream)
        nvq.nvfp4_linear_dgrad(bwd_bufs["dy_row"], fwd_bufs["w_col"], dx=dx)
        if record:
            ev[3].record(stream)
            ev[4].record(stream)
        nvq.nvfp4_linear_wgrad(bwd_bufs["dy_col"], fwd_bufs["x_col"], dw=dw)
        if record:
            ev[5].record(stream)
            gemm_events.append(ev)

    side = torch.cuda.Stream(dev)

    def step_overlapped():
        """The same calls in the same dependency order, with the two independent
        pairs on two streams: x's and W's quantizations (both feed the forward
        GEMM), and dgrad / wgrad (disjoint operands), so each can run in the
        other's last partial wave."""
        cur = torch.cuda.current_stream(dev)
        fork = torch.cuda.Event()
        fork.record(cur)
        side.wait_event(fork)
        nvq.nvfp4_quantize(x, 3, rht_sign=sign, out_row=fwd_bufs["x_row"], out_col=fwd_bufs["x_col"], stream=cur)
        nvq.nvfp4_quantize(w, 3, out_row=fwd_bufs["w_row"], out_col=fwd_bufs["w_col"], stream=side)
        join = torch.cuda.Event()
        join.record(side)
        cur.wait_event(join)
        nvq.gemm_tn(fwd_bufs["x_row"], fwd_bufs["w_row"], out=y, stream=cur)
        nvq.nvfp4_linear_bwd_quantize(dy, rht_sign=sign, sr=sr, bufs=bwd_bufs, stream=cur)
        fork2 = torch.cuda.Event()
        fork2.record(cur)
        side.wait_event(fork2)
        nvq.nvfp4_linear_dgrad(bwd_bufs["dy_row"], fwd_bufs["w_col"], dx=dx, stream=cur)
        nvq.nvfp4_linear_wgrad(bwd_bufs["dy_col"], fwd_bufs["x_col"], dw=dw, stream=side)
        join2 = torch.cuda.Event()
        join2.record(side)
        cur.wait_event(join2)

    for _ in range(args.warmup):
        step(False)
        if not args.serial_step:
            step_overlapped()
    torch.cuda.synchronize()
    if nvq.device_status() != 0:
        raise RuntimeError("device status error during warm-up")

    # The step is captured once into a CUDA graph (every library call is a
    # stream-ordered memset or kernel launch on the capturing stream) and
    # replayed; per-kernel GEMM times come from an eager pass with events.
    graph = None
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            if args.serial_step:
                step(False)
            else:
                step_overlapped()
        torch.cuda.synchronize()
        for _ in range(args.warmup):
            graph.replay()
    for _ in range(max(2, args.steps // 2)):
        step(True)
    torch.cuda.synchronize()

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step(False)
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1) / args.steps
    gemm_ms = [ev[0].elapsed_time(ev[1]) for ev in gemm_events]
    dgrad_ms = [ev[2].elapsed_time(ev[3]) for ev in gemm_events]
    wgrad_ms = [ev[4].elapsed_time(ev[5]) for ev in gemm_events]
    avg_gemm_ms = statistics.mean(gemm_ms + dgrad_ms + wgrad_ms)
    status = nvq.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")

    # whole-step device time, max over ranks
    ms_max = max_over_ranks(ms, world, dev)
    value = job_rate(STEP_FLOP, world, ms_max) / 1e12

    # quantize-only throughput (x, W, dy: amax pass + fused row/col pass)
    q_ms = time_quantize(nvq, x, w, dy, sign, sr, fwd_bufs, bwd_bufs, stream)

    e2e = measure_e2e(args, nvq, x_h, w_h, dy_h, sign, sr, dev, stream, world) if not args.no_e2e else None

    if rank != 0:
        return 0
    peaks, src = _peaks()
    # The GEMM launch times come from a short eager pass (a few ms of GEMMs between
    # idle gaps), not from a seconds-long loop, so the burst bf16 figure applies.
    peak_fp4 = peaks["bf16_tflops"] * FP4_OVER_BF16
    achieved = GEMM_FLOP / (avg_gemm_ms * 1e-3) / 1e12
    q_bytes = (M * K + N * K + M * N) * 5.125  # 2 reads of bf16 + 2 x (codes + scales) writes
    q_gbs = q_bytes / (q_ms * 1e-3) / 1e9
    st_v, st_desc = None, "not measured"
    if args.no_cpu_baseline:
        cpu_v, cpu_desc, cpu_threads = None, "skipped (--no-cpu-baseline)", 0
    elif world > 1:
        cpu_v, cpu_desc, cpu_threads = None, "measured at N=1 only", 0
    else:
        cpu_v, cpu_desc, cpu_threads, _ = oracle_sample(x_h, w_h, dy_h, sign)
        st_v, st_desc = oracle_single_thread()
    # which GEMM kernel ran: the CTA pair unless the library fell back to the single-CTA kernel
    pair = nvq.gemm_pair_available()
    gemm_label = ("gemm_pair_kernel<NVFP4> (CTA pair; fwd, dgrad, wgrad)" if pair
                  else "gemm_kernel<NVFP4> (single CTA; fwd, dgrad, wgrad)")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4", "data": "synthetic", "config": CONFIG,
        "gpu_launches": 9 * args.steps,
        "launch_mode": "eager" if args.eager else "cuda_graph",
        "step_schedule": "one stream" if (args.eager or args.serial_step) else
                         "two streams: x / W quantization, then dgrad / wgrad, side by side",
        "roofline": {"bound": "tensor", "kernel": gemm_label,
                     "achieved": achieved, "peak": peak_fp4, "unit": "TFLOP/s", "frac": achieved / peak_fp4,
                     "traffic": GEMM_TRAFFIC_BYTES if pair else None,
                     "traffic_note": "bytes per launch, ncu capture of the forward GEMM (CTA-pair kernel)",
                     "peak_note": f"{src} bf16 burst x {FP4_OVER_BF16} (fp4/bf16 nominal dense ratio); the GEMMs "
                                  "are timed in a short eager pass, so the burst figure applies",
                     "frac_of_sustained": achieved / (peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
                                                      * FP4_OVER_BF16)},
        "roofline_quantize": {"bound": "hbm", "achieved": q_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                              "frac": q_gbs / peaks["hbm_gbs"], "traffic": QUANT_TRAFFIC_BYTES,
                              "traffic_note": "bytes per step (x, W, dy amax + quantize), ncu captures",
                              "algorithmic_bytes": q_bytes, "peak_note": f"{src} HBM copy"},
        "breakdown_ms": {"step": ms_max, "gemm_fwd": statistics.mean(gemm_ms), "gemm_dgrad": statistics.mean(dgrad_ms),
                         "gemm_wgrad": statistics.mean(wgrad_ms), "quantize_x_w_dy": q_ms},
        "clocks": clk,
        "cpu_baseline": {"value": cpu_v, "unit": UNIT, "cores": cpu_threads, "kind": "oracle", "sample": cpu_desc,
                         "extrapolated": cpu_v is not None,
                         "single_thread": {"value": st_v, "unit": UNIT, "cores": 1, "sample": st_desc,
                                           "extrapolated": st_v is not None}},
        "e2e": e2e,
    }
    print(json.dumps(line), flush=True)
    return 0


def time_quantize(nvq, x, w, dy, sign, sr, fb, bb, stream, reps=5):
    import torch
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(reps):
        nvq.nvfp4_quantize(x, 3, rht_sign=sign, out_row=fb["x_row"], out_col=fb["x_col"])
        nvq.nvfp4_quantize(w, 3, out_row=fb["w_row"], out_col=fb["w_col"])
        nvq.nvfp4_linear_bwd_quantize(dy, rht_sign=sign, sr=sr, bufs=bb)
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / reps


def max_over_ranks(ms: float, world: int, device="cpu") -> float:
    """The job's step time: the slowest replica's (all-reduce MAX over ranks)."""
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job throughput: every replica processes units_per_rank per step
    (weak scaling), the job advances one step per ms_max."""
    return world * units_per_rank / (ms_max * 1e-3)


def measure_e2e(args, nvq, x_h, w_h, dy_h, sign, sr, dev, stream, world):
    """Same step through the public linear API with host buffers: every step
    copies its inputs x, W, dy from pinned host memory to the device and reads
    its results y, dx, dW back, all inside the timed region.  Steps are
    pipelined over two device buffer sets and three streams (copy-in, compute,
    copy-out), so step i+1's uploads and step i's downloads overlap compute."""
    import torch
    xh, wh, dyh = x_h.pin_memory(), w_h.pin_memory(), dy_h.pin_memory()
    outs_h = [(torch.empty(M, N, dtype=torch.bfloat16).pin_memory(),
               torch.empty(M, K, dtype=torch.bfloat16).pin_memory(),
               torch.empty(N, K, dtype=torch.bfloat16).pin_memory()) for _ in range(2)]
    sets = []
    for _ in range(2):
        sets.append(dict(x=torch.empty_like(xh, device=dev), w=torch.empty_like(wh, device=dev),
                         dy=torch.empty_like(dyh, device=dev),
                         y=torch.empty(M, N, dtype=torch.bfloat16, device=dev),
                         dx=torch.empty(M, K, dtype=torch.bfloat16, device=dev),
                         dw=torch.empty(N, K, dtype=torch.bfloat16, device=dev), fb=None, bb=None))
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_ready = [ev(), ev()]
    comp_done = [ev(), ev()]
    out_done = [ev(), ev()]
    used = [False, False]

    def step(i):
        b = i & 1
        d = sets[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(comp_done[b])  # the previous step on this set has read its inputs
            d["x"].copy_(xh, non_blocking=True)
            d["w"].copy_(wh, non_blocking=True)
            d["dy"].copy_(dyh, non_blocking=True)
            in_ready[b].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(in_ready[b])
            if used[b]:
                s_comp.wait_event(out_done[b])  # its results have been read back
            _, d["fb"] = nvq.nvfp4_linear_fwd(d["x"], d["w"], rht_sign=sign, y=d["y"], bufs=d["fb"], stream=s_comp)
            d["bb"] = nvq.nvfp4_linear_bwd_quantize(d["dy"], rht_sign=sign, sr=sr, bufs=d["bb"], stream=s_comp)
            nvq.nvfp4_linear_dgrad(d["bb"]["dy_row"], d["fb"]["w_col"], dx=d["dx"], stream=s_comp)
            nvq.nvfp4_linear_wgrad(d["bb"]["dy_col"], d["fb"]["x_col"], dw=d["dw"], stream=s_comp)
            comp_done[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            yh, dxh, dwh = outs_h[b]
            yh.copy_(d["y"], non_blocking=True)
            dxh.copy_(d["dx"], non_blocking=True)
            dwh.copy_(d["dw"], non_blocking=True)
            out_done[b].record(s_out)
        used[b] = True

    for i in range(max(2, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    steps = max(2, min(args.steps, 10))
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    s_comp.wait_event(t0)
    s_out.wait_event(t0)
    for i in range(steps):
        step(i)
    s_in.wait_stream(s_out)
    s_in.wait_stream(s_comp)
    t1.record(s_in)
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1) / steps, world, dev)
    bi = (M * K + N * K + M * N) * 2
    bo = (M * N + M * K + N * K) * 2
    return {"value": job_rate(STEP_FLOP, world, ms) / 1e12, "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "api": "nvq_nvfp4_linear_fwd / _bwd_quantize / _dgrad / _wgrad with pinned host buffers; "
                   "copy-in, compute and copy-out streams over two buffer sets"}


# ---------------------------------------------------------------- other workloads
def _side_by_side(side, fa, fb):
    """fa(stream) on the current stream and fb(stream) on `side`, forked from and
    joined back into the current stream with events (captured as such inside a
    CUDA graph)."""
    import torch
    cur = torch.cuda.current_stream()
    fork = torch.cuda.Event()
    fork.record(cur)
    side.wait_event(fork)
    fa(cur)
    fb(side)
    join = torch.cuda.Event()
    join.record(side)
    cur.wait_event(join)


def _graph_ms(fn, steps, warmup, eager=False):
    """Warm up, capture fn into a CUDA graph and replay it `steps` times between
    CUDA events on the current stream; ms per replay."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    g = None
    if not eager:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        for _ in range(warmup):
            g.replay()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s)
    for _ in range(steps):
        g.replay() if g is not None else fn()
    t1.record(s)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps


def _flushed_ms(fn, reps, warmup):
    """Per-call time with L2 flushed (a 512 MB write) before every timed call:
    for inputs that fit in L2.  The call itself is replayed from a CUDA graph."""
    import torch
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    tot = 0.0
    for _ in range(reps):
        flush.fill_(1)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s)
        g.replay()
        t1.record(s)
        torch.cuda.synchronize()
        tot += t0.elapsed_time(t1)
    return tot / reps


def run_quant_sweep(args, nvq, inputs):
    """Standalone quantize sweep: [M,4096] 0.1*t(3) with outlier channels,
    M in {2048, 8192, 32768, 131072}; NVFP4 row+col (RTN), NVFP4 row+col with
    RHT (col) and SR, MXFP8 row+col.  Algorithmic bytes: NVFP4 2 reads + 2 x
    (0.5 + 1/16) B written per element = 5.125 B; MXFP8 2 + 2 x (1 + 1/32) =
    4.0625 B.  Inputs below 129 MB are timed with L2 flushed before each call."""
    import torch
    sign = inputs.rht_sign_vector()
    sr = (inputs.SR_SEED, 0)
    entries, tot_b, tot_ms = [], 0.0, 0.0
    for Mq in inputs.QUANT_SWEEP_M:
        x = inputs.student_t3_outliers(Mq).cuda()
        Kq = x.shape[1]
        nr = nvq.alloc_qtensor(nvq.NVFP4, Mq, Kq)
        nc = nvq.alloc_qtensor(nvq.NVFP4, Kq, nvq.colwise_cols(nvq.NVFP4, Mq))
        mr = nvq.alloc_qtensor(nvq.MXFP8, Mq, Kq)
        mc = nvq.alloc_qtensor(nvq.MXFP8, Kq, nvq.colwise_cols(nvq.MXFP8, Mq))
        variants = [
            ("nvfp4_rtn", 5.125, lambda: nvq.nvfp4_quantize(x, 3, out_row=nr, out_col=nc)),
            ("nvfp4_rht_sr", 5.125, lambda: nvq.nvfp4_quantize(x, 3, rht_sign=sign, sr=sr, out_row=nr, out_col=nc)),
            ("mxfp8", 4.0625, lambda: nvq.mxfp8_quantize(x, 3, out_row=mr, out_col=mc)),
        ]
        for name, bpe, fn in variants:
            small = Mq * Kq * 2 < 129e6
            ms = _flushed_ms(fn, max(5, args.steps), args.warmup) if small else _graph_ms(fn, args.steps, args.warmup)
            b = Mq * Kq * bpe
            entries.append({"M": Mq, "variant": name, "ms": ms, "GB/s": b / (ms * 1e-3) / 1e9,
                            "l2": "flushed" if small else "inputs larger than L2"})
            tot_b += b
            tot_ms += ms
        del x, nr, nc, mr, mc
        torch.cuda.empty_cache()
    value = tot_b / (tot_ms * 1e-3) / 1e9
    line = {"metric": "quantize sweep GB/s (algorithmic bytes, NVFP4 RTN / RHT+SR / MXFP8, row+col)",
            "value": value, "unit": "GB/s", "ms_per_step": tot_ms, "dtype": "bf16 -> nvfp4 / mxfp8",
            "config": {"workload": "quantize_sweep_Mx4096_student_t3", "M": list(inputs.QUANT_SWEEP_M), "K": 4096},
            "sweep": entries, "roofline_bound": "hbm", "step_bytes": tot_b}
    if not args.no_cpu_baseline:
        # the oracle on the full sweep tensors with every host core, and with
        # one thread (a child process) on the smallest tensor
        cpu_v, cpu_s = oracle_sweep_rate(inputs.QUANT_SWEEP_M)
        threads = _env_int("OMP_NUM_THREADS", os.cpu_count() or 1)
        st_v, st_desc = oracle_single_thread(-1.0)
        line["cpu_baseline"] = {
            "value": cpu_v, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"the full sweep tensors (M = {list(inputs.QUANT_SWEEP_M)}, three variants), measured {cpu_s:.1f} s",
            "extrapolated": False,
            "single_thread": {"value": st_v, "unit": "GB/s", "cores": 1, "sample": st_desc, "extrapolated": False}}
    return line


def run_moe_grouped(args, nvq, inputs):
    """64 experts 4096->1536, 65536 Zipf(1.1) tokens: grouped hybrid quantize of
    x (NVFP4 row + MXFP8 col), W (NVFP4 row + MXFP8 col), dy (MXFP8 row + col);
    grouped NVFP4 forward, MXFP8 dgrad and wgrad (3 x 2*65536*1536*4096 FLOP)."""
    import torch
    sizes, x, w, dy = inputs.moe_grouped()
    sizes = [int(v) for v in sizes]
    G, Nn, Kk = w.shape
    x, dy = x.cuda(), dy.cuda()
    w2 = w.reshape(G * Nn, Kk).cuda()
    del w
    P = nvq.grouped_padded_rows(sizes)
    xr = nvq.alloc_qtensor(nvq.NVFP4, P, Kk, n_amax=G); xc = nvq.alloc_qtensor(nvq.MXFP8, Kk, P)
    wr = nvq.alloc_qtensor(nvq.NVFP4, G * Nn, Kk, n_amax=G); wc = nvq.alloc_qtensor(nvq.MXFP8, Kk, G * Nn)
    dr = nvq.alloc_qtensor(nvq.MXFP8, P, Nn); dc = nvq.alloc_qtensor(nvq.MXFP8, Nn, P)
    T = sum(sizes)
    y = torch.empty(T, Nn, dtype=torch.bfloat16, device="cuda")
    dx = torch.empty(T, Kk, dtype=torch.bfloat16, device="cuda")
    dwt = torch.empty(G, Nn, Kk, dtype=torch.bfloat16, device="cuda")

    def step():
        nvq.grouped_hybrid_quantize(x, sizes, nvq.NVFP4, nvq.MXFP8, out_row=xr, out_col=xc)
        nvq.grouped_hybrid_quantize(w2, [Nn] * G, nvq.NVFP4, nvq.MXFP8, out_row=wr, out_col=wc)
        nvq.grouped_gemm_rows(xr, wr, sizes, Nn, b_col_groups=False, out=y)
        nvq.grouped_hybrid_quantize(dy, sizes, nvq.MXFP8, nvq.MXFP8, out_row=dr, out_col=dc)
        nvq.grouped_gemm_rows(dr, wc, sizes, Nn, b_col_groups=True, out=dx)
        nvq.grouped_gemm_wgrad(dc, xc, sizes, out=dwt)

    side = torch.cuda.Stream()

    def step_overlapped():
        # the same calls; x / W quantization and dgrad / wgrad side by side
        _side_by_side(side, lambda s: nvq.grouped_hybrid_quantize(x, sizes, nvq.NVFP4, nvq.MXFP8, out_row=xr,
                                                                  out_col=xc, stream=s),
                      lambda s: nvq.grouped_hybrid_quantize(w2, [Nn] * G, nvq.NVFP4, nvq.MXFP8, out_row=wr,
                                                            out_col=wc, stream=s))
        nvq.grouped_gemm_rows(xr, wr, sizes, Nn, b_col_groups=False, out=y)
        nvq.grouped_hybrid_quantize(dy, sizes, nvq.MXFP8, nvq.MXFP8, out_row=dr, out_col=dc)
        _side_by_side(side, lambda s: nvq.grouped_gemm_rows(dr, wc, sizes, Nn, b_col_groups=True, out=dx, stream=s),
                      lambda s: nvq.grouped_gemm_wgrad(dc, xc, sizes, out=dwt, stream=s))

    serial = args.eager or args.serial_step
    ms = _graph_ms(step if serial else step_overlapped, args.steps, args.warmup, args.eager)
    flop = 3 * 2.0 * T * Nn * Kk

    # per-phase times from an eager pass with events between the calls
    names = ["quant_x", "quant_w", "gemm_fwd_nvfp4", "quant_dy", "gemm_dgrad_mxfp8", "gemm_wgrad_mxfp8"]
    calls = [lambda: nvq.grouped_hybrid_quantize(x, sizes, nvq.NVFP4, nvq.MXFP8, out_row=xr, out_col=xc),
             lambda: nvq.grouped_hybrid_quantize(w2, [Nn] * G, nvq.NVFP4, nvq.MXFP8, out_row=wr, out_col=wc),
             lambda: nvq.grouped_gemm_rows(xr, wr, sizes, Nn, b_col_groups=False, out=y),
             lambda: nvq.grouped_hybrid_quantize(dy, sizes, nvq.MXFP8, nvq.MXFP8, out_row=dr, out_col=dc),
             lambda: nvq.grouped_gemm_rows(dr, wc, sizes, Nn, b_col_groups=True, out=dx),
             lambda: nvq.grouped_gemm_wgrad(dc, xc, sizes, out=dwt)]
    acc = [0.0] * len(calls)
    reps = 5
    for _ in range(reps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
        ev[0].record()
        for i, c in enumerate(calls):
            c()
            ev[i + 1].record()
        torch.cuda.synchronize()
        for i in range(len(calls)):
            acc[i] += ev[i].elapsed_time(ev[i + 1]) / reps
    breakdown = dict(zip(names, acc))
    peaks, _src = _peaks()
    gemm_flop = 2.0 * T * Nn * Kk
    # the per-GEMM times come from a short eager pass, so the burst figure applies
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    fp8_peak = peaks["bf16_tflops"] * 2.0
    rates = {"gemm_fwd_nvfp4": gemm_flop / (acc[2] * 1e-3) / 1e12, "gemm_dgrad_mxfp8": gemm_flop / (acc[4] * 1e-3) / 1e12,
             "gemm_wgrad_mxfp8": gemm_flop / (acc[5] * 1e-3) / 1e12}
    return {"metric": "MoE grouped hybrid linear fwd+dgrad+wgrad TFLOP/s (64 experts 4096->1536)",
            "value": flop / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "breakdown_ms_eager": breakdown,
            "gemm_tflops": rates,
            "gemm_frac": {"gemm_fwd_nvfp4": rates["gemm_fwd_nvfp4"] / fp4_peak,
                          "gemm_dgrad_mxfp8": rates["gemm_dgrad_mxfp8"] / fp8_peak,
                          "gemm_wgrad_mxfp8": rates["gemm_wgrad_mxfp8"] / fp8_peak},
            "peak_note": "FP4 = measured bf16 burst x 6, FP8 = x 2 (nominal dense ratios); GEMM FLOPs count "
                         "unpadded tokens",
            "step_schedule": "one stream" if serial else "two streams: x / W quantization, then dgrad / wgrad, "
                                                         "side by side",
            "dtype": "nvfp4 fwd / mxfp8 bwd",
            "config": {"workload": "moe_grouped_64x4096x1536_zipf1.1", "tokens": T, "experts": G,
                       "group_sizes_min_max": [min(sizes), max(sizes)], "padded_rows": P},
            "gpu_launches_per_step": 9}


def run_qwen3_stack(args, nvq, inputs):
    """Qwen3-8B-shaped linear stack: 36 layers, 16384 tokens; layers 0-29 NVFP4
    (RHT on wgrad operands, SR on dy), layers 30-35 and the 151936x4096 lm_head
    in bf16 (torch.matmul).  Attention core, norms and activations are not on
    the path: the o input is the q output, the down input the up output.
    FLOPs per step = 6 x tokens x parameters.

    With the amax chain (the default; --no-amax-chain turns it off), the q and
    up GEMMs also write their outputs' amaxes (plain and Hadamard-domain) into
    the o and down input buffers, whose quantization then skips its amax pass."""
    import torch
    cfg = inputs.QWEN3_8B_STACK
    chain = not args.no_amax_chain
    Tk, H = cfg["tokens"], cfg["hidden"]
    n_nv = cfg["n_layers"] - cfg["bf16_tail"]
    sign = inputs.rht_sign_vector()
    sr = (inputs.SR_SEED, 0)
    cc = nvq.colwise_cols
    al = nvq.alloc_qtensor
    h = inputs.normal_bf16_on((Tk, H), 1.0, 1, "cuda")
    layers = []
    params = 0
    for l in range(cfg["n_layers"]):
        ws = dict(inputs.qwen3_layer_weights(l, device="cuda"))
        params += sum(t.numel() for t in ws.values())
        layers.append(ws)
    lm_head = inputs.normal_bf16_on((cfg["vocab"], H), 0.02, 3, "cuda")
    params += lm_head.numel()
    dys = {n: inputs.normal_bf16_on((Tk, n), 0.01, 2, "cuda") for n in {H, cfg["kv_dim"], cfg["mlp"]}}
    dlog = inputs.normal_bf16_on((Tk, cfg["vocab"]), 0.01, 4, "cuda")

    # per NVFP4 layer: quantized weights (row + col), saved activations (col), outputs
    st = []
    for l in range(n_nv):
        ws = layers[l]
        e = {"w": {}, "y": {}}
        for n, W in ws.items():
            No, Ki = W.shape
            e["w"][n] = (al(nvq.NVFP4, No, Ki), al(nvq.NVFP4, Ki, cc(nvq.NVFP4, No)))
            e["y"][n] = torch.empty(Tk, No, dtype=torch.bfloat16, device="cuda")
        e["a"] = {k: (al(nvq.NVFP4, Tk, d), al(nvq.NVFP4, d, cc(nvq.NVFP4, Tk)))
                  for k, d in (("h", H), ("attn", H), ("mlp", cfg["mlp"]))}
        st.append(e)
    bw = {d: dict(dy_row=al(nvq.NVFP4, Tk, d), dy_col=al(nvq.NVFP4, d, cc(nvq.NVFP4, Tk)))
          for d in {H, cfg["kv_dim"], cfg["mlp"]}}
    dxb = {d: torch.empty(Tk, d, dtype=torch.bfloat16, device="cuda") for d in (H, cfg["mlp"])}
    dwb = {n: torch.empty_like(W) for n, W in layers[0].items()}
    src = {"q": "h", "k": "h", "v": "h", "gate": "h", "up": "h", "o": "attn", "down": "mlp"}
    side = torch.cuda.Stream()
    overlap = not (args.eager or args.serial_step)

    def step():
        # the NVFP4 layers' weights are known at the start of the step: with the
        # overlapped schedule they are quantized on the side stream, in layer
        # order, and each layer's GEMMs wait only for that layer's weights
        w_ready = []
        if overlap:
            cur = torch.cuda.current_stream()
            fork = torch.cuda.Event()
            fork.record(cur)
            side.wait_event(fork)
            for l in range(n_nv):
                for n in ("q", "k", "v", "gate", "up", "o", "down"):
                    wr, wc = st[l]["w"][n]
                    nvq.nvfp4_quantize(layers[l][n], 3, out_row=wr, out_col=wc, stream=side)
                ev = torch.cuda.Event()
                ev.record(side)
                w_ready.append(ev)
        # forward
        for l in range(n_nv):
            e, ws = st[l], layers[l]
            if overlap:
                torch.cuda.current_stream().wait_event(w_ready[l])
            nvq.nvfp4_quantize(h, 3, rht_sign=sign, out_row=e["a"]["h"][0], out_col=e["a"]["h"][1])
            for n in ("q", "k", "v", "gate", "up", "o", "down"):
                if n == "o":
                    nvq.nvfp4_quantize(e["y"]["q"], 3, rht_sign=sign, out_row=e["a"]["attn"][0], out_col=e["a"]["attn"][1],
                                       amax_given=chain)
                if n == "down":
                    nvq.nvfp4_quantize(e["y"]["up"], 3, rht_sign=sign, out_row=e["a"]["mlp"][0], out_col=e["a"]["mlp"][1],
                                       amax_given=chain)
                wr, wc = e["w"][n]
                if not overlap:
                    nvq.nvfp4_quantize(ws[n], 3, out_row=wr, out_col=wc)
                nxt = {"q": "attn", "up": "mlp"}.get(n) if chain else None
                if nxt:  # the output's amaxes go straight into its consumer's quantized buffers
                    nvq.gemm_tn(e["a"][src[n]][0], wr, out=e["y"][n], rht_sign=sign, amax_out=e["a"][nxt][0].amax,
                                amax_rht_out=e["a"][nxt][1].amax)
                else:
                    nvq.gemm_tn(e["a"][src[n]][0], wr, out=e["y"][n])
        tail = [torch.matmul(h if W.shape[1] == H else dys[cfg["mlp"]], W.t())
                for l in range(n_nv, cfg["n_layers"]) for W in layers[l].values()]
        logits = torch.matmul(h, lm_head.t())
        # backward (reverse order)
        torch.matmul(dlog, lm_head)
        torch.matmul(dlog.t(), h)
        for l in range(cfg["n_layers"] - 1, n_nv - 1, -1):
            for n, W in layers[l].items():
                d = dys[W.shape[0]]
                xin = h if W.shape[1] == H else dys[cfg["mlp"]]
                torch.matmul(d, W)
                torch.matmul(d.t(), xin)
        for l in range(n_nv - 1, -1, -1):
            e = st[l]
            for n in ("down", "o", "up", "gate", "v", "k", "q"):
                No = layers[l][n].shape[0]
                b = nvq.nvfp4_linear_bwd_quantize(dys[No], rht_sign=sign, sr=sr, bufs=bw[No])
                wr, wc = e["w"][n]
                dgrad = lambda s: nvq.nvfp4_linear_dgrad(b["dy_row"], wc, dx=dxb[layers[l][n].shape[1]], stream=s)
                wgrad = lambda s: nvq.nvfp4_linear_wgrad(b["dy_col"], e["a"][src[n]][1], dw=dwb[n], stream=s)
                if overlap:  # dgrad and wgrad (disjoint operands) side by side
                    _side_by_side(side, dgrad, wgrad)
                else:
                    dgrad(None)
                    wgrad(None)
        del tail, logits

    steps = max(2, min(args.steps, 5))
    ms = _graph_ms(step, steps, min(args.warmup, 3), args.eager)
    flop = 6.0 * Tk * params
    return {"metric": "Qwen3-8B-shaped 36-layer linear stack fwd+bwd TFLOP/s (30 NVFP4 + 6 bf16 layers + bf16 lm_head)",
            "value": flop / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "dtype": "nvfp4 (layers 0-29) / bf16 (tail, lm_head)",
            "config": {"workload": "qwen3_8b_linear_stack", "tokens": Tk, "layers": cfg["n_layers"],
                       "nvfp4_layers": n_nv, "params": params,
                       "amax_chain": "q -> o and up -> down: GEMM epilogue amaxes, no amax pass" if chain else "off",
                       "step_schedule": "weights quantized ahead on a second stream; each NVFP4 linear's dgrad / "
                                        "wgrad on two streams" if overlap else "one stream"},
            "tokens_per_s": Tk / (ms * 1e-3)}


def run_variants(args, nvq, inputs):
    """The recipe variants beside the base paths they extend, at the Llama-3-8B
    up-projection shapes (x[16384,4096], W[14336,4096]) and the MoE workload:

      amax_chain   forward GEMM with and without its output amaxes (plain + Hadamard
                   domain) in the epilogue; x's quantization with the amax given vs measured
      dequant_src  x: NVFP4 rows with an MXFP8 / NVFP4 / identity columnwise direction built
                   from the dequantized rowwise value (columnwise_source = rowwise_dequantized)
      row_scaled   MoE x[65536,4096]: row-scaled NVFP4 rows + MXFP8 columns, and the grouped
                   forward GEMM with a row-scaled A vs a per-group-scaled A
      two_d        W: MXFP8 rows + NVFP4 columns with 16x16 tile scales vs 1x16 blocks
      hybrid_linear  MXFP8 forward + NVFP4 backward step (W columns 2D) vs the NVFP4 step
      grouped_nvfp4_bwd  MoE workload, NVFP4 backward: dy rows + columns with SR (columns with
                   RHT), x and W columns (x with RHT), grouped NVFP4 dgrad and wgrad

    Quantize rates are algorithmic bytes (each pass's bf16 read + the outputs written) per
    second; GEMM / step rates are FLOPs per second.  Inputs above L2 are timed back to back
    from a CUDA graph, those below it with L2 flushed before each call."""
    import torch
    sign = inputs.rht_sign_vector()
    sr = (inputs.SR_SEED, 0)
    Mq, Nq, Kq = inputs.LLAMA3_8B_UP["M"], inputs.LLAMA3_8B_UP["N"], inputs.LLAMA3_8B_UP["K"]
    xh, wh, dyh = inputs.llama_up()
    x, w, dy = xh.cuda(), wh.cuda(), dyh.cuda()
    del xh, wh, dyh
    al, cc = nvq.alloc_qtensor, nvq.colwise_cols
    out = {}

    def timed(fn, nbytes_in):
        small = nbytes_in < 129e6
        return _flushed_ms(fn, max(5, args.steps), args.warmup) if small else _graph_ms(fn, args.steps, args.warmup)

    def gbs(b, ms):
        return b / (ms * 1e-3) / 1e9

    ex = Mq * Kq
    # ---- f-1: the amax produced upstream
    xr, xcol = al(nvq.NVFP4, Mq, Kq), al(nvq.NVFP4, Kq, cc(nvq.NVFP4, Mq))
    wr = al(nvq.NVFP4, Nq, Kq)
    nvq.nvfp4_quantize(x, 3, rht_sign=sign, out_row=xr, out_col=xcol)
    nvq.nvfp4_quantize(w, nvq.DIR_ROW, out_row=wr)
    y = torch.empty(Mq, Nq, dtype=torch.bfloat16, device="cuda")
    a1, a2 = torch.empty(1, device="cuda"), torch.empty(1, device="cuda")
    gflop = 2.0 * Mq * Nq * Kq
    t_plain = timed(lambda: nvq.gemm_tn(xr, wr, out=y), 1e12)
    t_amax = timed(lambda: nvq.gemm_tn(xr, wr, out=y, rht_sign=sign, amax_out=a1, amax_rht_out=a2), 1e12)
    t_meas = timed(lambda: nvq.nvfp4_quantize(x, 3, rht_sign=sign, out_row=xr, out_col=xcol), ex * 2)
    t_given = timed(lambda: nvq.nvfp4_quantize(x, 3, rht_sign=sign, out_row=xr, out_col=xcol, amax_given=True), ex * 2)
    out["amax_chain"] = {
        "gemm_fwd_ms": t_plain, "gemm_fwd_with_output_amaxes_ms": t_amax,
        "gemm_tflops": gflop / (t_plain * 1e-3) / 1e12, "gemm_with_amax_tflops": gflop / (t_amax * 1e-3) / 1e12,
        "x_quantize_measured_amax_ms": t_meas, "x_quantize_given_amax_ms": t_given,
        "x_quantize_measured_gbs": gbs(ex * 5.125, t_meas), "x_quantize_given_gbs": gbs(ex * 3.125, t_given),
        "bytes_per_element": {"measured": 5.125, "given": 3.125}}
    # ---- f-2: rowwise-dequantized source
    dq = nvq.COL_SOURCE_ROWWISE_DEQUANTIZED
    cols = {nvq.MXFP8: al(nvq.MXFP8, Kq, cc(nvq.MXFP8, Mq)), nvq.NVFP4: xcol,
            nvq.IDENTITY: al(nvq.IDENTITY, Kq, cc(nvq.IDENTITY, Mq))}
    bpe = {nvq.MXFP8: 2 + 2 + 0.5625 + 1.03125, nvq.NVFP4: 2 + 2 + 2 + 0.5625 + 0.5625,
           nvq.IDENTITY: 2 + 2 + 0.5625 + 2.0}
    names = {nvq.MXFP8: "nvfp4_row_mxfp8_col", nvq.NVFP4: "nvfp4_row_nvfp4_col", nvq.IDENTITY: "nvfp4_row_identity_col"}
    d = {}
    for cf, q in cols.items():
        t = timed(lambda q=q, cf=cf: nvq.hybrid_quantize(x, nvq.NVFP4, cf, out_row=xr, out_col=q, col_source=dq), ex * 2)
        d[names[cf]] = {"ms": t, "GB/s": gbs(ex * bpe[cf], t), "bytes_per_element": bpe[cf]}
    t = timed(lambda: nvq.hybrid_quantize(x, nvq.NVFP4, nvq.MXFP8, out_row=xr, out_col=cols[nvq.MXFP8]), ex * 2)
    d["original_source_nvfp4_row_mxfp8_col"] = {"ms": t, "GB/s": gbs(ex * bpe[nvq.MXFP8], t)}
    out["dequant_src"] = d
    del cols
    # ---- f-4: 2D columnwise scaling of W, and the hybrid-format linear step
    ew = Nq * Kq
    wrm, wc2 = al(nvq.MXFP8, Nq, Kq), al(nvq.NVFP4, Kq, cc(nvq.NVFP4, Nq))
    b2d = 2 + 2 + 1.03125 + 0.5625
    t2 = timed(lambda: nvq.hybrid_quantize(w, nvq.MXFP8, nvq.NVFP4, out_row=wrm, out_col=wc2, col_2d=True), ew * 2)
    t1 = timed(lambda: nvq.hybrid_quantize(w, nvq.MXFP8, nvq.NVFP4, out_row=wrm, out_col=wc2), ew * 2)
    out["two_d"] = {"w_mxfp8_row_nvfp4_2d_col": {"ms": t2, "GB/s": gbs(ew * b2d, t2)},
                    "w_mxfp8_row_nvfp4_1d_col": {"ms": t1, "GB/s": gbs(ew * b2d, t1)}, "bytes_per_element": b2d}
    del wrm, wc2
    ybuf = torch.empty(Mq, Nq, dtype=torch.bfloat16, device="cuda")
    dxb = torch.empty(Mq, Kq, dtype=torch.bfloat16, device="cuda")
    dwb = torch.empty(Nq, Kq, dtype=torch.bfloat16, device="cuda")
    hb = {}

    def hstep():
        _, hb["f"] = nvq.hybrid_linear_fwd(x, w, nvq.MXFP8, nvq.NVFP4, rht_sign=sign, w_col_2d=True, y=ybuf,
                                           bufs=hb.get("f"))
        hb["b"] = nvq.hybrid_linear_bwd_quantize(dy, nvq.NVFP4, rht_sign=sign, sr=sr, bufs=hb.get("b"))
        nvq.linear_dgrad(hb["b"]["dy_row"], hb["f"]["w_col"], dx=dxb)
        nvq.linear_wgrad(hb["b"]["dy_col"], hb["f"]["x_col"], dw=dwb)

    hstep()
    th = _graph_ms(hstep, args.steps, args.warmup)
    out["hybrid_linear"] = {"mxfp8_fwd_nvfp4_bwd_step_ms": th, "TFLOP/s": 3 * gflop / (th * 1e-3) / 1e12,
                            "note": "x, W MXFP8 rows + NVFP4 columns (x RHT, W 2D), dy NVFP4 SR + RHT; fwd MXFP8 GEMM, "
                                    "dgrad / wgrad NVFP4"}
    del hb, ybuf, dxb, dwb, y, x, w, dy, xr, xcol, wr
    torch.cuda.empty_cache()
    # ---- f-3: row-scaled NVFP4 on the MoE workload
    sizes, xm, wm, dyh_m = inputs.moe_grouped()
    sizes = [int(v) for v in sizes]
    G, Nn, Km = wm.shape
    xm = xm.cuda()
    w2 = wm.reshape(G * Nn, Km).cuda()
    del wm
    P = nvq.grouped_padded_rows(sizes)
    T = sum(sizes)
    xrs, xrp = al(nvq.NVFP4_ROWSCALED, P, Km), al(nvq.NVFP4, P, Km, n_amax=G)
    xcm = al(nvq.MXFP8, Km, P)
    wrg, _ = nvq.grouped_hybrid_quantize(w2, [Nn] * G, nvq.NVFP4, nvq.NONE)
    ym = torch.empty(T, Nn, dtype=torch.bfloat16, device="cuda")
    em = T * Km
    brs = 2 + 2 + 0.5625 + 1.03125
    trs = timed(lambda: nvq.grouped_hybrid_quantize(xm, sizes, nvq.NVFP4_ROWSCALED, nvq.MXFP8, out_row=xrs, out_col=xcm),
                em * 2)
    tpg = timed(lambda: nvq.grouped_hybrid_quantize(xm, sizes, nvq.NVFP4, nvq.MXFP8, out_row=xrp, out_col=xcm), em * 2)
    mflop = 2.0 * T * Nn * Km
    tgr = timed(lambda: nvq.grouped_gemm_rows(xrs, wrg, sizes, Nn, b_col_groups=False, out=ym), 1e12)
    tgp = timed(lambda: nvq.grouped_gemm_rows(xrp, wrg, sizes, Nn, b_col_groups=False, out=ym), 1e12)
    out["row_scaled"] = {"x_quantize_row_scaled_ms": trs, "x_quantize_row_scaled_GB/s": gbs(em * brs, trs),
                         "x_quantize_per_group_ms": tpg, "x_quantize_per_group_GB/s": gbs(em * brs, tpg),
                         "grouped_fwd_row_scaled_ms": tgr, "grouped_fwd_row_scaled_TFLOP/s": mflop / (tgr * 1e-3) / 1e12,
                         "grouped_fwd_per_group_ms": tgp, "grouped_fwd_per_group_TFLOP/s": mflop / (tgp * 1e-3) / 1e12,
                         "bytes_per_element": brs}
    del xrs, xrp, xcm, wrg, ym
    torch.cuda.empty_cache()
    # ---- grouped NVFP4 backward on the MoE workload
    dym = dyh_m.cuda()
    del dyh_m
    dyr, dyc = al(nvq.NVFP4, P, Nn, n_amax=G), al(nvq.NVFP4, Nn, P, n_amax=G)
    xcn, wcn = al(nvq.NVFP4, Km, P, n_amax=G), al(nvq.NVFP4, Km, G * Nn, n_amax=G)
    dxm = torch.empty(T, Km, dtype=torch.bfloat16, device="cuda")
    dwm = torch.empty(G, Nn, Km, dtype=torch.bfloat16, device="cuda")

    def q_dy():
        nvq.grouped_hybrid_quantize(dym, sizes, nvq.NVFP4, nvq.NVFP4, out_row=dyr, out_col=dyc, rht_sign=sign, sr=sr)

    def q_x():
        nvq.grouped_hybrid_quantize(xm, sizes, nvq.NONE, nvq.NVFP4, out_col=xcn, rht_sign=sign)

    def q_w():
        nvq.grouped_hybrid_quantize(w2, [Nn] * G, nvq.NONE, nvq.NVFP4, out_col=wcn)

    def dgrad():
        nvq.grouped_gemm_rows(dyr, wcn, sizes, Nn, b_col_groups=True, out=dxm)

    def wgrad():
        nvq.grouped_gemm_wgrad(dyc, xcn, sizes, out=dwm)

    def bwd():
        q_dy(); q_x(); q_w(); dgrad(); wgrad()

    bwd()
    tqd, tqx, tqw = timed(q_dy, 1e12), timed(q_x, 1e12), timed(q_w, 1e12)
    tdg, twg, tbw = timed(dgrad, 1e12), timed(wgrad, 1e12), _graph_ms(bwd, args.steps, args.warmup)
    out["grouped_nvfp4_bwd"] = {
        "quantize_ms": {"dy_row_col_sr_rht": tqd, "x_col_rht": tqx, "w_col": tqw},
        "dgrad_ms": tdg, "dgrad_TFLOP/s": mflop / (tdg * 1e-3) / 1e12,
        "wgrad_ms": twg, "wgrad_TFLOP/s": mflop / (twg * 1e-3) / 1e12,
        "bwd_step_ms": tbw, "bwd_TFLOP/s": 2 * mflop / (tbw * 1e-3) / 1e12,
        "note": "the quantizations with their amax passes; dgrad dx_g = dy_g W_g, wgrad dW_g = dy_g^T x_g"}
    peaks, src = _peaks()
    return {"metric": "recipe variants (amax chain, rowwise-dequantized source, row scaling, 2D scaling, hybrid linear)",
            "value": out["hybrid_linear"]["TFLOP/s"], "unit": "TFLOP/s (hybrid-format linear step)",
            "variants": out, "hbm_peak_gbs": peaks["hbm_gbs"], "peak_source": src, "dtype": "mixed",
            "config": {"workload": "recipe_variants_llama3_8b_up_and_moe"}}


def run_single_linear(args, nvq, inputs):
    """x, W bf16[256,512]: quantize both rowwise and y = x W^T (latency)."""
    x, w = inputs.single_linear()
    x, w = x.cuda(), w.cuda()
    xr = nvq.alloc_qtensor(nvq.NVFP4, 256, 512)
    wr = nvq.alloc_qtensor(nvq.NVFP4, 256, 512)
    import torch
    y = torch.empty(256, 256, dtype=torch.bfloat16, device="cuda")

    def step():
        nvq.nvfp4_quantize(x, nvq.DIR_ROW, out_row=xr)
        nvq.nvfp4_quantize(w, nvq.DIR_ROW, out_row=wr)
        nvq.gemm_tn(xr, wr, out=y)

    ms = _flushed_ms(step, max(20, args.steps), args.warmup)
    return {"metric": "single NVFP4 linear forward latency (256x256x512)", "value": ms * 1e3, "unit": "us",
            "higher_is_better": False, "ms_per_step": ms, "dtype": "nvfp4",
            "config": {"workload": "single_linear_256x256x512"}}


def run_workload(args, rank, world, local_rank):
    """The other configurations (quantize sweep, MoE grouped, Qwen3-8B stack,
    single linear) are one-GPU measurements."""
    if world > 1:
        raise SystemExit(f"--workload {args.workload} runs on one GPU; the multi-GPU line is the default workload")
    import torch
    import __graft_entry__
    import mxfp8_block_scaled_bf16_gb300 as nvq
    from mxfp8_block_scaled_bf16_gb300 import inputs
    __graft_entry__.build()
    torch.cuda.set_device(local_rank)
    fn = {"quant_sweep": run_quant_sweep, "moe_grouped": run_moe_grouped, "qwen3_stack": run_qwen3_stack,
          "single_linear": run_single_linear, "variants": run_variants}[args.workload]
    clocks = ClockSampler(local_rank)
    clocks.start()
    r = fn(args, nvq, inputs)
    clk = clocks.stop()
    if nvq.device_status() != 0:
        raise RuntimeError("device status error")
    if rank != 0:
        return 0
    line = {"metric": r.pop("metric"), "value": r.pop("value"), "unit": r.pop("unit"), "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": r.pop("higher_is_better", True),
            "scaling": "weak", "vs_baseline": None, "data": "synthetic", "clocks": clk, **r}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip timing the CPU oracle")
    ap.add_argument("--eager", action="store_true", help="launch the step eagerly instead of replaying a CUDA graph")
    ap.add_argument("--serial-step", action="store_true",
                    help="replay the step's calls on one stream (default: the two independent pairs on two streams)")
    ap.add_argument("--oracle-child", type=float, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--no-amax-chain", action="store_true",
                    help="qwen3_stack: measure every amax with its own pass instead of taking it from the producing GEMM")
    ap.add_argument("--workload", default="llama_up",
                    choices=["llama_up", "quant_sweep", "moe_grouped", "qwen3_stack", "single_linear", "variants"],
                    help="llama_up (default: the headline line) or one of the other configurations")
    args = ap.parse_args()
    if args.oracle_child is not None:
        return _oracle_child(args.oracle_child)
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup
    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local_rank = _env_int("LOCAL_RANK", 0)
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        import torch
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        if args.workload != "llama_up":
            return run_workload(args, rank, world, local_rank)
        return run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
