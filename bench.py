"""Benchmark: NVFP4 quantize throughput (GB/s of bf16) on one GB300.

Headline workload: the 8192x28672 bf16 tensor (70B-style MLP, N(0, 0.01) with
0.05 % of the entries set to +-U(0.3, 1)).  One step = the whole hot path on
it: quantize with the max rule, FourOverSix, CJSO(5) and decoupled CJSO(5),
then dequantize, back to back (20 steps by default: the sustained form).  The
tensor (448 MiB) is larger than L2, and two device copies alternate, so every
step reads W from HBM.

    python bench.py [--gpus N --steps K --warmup W] [--impl reference]
                    [--workload NAME --modes a,b --iters T] [--no-stack] [--quick]

Prints one JSON line (rank 0).
  value        bf16 bytes of all ranks' steps (2 bytes per element for every
               mode: the quantizers' input, the dequantizer's output) / device
               time of the K steps (CUDA-graph replays of the C-ABI call
               sequence; CUDA events on the launching stream; barrier +
               synchronize on both sides; max over ranks).
  per_mode     each mode alone: call time, GB/s, its roofline (HBM copy
               bandwidth, or the measured fp32 FMA peak for the decoupled
               search), per-kernel device times (the library's per-launch CUDA
               events), reconstruction MSE in double, the M=4 block share of
               FourOverSix, and the C oracle on the host cores on a bounded
               sample of the same tensor.
  roofline     the dominant kernel of the step (largest share of the step's
               device time) against its bound.
  e2e          the same step through the C ABI with pinned host buffers: H2D of
               W and D2H of every output inside the timed region.
  workloads    further records of the same form (skipped with --no-stack or
               N > 1): the 224-tensor Llama-3-8B-shaped stack (FourOverSix
               grouped, decoupled CJSO(5)) and the 4096x14336 tensor (every mode).

--impl reference runs the C oracle on a bounded sample of the same workload
per step and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NVFP4 quantize GB/s (bf16 in) per mode; % of HBM or FP32 roofline, 1 GB300"
HEADLINE = "mlp_70b"
MODE_IDS = {"max": 0, "four_over_six": 1, "cjso": 2, "cjso_decoupled": 3, "dequant": 4, "gemv": 5, "swizzle": 6,
            "gemm": 7, "max_noalloc": 8, "four_over_six_noalloc": 9}
QUANTIZERS = (0, 1, 2, 3, 8, 9)  # modes that quantize W (8, 9: the allocation-free entry point, rule 0 or 1)
CONSUMERS = ("dequant", "gemv", "swizzle", "gemm")  # modes that read a quantized tensor instead of producing one
HOT_PATH = ("max", "four_over_six", "cjso", "cjso_decoupled", "dequant")


def _synth():
    import synthetic
    return synthetic


# name -> (generator(rank), description, default modes)
WORKLOADS = {
    "mlp_70b": (lambda r: _synth().mlp_70b(seed=4 + r),
                "8192x28672 bf16, N(0,0.01), 0.05% entries +-U(0.3,1) (seed 4 + rank)", HOT_PATH),
    "studentt_4k": (lambda r: _synth().studentt_4k(seed=1 + r),
                    "4096x4096 bf16, Student-t df=4 std 0.02, 0.1% columns x20 (seed 1 + rank)",
                    ("max", "four_over_six")),
    "gauss_1k": (lambda r: _synth().gauss_1k(seed=0 + r),
                 "1024x1024 bf16, N(0,0.02) (seed 0 + rank)", HOT_PATH),
    "mlp_up": (lambda r: _synth().mlp_up(seed=2 + r),
               "4096x14336 bf16, 10% rows N(0,0.05), rest N(0,0.015) (seed 2 + rank)", HOT_PATH),
}

NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal (the measured copy bandwidth is the roofline)
ONE_PASS = 2.5625   # B/elem: W read once (2) + codes (0.5) + scales (1/16)
TWO_PASS = 4.5625   # B/elem: W read twice (alpha needs the global max first)
DECOUPLED_FLOPS = 101 * 5  # per element: 101 candidates x (quotient FMUL 1 + P FMA 2 + R FMA 2)


def kernels_per_call(mode: int, iters: int) -> int:
    """Kernels one call launches: amax + quantize; amax + init sweep + one
    sweep per iteration (+ the search and its deferred-block pass); one kernel
    for the consumers."""
    return {0: 2, 1: 2, 2: 2 + iters, 3: 4 + iters, 4: 1, 5: 1, 6: 1, 7: 2, 8: 2, 9: 2}[mode]


def algorithmic(mode: int, iters: int, n: int, l2_bytes: int, batch: int = 1, hbm_gbs: float = 6660.0,
                tc_tflops: float = 1884.6):
    """(bound, unit, algorithmic work of one call, rule) for a mode."""
    fits = 2 * n <= l2_bytes // 2
    if mode in (0, 1, 8, 9):
        b = ONE_PASS if fits else TWO_PASS
        return "hbm", "GB/s", b * n, f"{b} B/elem ({'W <= L2/2: one HBM read' if fits else 'W read twice'})"
    if mode == 4:  # dequantize: codes + scales in, bf16 out
        return "hbm", "GB/s", ONE_PASS * n, "2.5625 B/elem (codes 0.5 + scales 1/16 read, bf16 2 written)"
    if mode == 5:  # W4A16 product: codes + scales once, x and y negligible
        return "hbm", "GB/s", 0.5625 * n, "0.5625 B/elem (codes + scales read once; + x, y)"
    if mode == 7:  # tensor-core W4A16 product of `batch` vectors: HBM or bf16 tensor bound, whichever is longer
        flops = 2.0 * n * batch
        if flops / (tc_tflops * 1e12) > 0.5625 * n / (hbm_gbs * 1e9):
            return "tensor", "TFLOP/s", flops, f"2 flop per weight and vector ({batch} vectors), bf16 tensor cores"
        return "hbm", "GB/s", 0.5625 * n, "0.5625 B/elem (codes + scales read once; + x, y)"
    if mode == 6:  # scale layout: scales read and written once
        return "hbm", "GB/s", 0.125 * n, "0.125 B/elem (scales read + written)"
    if mode == 2:
        b = ONE_PASS if fits else (iters + 2) * 2 + 0.5625
        return "hbm", "GB/s", b * n, f"{b} B/elem ({'W stays in L2' if fits else f'{iters + 2} reads of W'})"
    return "alu", "TFLOP/s", DECOUPLED_FLOPS * n, "505 fp32 flop/elem (101 candidates x [1 FMUL + 2 FMA])"


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (read-only)."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, index: int):
        self.ok = False
        self.samples = []
        self.reasons = 0
        self.max_mhz = None
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            self.ok = True
        except OSError:
            self.ok = False

    def _sample(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0:
            self.samples.append(int(clk.value))
        if self.nvml.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rs)) == 0:
            self.reasons |= int(rs.value)

    def start(self):
        self.samples, self.reasons = [], 0
        self._stop = threading.Event()
        if not self.ok:
            return

        def run():
            while not self._stop.is_set():
                self._sample()
                time.sleep(0.001)
        self._t = threading.Thread(target=run, daemon=True)
        self._t.start()

    def stop(self):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.ok:
            return {"unavailable": "NVML not loadable"}
        reasons = [n for b, n in self.REASONS.items() if self.reasons & b]
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(self.samples)}


BAD_REASONS = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}


# --------------------------------------------------------------------------- helpers

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def measured_bf16_tflops():
    """Dense bf16 tensor-core peak (burst: the product is timed alone)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return float(json.load(open(p))["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def fp32_peak_derived(sms: int, mhz: float) -> float:
    """FP32 FMA peak from the unit count: SMs x 128 lanes x 2 flop x clock."""
    return sms * 128 * 2 * mhz * 1e6 / 1e12


def source_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "nvfp4_block_scale_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(key: str):
    """DRAM bytes per launch (or call) from the committed ncu summary, if taken
    on the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        e = json.load(open(p))[key]
        if e.get("source_digest") == source_digest():
            return e["dram_bytes"]
    except Exception:
        pass
    return None


def max_over_ranks(x: float, device, ws: int) -> float:
    """The largest of every rank's x (each rank passes its own; ws == 1: x)."""
    if ws == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(ws: int, bytes_per_step_per_rank: float, steps: int, ms: float) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's time."""
    return ws * bytes_per_step_per_rank * steps / (ms / 1e3) / 1e9


def dist_env():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def input_sha256(w_bits: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(w_bits).tobytes()).hexdigest()


def oracle_rows(mode: str, cols: int, rows: int, batch: int = 1) -> int:
    """Rows of the bounded CPU sample per mode (a few seconds of oracle work on
    16 host cores): the decoupled search is ~100x slower per element."""
    budget = {"max": 1 << 23, "four_over_six": 1 << 23, "cjso": 1 << 22, "cjso_decoupled": 1 << 18,
              "dequant": 1 << 23, "swizzle": 1 << 23, "gemv": (1 << 23) // batch, "gemm": (1 << 23) // batch}[mode]
    return int(max(16, min(rows, budget // cols)))


# the oracle function a mode is timed against: the allocation-free entry point computes the
# max rule / FourOverSix; the consumers read a max-rule tensor
ORACLE_OF = {"max_noalloc": "max", "four_over_six_noalloc": "four_over_six"}


def oracle_time_mode(w_bits, mode: str, iters: int, min_seconds: float, batch: int = 1):
    """The oracle as it stands, on all host cores, on the first rows of W;
    returns (GB/s of bf16 W, seconds, repetitions, rows)."""
    import oracle
    import synthetic
    threads = os.cpu_count() or 1
    mode = ORACLE_OF.get(mode, mode)
    rows = oracle_rows(mode, w_bits.shape[1], w_bits.shape[0], batch)
    sample = np.ascontiguousarray(w_bits[:rows])
    cols = sample.shape[1]
    if mode in CONSUMERS:
        c, s, a = oracle.quantize(sample, oracle.MAX, 0, threads=threads)
        if mode == "dequant":
            fn = lambda: oracle.dequantize(c, s, a, rows, cols)
        elif mode == "swizzle":
            fn = lambda: oracle.swizzle_scales(s, rows, cols // 16)
        else:  # the W4A16 product with `batch` vectors
            x = synthetic.gaussian(batch, cols, 1.0, 7)
            fn = lambda: oracle.gemv(c, s, a, rows, cols, x)
    else:
        fn = lambda: oracle.quantize(sample, MODE_IDS[mode], iters, threads=threads)
    t0 = time.perf_counter()
    reps = 0
    while True:
        fn()
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            break
    return reps * sample.nbytes / el / 1e9, el, reps, rows


def oracle_cpu_baseline(w_bits, modes, iters, min_seconds=4.0, batch=1):
    """Per mode and for the whole step: the oracle on host cores, bounded samples."""
    threads = os.cpu_count() or 1
    per, tot_bytes, tot_s = {}, 0.0, 0.0
    for m in modes:
        gbs, el, reps, rows = oracle_time_mode(w_bits, m, iters, min_seconds, batch)
        what = {"dequant": " (dequantize of the max-rule output)",
                "swizzle": " (scale layout of the max-rule output)",
                "gemv": f" (oracle_gemv of the max-rule output, {batch} vector(s))",
                "gemm": f" (oracle_gemv of the max-rule output, {batch} vector(s))"}.get(m, "")
        if m in ORACLE_OF:
            what = f" (the {ORACLE_OF[m]} oracle: the function this entry point computes)"
        per[m] = {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                  "sample": f"rows 0..{rows - 1} of {w_bits.shape[0]}x{w_bits.shape[1]}, {reps} repetition(s) "
                            f"in {el:.1f} s" + what}
        tot_bytes += w_bits.shape[1] * 2  # one row of bf16 per mode: combine per-row costs
        tot_s += w_bits.shape[1] * 2 / (gbs * 1e9)
    step = {"value": tot_bytes / tot_s / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": "the step's modes, each timed on its own row sample (per_mode[*].cpu_baseline); value = "
                      "bf16 bytes of one row through every mode / the summed per-row times"}
    return step, per


def mse_on_device(W, codes, scales, alpha, chunk_rows=1024) -> float:
    """(1/N) sum (x - q * fl(alpha * Delta))^2 in double, on the device (a
    statistic of the outputs, computed outside the timed region)."""
    import torch
    mags = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0],
                        dtype=torch.float64, device=W.device)
    rows, cols = W.shape
    a32 = alpha.reshape(1).to(torch.float32)
    acc = torch.zeros((), dtype=torch.float64, device=W.device)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        c = codes[r0:r1].to(torch.int64)
        idx = torch.stack([c & 0xF, c >> 4], dim=-1).reshape(r1 - r0, cols)
        q = mags[idx]
        d = scales[r0:r1].contiguous().view(torch.float8_e4m3fn).to(torch.float32)
        s = (a32 * d).to(torch.float64).repeat_interleave(16, dim=1)  # fl32(alpha * Delta)
        e = W[r0:r1].to(torch.float64) - q * s
        acc += (e * e).sum()
    return float(acc.item()) / (rows * cols)


# --------------------------------------------------------------------------- our arm

def run_ours(args, modes):
    import torch
    import torch.distributed as dist

    import nvfp4_block_scale_gb300 as nv

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    make, desc, _ = WORKLOADS[args.workload]
    w_bits = make(rank)
    rows, cols = w_bits.shape
    n = w_bits.size
    props = torch.cuda.get_device_properties(dev)
    l2 = props.L2_cache_size
    ncopy = max(2, min(8, math.ceil(2 * l2 / w_bits.nbytes) + 1))
    W_host = torch.from_numpy(w_bits.view(np.int16)).view(torch.bfloat16)
    Wd = [W_host.to(dev) for _ in range(ncopy)]
    mids = [MODE_IDS[m] for m in modes]
    # outputs rotate with the inputs (one set per copy and mode), so they are
    # written back to HBM as a real sequence of tensors would be
    outs = {m: [(torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev),
                 torch.empty((rows, cols // 16), dtype=torch.uint8, device=dev),
                 torch.empty(1, dtype=torch.float32, device=dev)) for _ in range(ncopy)] for m in mids if m in QUANTIZERS}

    if any(m >= 4 for m in mids):  # consumer inputs: this tensor quantized (max rule) once per rotation slot
        dq_in = []
        for i in range(ncopy):
            c, sc, a = nv.quantize(Wd[i], nv.MAX)
            dq_in.append((c, sc, a))
        dq_out = [torch.empty((rows, cols), dtype=torch.bfloat16, device=dev) for _ in range(ncopy)]
        gx = torch.randn((args.batch, cols), device=dev).to(torch.bfloat16)
        gy = torch.empty((args.batch, rows), dtype=torch.float32, device=dev)
        gz = torch.empty(nv.nvfp4_swizzled_scales_bytes(rows, cols), dtype=torch.uint8, device=dev)

    def slot_of(w):
        return next(k for k in range(ncopy) if Wd[k] is w)

    def call(mode, w, s):
        if mode in (8, 9):  # the allocation-free entry point (max rule / FourOverSix)
            c, sc, a = outs[mode][slot_of(w)]
            st = nv.nvfp4_quantize_noalloc(w.data_ptr(), rows, cols, mode - 8, c.data_ptr(), sc.data_ptr(),
                                           a.data_ptr(), s.cuda_stream)
        elif mode == 6:  # the slot's scales into the tensor-core layout
            st = nv.nvfp4_swizzle_scales(dq_in[slot_of(w)][1].data_ptr(), rows, cols, gz.data_ptr(), s.cuda_stream)
        elif mode == 7:  # tensor-core product of `batch` vectors with the slot's quantized tensor
            c, sc, a = dq_in[slot_of(w)]
            st = nv.nvfp4_gemm(c.data_ptr(), sc.data_ptr(), a.data_ptr(), rows, cols, gx.data_ptr(), args.batch,
                               gy.data_ptr(), s.cuda_stream)
        elif mode == 5:  # one-vector product with the slot's quantized tensor
            c, sc, a = dq_in[slot_of(w)]
            st = nv.nvfp4_gemv(c.data_ptr(), sc.data_ptr(), a.data_ptr(), rows, cols, gx.data_ptr(), args.batch,
                               gy.data_ptr(), s.cuda_stream)
        elif mode == 4:  # dequantize the slot of this W into that slot's output
            i = slot_of(w)
            c, sc, a = dq_in[i]
            st = nv.nvfp4_dequantize(c.data_ptr(), sc.data_ptr(), a.data_ptr(), rows, cols, dq_out[i].data_ptr(),
                                     s.cuda_stream)
        else:
            c, sc, a = outs[mode][slot_of(w)]
            st = nv.nvfp4_quantize(w.data_ptr(), rows, cols, mode, args.iters, c.data_ptr(), sc.data_ptr(),
                                   a.data_ptr(), s.cuda_stream)
        if st != 0:
            raise RuntimeError(f"nvfp4 call: {nv.nvfp4_status_string(st)}")

    def step(i, s):
        for j, m in enumerate(mids):
            call(m, Wd[(i * len(mids) + j) % ncopy], s)

    for i in range(max(args.warmup, 3)):
        step(i, stream)
    torch.cuda.synchronize()

    launch = "eager"
    graphs = []
    # steps per CUDA graph: back-to-back calls chain by programmatic dependent
    # launch inside a graph, and the graph boundary costs a launch gap
    per_graph = 4 if args.steps % 4 == 0 and not args.quick else 1
    if not args.quick:  # ncopy CUDA graphs of `per_graph` consecutive steps each (the rotation continues)
        try:
            for i in range(ncopy):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for t in range(per_graph):
                        step(i * per_graph + t, torch.cuda.current_stream())
                graphs.append(g)
            for g in graphs:
                g.replay()
            torch.cuda.synchronize()
            launch = f"cuda_graph ({per_graph} step(s) per graph)"
        except Exception as e:  # eager fallback, reported in config
            launch = f"eager ({type(e).__name__})"
            graphs = []

    def run_steps(k, s):  # k steps (a multiple of per_graph when graphs are used)
        if graphs:
            for i in range(k // per_graph):
                graphs[i % len(graphs)].replay()
        else:
            for i in range(k):
                step(i, s)

    def whole(k):  # k rounded up to whole graphs
        return -(-k // per_graph) * per_graph if graphs else k

    def timed(k):
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run_steps(k, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
        return e0.elapsed_time(e1)

    clocks = ClockSampler(local)
    for attempt in range(2):
        run_steps(whole(max(args.warmup, 3)), stream)
        clocks.start()
        ms = timed(args.steps)
        if len(clocks.samples) < 5 and not args.quick:  # short region: keep sampling over the same loop
            timed(whole(max(args.steps, int(200.0 / max(ms / args.steps, 1e-3)))))
        clocks.stop()
        csum = clocks.summary()
        if not (set(csum.get("reasons", [])) & BAD_REASONS):
            break
        csum["remeasured"] = True
    ms = max_over_ranks(ms, dev, ws)
    bytes_per_step = len(mids) * 2 * n
    value = job_gbs(ws, bytes_per_step, args.steps, ms)
    out = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16 in, fp32 arithmetic, e2m1+e4m3 out", "data": "synthetic",
           "config": {"workload": args.workload, "desc": desc, "rows": rows, "cols": cols, "modes": list(modes),
                      "value_is": "2 bytes per element per mode (bf16 in of each quantizer, bf16 out of the "
                                  "dequantizer) / device time of the whole step",
                      "cjso_iters": args.iters if any(2 <= m <= 3 for m in mids) else None,
                      "batch": args.batch if (5 in mids or 7 in mids) else None,
                      "input_sha256": input_sha256(w_bits),
                      "l2": f"rotate {ncopy} input copies ({ncopy * w_bits.nbytes >> 20} MiB; L2 {l2 >> 20} MiB) "
                            f"and {ncopy} output sets per mode: every step reads W from HBM",
                      "launch": launch, "parallelism": f"{ws} independent replica(s), one tensor per rank"},
           "gpu_launches": sum(kernels_per_call(m, args.iters) for m in mids) * args.steps, "clocks": csum}
    if args.quick:
        if ws > 1:
            dist.destroy_process_group()
        return out if rank == 0 else None

    # ---- the fp32 peak of this GPU, measured now (the decoupled search's roofline)
    fp32 = nv.fp32_peak_tflops()
    sm_mhz = csum.get("sm_mhz") or 1900.0
    fp32["derived_at_sampled_clock"] = fp32_peak_derived(props.multi_processor_count, sm_mhz)
    out["fp32_peak"] = fp32

    # ---- per mode: device throughput and per-kernel times (library CUDA events)
    per_mode = {}
    peak_hbm, peak_kind = measured_peaks()
    tc_peak, tc_kind = measured_bf16_tflops()
    for name, m in zip(modes, mids):
        # device time of this mode alone: graphs of 4 back-to-back calls on rotating
        # copies (steady state), and graphs of one call (an isolated call's latency)
        k = max(min(args.steps, 240), 24)
        times = {}
        for chain in (4, 1):
            gm = []
            if graphs:
                for i in range(ncopy):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g):
                        for t in range(chain):
                            call(m, Wd[(i * chain + t) % ncopy], torch.cuda.current_stream())
                    gm.append(g)
            for g in gm:
                g.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            if gm:
                for i in range(k // chain):
                    gm[i % ncopy].replay()
            else:
                for i in range(k):
                    call(m, Wd[i % ncopy], stream)
            e1.record(stream)
            torch.cuda.synchronize()
            times[chain] = e0.elapsed_time(e1) / k
            del gm
        call_ms = times[4]
        # per-kernel breakdown from the library tracer (event-bracketed launches,
        # so each includes its launch gap)
        nv.nvfp4_profiler_reset()
        nv.nvfp4_profiler_enable(1)
        for i in range(8):
            call(m, Wd[i % ncopy], stream)
        torch.cuda.synchronize()
        nv.nvfp4_profiler_enable(0)
        rep = nv.profiler_report()
        bound, unit, work, rule = algorithmic(m, args.iters, n, l2, args.batch, peak_hbm, tc_peak)
        if bound == "hbm":
            achieved, peak, pk = work / (call_ms / 1e3) / 1e9, peak_hbm, peak_kind
            over, tkey = "the whole call", f"nvfp4_{'dequantize' if m == 4 else 'quantize'}({name})@{args.workload}"
        elif bound == "tensor":
            achieved, peak, pk = work / (call_ms / 1e3) / 1e12, tc_peak, tc_kind
            over, tkey = "the whole call", None
        else:  # the search kernel alone (its event-bracketed duration), not the CJSO sweeps before it
            kc, kt = rep["k_decoupled"]
            achieved = work / (kt / kc / 1e3) / 1e12
            peak, pk = fp32["tflops"], "measured (fp32 FMA probe, this run)"
            over, tkey = "k_decoupled", f"k_decoupled@{args.workload}"
        pm = {"GBps_bf16_in" if m != 4 else "GBps_bf16_out": 2 * n / (call_ms / 1e3) / 1e9,
              "us_per_call": call_ms * 1e3, "us_isolated_call": times[1] * 1e3,
              "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                           "frac": achieved / peak, "peak_kind": pk, "rule": rule, "over": over,
                           "traffic": recorded_traffic(tkey) if tkey else None,
                           "frac_of_nominal": (achieved / NOMINAL_HBM_GBS if bound == "hbm" else None)},
              "kernels_event_bracketed": {kn: {"launches": c, "avg_us": t / c * 1e3} for kn, (c, t) in rep.items()}}
        if bound == "alu":
            pm["roofline"]["frac_of_derived_peak"] = achieved / fp32["derived_at_sampled_clock"]
        if m in QUANTIZERS:  # reconstruction error of this mode's output, in double
            c, sc, a = outs[m][0]
            pm["mse"] = mse_on_device(Wd[0], c, sc, a)
        per_mode[name] = pm
    if "four_over_six" in per_mode:  # share of blocks whose FourOverSix scale is the M=4 one
        f = outs[1][0][1]
        mx = outs[0][0][1] if 0 in outs else nv.quantize(Wd[0], nv.MAX)[1]
        per_mode["four_over_six"]["m4_share"] = float((f != mx).to(torch.float64).mean().item())
    out["per_mode"] = per_mode

    # ---- the dominant kernel of the step: the largest share of the step's device time
    shares = {}
    for name, pm in per_mode.items():
        for kn, kv in pm["kernels_event_bracketed"].items():
            shares[(name, kn)] = kv["launches"] / 8 * kv["avg_us"]
    (dm, dk), _ = max(shares.items(), key=lambda x: x[1])
    pm = per_mode[dm]
    bound, unit, work, rule = algorithmic(MODE_IDS[dm], args.iters, n, l2, args.batch, peak_hbm, tc_peak)
    k_us = pm["kernels_event_bracketed"][dk]["avg_us"]
    if bound == "alu" and dk == "k_decoupled":
        achieved, peak, pk, ru = work / (k_us / 1e6) / 1e12, fp32["tflops"], "measured (fp32 FMA probe, this run)", rule
    else:  # an HBM-bound kernel: its own bytes per launch (one read of W, or the mode's rule)
        kb = {"k_amax_bulk": 2.0, "k_amax_partials": 2.0, "k_dequant": ONE_PASS, "k_cjso_sweep<iter>": 2.0 + 2 / 16,
              "k_cjso_sweep<init>": 2.0 + 1 / 16}.get(dk, 2.5625)
        achieved, peak, pk, unit = kb * n / (k_us / 1e6) / 1e9, peak_hbm, peak_kind, "GB/s"
        bound, ru = "hbm", f"{kb} B/elem per launch"
    total_us = sum(shares.values())
    out["roofline"] = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                       "traffic": recorded_traffic(f"{dk}@{args.workload}"), "kernel": dk, "mode": dm,
                       "share_of_step": shares[(dm, dk)] / total_us, "peak_kind": pk, "rule": ru,
                       "timing": "the library's CUDA events around each launch of the kernel, on its stream "
                                 "(average over the traced launches)"}

    # ---- end to end through the C ABI with pinned host buffers: every step copies
    # its W in (H2D), quantizes it with each mode, dequantizes the max-rule output
    # (when the step has dequant) and copies every output back (D2H).  Steps are
    # pipelined over two buffer slots and three streams, so the copies of one
    # step overlap the kernels of its neighbours.
    W_pin = W_host.pin_memory()
    qmids = [m for m in mids if m in QUANTIZERS]
    with_dq = 4 in mids
    slots = []
    for _ in range(2):
        o = {m: tuple(torch.empty_like(t) for t in outs[m][0]) for m in qmids}
        ho = {m: tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs[m][0]) for m in qmids}
        dq = (torch.empty((rows, cols), dtype=torch.bfloat16, device=dev),
              torch.empty((rows, cols), dtype=torch.bfloat16).pin_memory()) if with_dq else None
        slots.append({"W": torch.empty_like(Wd[0]), "outs": o, "host": ho, "dq": dq,
                      "h2d": torch.cuda.Event(), "comp": torch.cuda.Event(), "d2h": torch.cuda.Event()})
    s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    dq_src = qmids[0] if qmids else None

    def qcall(mode, w, o, st):
        c, sc, a = o
        if mode in (8, 9):
            r = nv.nvfp4_quantize_noalloc(w.data_ptr(), rows, cols, mode - 8, c.data_ptr(), sc.data_ptr(),
                                          a.data_ptr(), st.cuda_stream)
        else:
            r = nv.nvfp4_quantize(w.data_ptr(), rows, cols, mode, args.iters, c.data_ptr(), sc.data_ptr(),
                                  a.data_ptr(), st.cuda_stream)
        if r != 0:
            raise RuntimeError(f"nvfp4_quantize: {nv.nvfp4_status_string(r)}")

    def e2e_step(i):
        sl = slots[i % 2]
        s_h2d.wait_event(sl["comp"])  # the slot's W is no longer read
        with torch.cuda.stream(s_h2d):
            sl["W"].copy_(W_pin, non_blocking=True)
        sl["h2d"].record(s_h2d)
        stream.wait_event(sl["h2d"])
        stream.wait_event(sl["d2h"])  # the slot's outputs have been copied out
        for m in qmids:
            qcall(m, sl["W"], sl["outs"][m], stream)
        if with_dq and dq_src is not None:
            c, sc, a = sl["outs"][dq_src]
            r = nv.nvfp4_dequantize(c.data_ptr(), sc.data_ptr(), a.data_ptr(), rows, cols, sl["dq"][0].data_ptr(),
                                    stream.cuda_stream)
            if r != 0:
                raise RuntimeError(f"nvfp4_dequantize: {nv.nvfp4_status_string(r)}")
        sl["comp"].record(stream)
        s_d2h.wait_event(sl["comp"])
        with torch.cuda.stream(s_d2h):
            for m in qmids:
                for dst, src in zip(sl["host"][m], sl["outs"][m]):
                    dst.copy_(src, non_blocking=True)
            if with_dq:
                sl["dq"][1].copy_(sl["dq"][0], non_blocking=True)
        sl["d2h"].record(s_d2h)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    k_e2e = max(min(args.steps, 200), 6)
    e0.record(stream)
    s_h2d.wait_stream(stream)
    for i in range(k_e2e):
        e2e_step(i)
    stream.wait_stream(s_d2h)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev, ws)
    d2h = sum(t.numel() * t.element_size() for m in slots[0]["host"] for t in slots[0]["host"][m])
    if with_dq:
        d2h += 2 * n
    out["e2e"] = {"value": job_gbs(ws, bytes_per_step, k_e2e, e2e_ms), "unit": "GB/s",
                  "modes": list(modes), "h2d_bytes_per_step": w_bits.nbytes, "d2h_bytes_per_step": d2h,
                  "steps": k_e2e, "pipelining": "2 buffer slots; H2D, kernels and D2H on three streams"}

    if rank == 0 and ws == 1:
        step_cpu, per_cpu = oracle_cpu_baseline(w_bits, list(modes), args.iters, batch=args.batch)
        out["cpu_baseline"] = step_cpu
        for m, v in per_cpu.items():
            per_mode[m]["cpu_baseline"] = v
    del Wd, outs, slots
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return out if rank == 0 else None


# --------------------------------------------------------------------------- model-stack workload

MODEL = "llama3_8b"
MODEL_DESC = ("224 bf16 tensors of a Llama-3-8B-shaped stack (32 layers x {q 4096x4096, k/v 1024x4096, "
              "o 4096x4096, gate/up 14336x4096, down 4096x14336}), Student-t df=5 std 0.02, generated on the "
              "device with torch.Generator seeded 1000 + tensor index")


def model_tensors(dev, layers=32):
    """The stack's tensors, generated on the device (Student-t df=5 scaled to std 0.02)."""
    import torch
    shapes = _synth().llama3_8b_shapes(layers)
    scale = 0.02 / math.sqrt(5.0 / 3.0)
    Ws = []
    for idx, (_, r, c) in enumerate(shapes):
        g = torch.Generator(device=dev).manual_seed(1000 + idx)
        z = torch.randn((r, c), generator=g, device=dev)
        chi2 = 2.0 * torch._standard_gamma(torch.full((r, c), 2.5, device=dev), generator=g)
        Ws.append((z * torch.rsqrt(chi2 / 5.0) * scale).to(torch.bfloat16))
        del z, chi2
    return shapes, Ws


def run_model(args, modes, fp32=None, steps=None):
    import torch

    import nvfp4_block_scale_gb300 as nv

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    props = torch.cuda.get_device_properties(dev)
    l2 = props.L2_cache_size
    shapes, Ws = model_tensors(dev, args.layers)
    ns = [W.numel() for W in Ws]
    n = sum(ns)
    outs = [(torch.empty((r, c // 2), dtype=torch.uint8, device=dev),
             torch.empty((r, c // 16), dtype=torch.uint8, device=dev),
             torch.empty(1, dtype=torch.float32, device=dev)) for (_, r, c) in shapes]
    qmodes = [m for m in modes if m not in CONSUMERS]
    mids = [MODE_IDS[m] for m in qmodes]

    def grouped(mode):
        nv.quantize_grouped(Ws, mode, args.iters, outs=outs)

    def per_tensor(mode):
        for W, o in zip(Ws, outs):
            nv.quantize(W, mode, args.iters, out=o)

    def step():
        for m in mids:
            grouped(m)

    def graph_of(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        g.replay()
        torch.cuda.synchronize()
        return g

    def event_ms(fn, k):
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(k):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    steps = args.steps if steps is None else steps
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    # kernels per step, counted by the library's tracer (a grouped call's launches depend on
    # how the library cuts the group into parts; the search's deferred-block kernel is traced
    # with the search)
    nv.nvfp4_profiler_reset()
    nv.nvfp4_profiler_enable(1)
    step()
    torch.cuda.synchronize()
    nv.nvfp4_profiler_enable(0)
    traced = nv.profiler_report()
    launches = sum(c for c, _ in traced.values()) + traced.get("k_decoupled", (0, 0.0))[0]
    gstep = graph_of(step)
    clocks = ClockSampler(local)
    for attempt in range(2):
        clocks.start()
        ms = event_ms(gstep.replay, steps)
        clocks.stop()
        csum = clocks.summary()
        if not (set(csum.get("reasons", [])) & BAD_REASONS):
            break
        csum["remeasured"] = True
    del gstep
    value = len(mids) * 2 * n * steps / (ms / 1e3) / 1e9
    out = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1, "steps": steps,
           "warmup": args.warmup, "ms_per_step": ms / steps, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16 in, fp32 arithmetic, e2m1+e4m3 out", "data": "synthetic",
           "config": {"workload": MODEL, "desc": MODEL_DESC, "layers": args.layers, "tensors": len(Ws),
                      "elements": n,
                      "modes": list(qmodes), "cjso_iters": args.iters if any(m >= 2 for m in mids) else None,
                      "l2": f"inputs {2 * n >> 30} GiB, larger than L2 ({l2 >> 20} MiB)",
                      "launch": "cuda_graph of nvfp4_quantize_grouped per mode",
                      "parallelism": "1 GPU"},
           "gpu_launches": launches * steps, "clocks": csum}
    if args.quick:
        return out

    peak_hbm, peak_kind = measured_peaks()
    if fp32 is None:
        fp32 = nv.fp32_peak_tflops()
    per_mode = {}
    for name, m in zip(qmodes, mids):
        k = 3 if m >= 2 else 20
        gm = graph_of(lambda: grouped(m))
        call_ms = event_ms(gm.replay, k) / k
        del gm
        gp = graph_of(lambda: per_tensor(m))
        per_tensor_ms = event_ms(gp.replay, k) / k
        del gp
        nv.nvfp4_profiler_reset()
        nv.nvfp4_profiler_enable(1)
        grouped(m)
        torch.cuda.synchronize()
        nv.nvfp4_profiler_enable(0)
        rep = nv.profiler_report()
        tkey = None
        if m in (0, 1):  # per tensor: one HBM read when it fits in half of L2, else two
            work = sum((ONE_PASS if 2 * x <= l2 // 2 else TWO_PASS) * x for x in ns)
            achieved, peak, pk, unit, bound = work / (call_ms / 1e3) / 1e9, peak_hbm, peak_kind, "GB/s", "hbm"
            rule, over = "2.5625 B/elem for tensors <= L2/2, 4.5625 above", "the whole call"
            tkey = f"nvfp4_quantize_grouped({name})@{MODEL}"
        elif m == 2:
            work = sum(((args.iters + 2) * 2 + 0.5625) * x for x in ns)
            achieved, peak, pk, unit, bound = work / (call_ms / 1e3) / 1e9, peak_hbm, peak_kind, "GB/s", "hbm"
            rule, over = f"{(args.iters + 2) * 2 + 0.5625} B/elem ({args.iters + 2} reads of W)", "the whole call"
        else:
            kc, kt = rep["k_decoupled"]
            work = DECOUPLED_FLOPS * n
            achieved = work / (kt / 1e3) / 1e12
            peak, pk = fp32["tflops"], "measured (fp32 FMA probe, this run)"
            unit, bound, over = "TFLOP/s", "alu", "k_decoupled (all tensors; sum of their durations)"
            rule = "505 fp32 flop/elem (101 candidates x [1 FMUL + 2 FMA])"
        pm = {"GBps_bf16_in": 2 * n / (call_ms / 1e3) / 1e9, "ms_per_call": call_ms,
              "per_tensor_calls_ms": per_tensor_ms,
              "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                           "frac": achieved / peak, "peak_kind": pk, "rule": rule, "over": over,
                           "traffic": recorded_traffic(tkey) if tkey else None,
                           "frac_of_nominal": (achieved / NOMINAL_HBM_GBS if bound == "hbm" else None)},
              "kernels_event_bracketed": {kn: {"launches": c, "avg_us": t / c * 1e3}
                                          for kn, (c, t) in rep.items()}}
        # reconstruction error and M=4 share over the stack (statistics of the outputs)
        pm["mse"] = sum(mse_on_device(W, *o) * W.numel() for W, o in zip(Ws, outs)) / n
        if m == 1:
            mx = [nv.quantize(W, nv.MAX)[1] for W in Ws[:7]]
            nb = sum(o[1].numel() for o in outs[:7])
            pm["m4_share_layer0"] = sum(float((o[1] != x).sum().item()) for o, x in zip(outs[:7], mx)) / nb
        per_mode[name] = pm
    heavy = max(per_mode, key=lambda x: per_mode[x]["ms_per_call"])
    hr = per_mode[heavy]["roofline"]
    out["per_mode"] = per_mode
    out["roofline"] = dict(hr, kernel=f"nvfp4_quantize_grouped({heavy})")

    # end to end over layer 0 (7 tensors) through the C ABI with pinned host buffers
    lay = list(range(7))
    host_w = [Ws[i].cpu().pin_memory() for i in lay]
    dev_w = [torch.empty_like(Ws[i]) for i in lay]
    host_o = [tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs[i]) for i in lay]
    fos = MODE_IDS["four_over_six"]

    def e2e_step():
        for hw, dw in zip(host_w, dev_w):
            dw.copy_(hw, non_blocking=True)
        nv.quantize_grouped(dev_w, fos, 0, outs=[outs[i] for i in lay])
        for i, ho in zip(lay, host_o):
            for dst, src in zip(ho, outs[i]):
                dst.copy_(src, non_blocking=True)

    for _ in range(3):
        e2e_step()
    k_e2e = 5
    e2e_ms = event_ms(e2e_step, k_e2e)
    n_lay = sum(ns[i] for i in lay)
    out["e2e"] = {"value": 2 * n_lay * k_e2e / (e2e_ms / 1e3) / 1e9, "unit": "GB/s", "modes": ["four_over_six"],
                  "sample": "layer 0 (7 tensors, 416 MiB), FourOverSix",
                  "h2d_bytes_per_step": 2 * n_lay,
                  "d2h_bytes_per_step": sum(t.numel() * t.element_size() for ho in host_o for t in ho),
                  "steps": k_e2e}
    w0 = Ws[0][:512].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    step_cpu, per_cpu = oracle_cpu_baseline(w0, qmodes, args.iters, min_seconds=3.0)
    out["cpu_baseline"] = dict(step_cpu, sample=step_cpu["sample"] + " (layer 0 q_proj)")
    for m, v in per_cpu.items():
        per_mode[m]["cpu_baseline"] = dict(v, sample=v["sample"] + " (layer 0 q_proj)")
    del Ws, outs
    torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------------------- reference arm

def run_reference(args, modes):
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    if args.workload == MODEL:  # the stack's first tensor (numpy recipe of the same distribution)
        w_bits, desc = _synth().llama3_8b_tensor(0), MODEL_DESC
    else:
        make, desc, _ = WORKLOADS[args.workload]
        w_bits = make(0)
    threads = os.cpu_count() or 1
    qmodes = [m for m in modes if m not in CONSUMERS or m == "dequant"]
    # a bounded per-step sample: each mode on its own first rows of W, about a
    # second of oracle work per mode on 16 host cores
    samples = {m: np.ascontiguousarray(w_bits[:max(16, oracle_rows(m, w_bits.shape[1], w_bits.shape[0]) // 4)])
               for m in qmodes}
    deq_in = {}
    if "dequant" in samples:
        s = samples["dequant"]
        deq_in = oracle.quantize(s, oracle.MAX, 0, threads=threads)

    def step():
        for m in qmodes:
            s = samples[m]
            if m == "dequant":
                oracle.dequantize(*deq_in, s.shape[0], s.shape[1])
            else:
                oracle.quantize(s, MODE_IDS[m], args.iters, threads=threads)

    for _ in range(max(args.warmup, 3)):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    # same definition as our arm's value: 2 bytes per element per mode over the step
    # time, with each mode's share of a step scaled from its sample to one row
    per_row_s = sum(el / args.steps / samples[m].shape[0] for m in qmodes)
    value = len(qmodes) * 2 * w_bits.shape[1] / per_row_s / 1e9
    sdesc = (f"C oracle, {threads} host threads, per step each mode on its own first rows of the "
             f"{w_bits.shape[0]}x{w_bits.shape[1]} tensor ("
             + ", ".join(f"{m}: {samples[m].shape[0]}" for m in qmodes) + " rows)")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 in, fp32 arithmetic, e2m1+e4m3 out", "data": "synthetic",
            "config": {"workload": args.workload, "desc": desc, "rows": int(w_bits.shape[0]),
                       "cols": int(w_bits.shape[1]), "modes": list(modes), "input_sha256": input_sha256(w_bits)},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sdesc},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS) + [MODEL])
    ap.add_argument("--modes", default=None, help="comma list of " + ",".join(MODE_IDS))
    ap.add_argument("--iters", type=int, default=5, help="CJSO iterations")
    ap.add_argument("--layers", type=int, default=32, help=f"layers of the {MODEL} stack (1..32)")
    ap.add_argument("--stack-steps", type=int, default=4, help=f"timed steps of the {MODEL} record")
    ap.add_argument("--batch", type=int, default=1, help="activation vectors of the gemv (1..8) and gemm (1..256) modes")
    ap.add_argument("--no-stack", action="store_true",
                    help=f"skip the further records ({MODEL}, mlp_up) of the headline run")
    ap.add_argument("--quick", action="store_true",
                    help="timed region only (eager; no graphs, e2e, oracle or tracing): for profiler runs")
    args = ap.parse_args()
    default_modes = ("four_over_six", "cjso_decoupled") if args.workload == MODEL else WORKLOADS[args.workload][2]
    modes = tuple(args.modes.split(",")) if args.modes else default_modes
    for m in modes:
        if m not in MODE_IDS:
            raise SystemExit(f"unknown mode {m}")
    if args.impl == "reference":
        out = run_reference(args, modes)
    elif args.workload == MODEL:
        out = run_model(args, modes)
    else:
        out = run_ours(args, modes)
        ws, rank, _ = dist_env()
        if (out is not None and ws == 1 and not args.quick and not args.no_stack and args.workload == HEADLINE
                and args.modes is None):
            out["workloads"] = {MODEL: run_model(args, ("four_over_six", "cjso_decoupled"), out.get("fp32_peak"),
                                                  steps=args.stack_steps)}
            up = argparse.Namespace(**vars(args))
            up.workload = "mlp_up"
            out["workloads"]["mlp_up"] = run_ours(up, WORKLOADS["mlp_up"][2])
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
