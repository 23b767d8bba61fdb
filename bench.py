"""Throughput of the NVFP4 quantization hot path on GB300.

One step = one pass of the whole path over the LLM-shaped bf16 sweep
(W1 [4096,14336], W2 [14336,4096] ~ 0.02*N(0,1); A [16384,4096] ~ Student-t(4)
with 0.1% outlier channels x100; seed 4):
  1. W1  SR + error feedback, 1x16            (fp32 residual read + written)
  2. W2  SR + error feedback, 16x16
  3. A   per-tensor amax, then four-over-six MAE, bound 256, 1x16 rowwise
  4. W1  per-tensor amax, then four-over-six MAE, bound 256, 16x16 rowwise + columnwise
  5. W2  the same as 4
  6. A   round-to-nearest, 1x16
  7. W2  stochastic rounding, 1x16
  8. A   dequantize (codes of 3) to bf16
The amax passes are separate nvfp4_amax calls whose result the quantize call
takes as given: the same two kernels the quantize call runs by itself with a
computed amax, timed apart.  Metric: algorithmic GB/s (bytes read + written
once each, amax passes counted with their real extra read) and Gelem/s
(elements quantized or dequantized), as a fraction of measured HBM peak; the
roofline line is for the kernel with the largest time per step.

Beside the step (not in its value) the line also reports the FP4 GEMM
consumer (fp4_mm), the fp32 [8192,8192] four-over-six 16x16 MSE row+col
configuration (c4_rowcol), plain rowwise + columnwise quantization of W1
(rowcol_plain) and the other graded variants (variants: SR + error feedback
on every c5 tensor in both block shapes, c3 four-over-six MAE/MSE with
per-tensor and per-row amax, the c2 stored-weight step).

e2e: the same step through the binding on pinned host buffers, every call
non-blocking: each step uploads its own inputs and brings every result back
(bytes counted per step); the steps run back to back and one synchronize
ends the timed region, a step's residual uploads waiting for the previous
step's residual downloads.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                  [--mm-only | --c4-only | --rowcol-only | --variants-only [--only VARIANT]]

N > 1 runs under torchrun: every rank processes its own copy of the sweep
(independent problems, no collective on the data path; weak scaling).
--impl reference times the CPU oracle, on every host core, on a bounded sample
of the same step.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

GB = 1e9


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--only", default=None,
                   help="time only the step's calls whose name contains this text (profiling); the "
                        "warm-up steps run every call")
    p.add_argument("--mm-only", action="store_true",
                   help="only the FP4 product measurement (quantize A and W2, then time nvfp4_mm)")
    p.add_argument("--c4-only", action="store_true",
                   help="only the fp32 [8192,8192] four-over-six 16x16 row+col measurement")
    p.add_argument("--rowcol-only", action="store_true",
                   help="only the plain rowwise + columnwise measurement on W1 (--only picks a variant)")
    p.add_argument("--variants-only", action="store_true",
                   help="only the graded variants outside the step (--only picks by name)")
    p.add_argument("--graph", type=int, default=1,
                   help="1: the timed steps replay as one captured CUDA graph; 0: issued call by call")
    p.add_argument("--single", default=None, choices=sorted(SINGLE),
                   help="time one kernel variant the step does not run (profiling)")
    return p.parse_args()


METRIC = "NVFP4 quantize GB/s (Gelem/s alongside); % of HBM roofline"
WORKLOAD = ("c5 LLM-shaped sweep, bf16: W1[4096,14336], W2[14336,4096] ~ 0.02*N(0,1), "
            "A[16384,4096] ~ Student-t(4) with 4 outlier channels x100 (seed 4); SR+EF 1x16 "
            "and 16x16 (seed 0, step t), four-over-six MAE bound 256 (1x16 rowwise on A, 16x16 "
            "row+col on W1/W2, per-tensor amax computed by a separate amax call), RTN, SR, dequantize")


def step_plan(M1, K1, M2, K2, Ma, Ka):
    """(call, kernel, elements, algorithmic bytes) per call of one step."""
    e1, e2, ea = M1 * K1, M2 * K2, Ma * Ka
    q = 0.5 + 1 / 16                       # codes + scales per element
    # Order: between two passes over the same tensor run at least 150 MB of
    # other traffic (more than the 129 MB L2), within a step and across steps,
    # so no pass is served from L2 by the previous one.
    return [
        ("W1 amax", "k_amax_tensor<bf16>", 0, e1 * 2),
        ("A amax", "k_amax_tensor<bf16>", 0, ea * 2),
        ("W2 amax", "k_amax_tensor<bf16>", 0, e2 * 2),
        ("W1 SR+EF 1x16", "k_rows<bf16, plain, SR, EF>", e1, e1 * (2 + 4 + 4 + q)),
        ("A 4o6 1x16", "k_rows<bf16, MAE>", ea, ea * (2 + q)),
        ("W2 SR+EF 16x16", "k_band16<bf16, plain, SR, EF>", e2, e2 * (2 + 4 + 4 + q)),
        ("W1 4o6 16x16 row+col", "k_tile_ts<bf16, MAE>", e1, e1 * (2 + 2 * q)),
        ("A RTN 1x16", "k_rows<bf16, plain, RTN>", ea, ea * (2 + q)),
        ("W2 4o6 16x16 row+col", "k_tile_ts<bf16, MAE>", e2, e2 * (2 + 2 * q)),
        ("A dequantize", "k_dequant<bf16>", ea, ea * (q + 2)),
        ("W2 SR 1x16", "k_rows<bf16, plain, SR>", e2, e2 * (2 + q)),
    ]


# ---------------------------------------------------------------------------------------
def clocks_sampler_start(path):
    try:
        f = open(path, "w")
        return subprocess.Popen(
            ["nvidia-smi", "--query-gpu=index,clocks.sm,clocks.max.sm,power.draw,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap", "--format=csv,noheader,nounits", "-lms", "200"],
            stdout=f, stderr=subprocess.DEVNULL), f
    except (OSError, FileNotFoundError):
        return None, None


def clocks_sampler_stop(proc, f, path, gpu_index):
    if proc is None:
        return None
    proc.terminate()
    try:
        proc.wait(timeout=5)
    except subprocess.TimeoutExpired:
        proc.kill()
    f.close()
    sm, smax, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    rows = [[s.strip() for s in line.split(",")] for line in open(path)]
    rows = [r for r in rows if len(r) >= 9]
    if any(r[0] == str(gpu_index) for r in rows) and len({r[0] for r in rows}) > 1:
        rows = [r for r in rows if r[0] == str(gpu_index)]
    for parts in rows:
        try:
            sm.append(float(parts[1]))
            smax.append(float(parts[2]))
        except ValueError:
            continue
        for n, v in zip(names, parts[5:9]):
            if v.lower() == "active":
                reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
            "samples": len(sm)}


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


def ncu_traffic(kernel_name):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, when it was taken on the current kernel source."""
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    except (OSError, ValueError):
        return None
    from nvfp4_block_quantization_quantize_gb300.build import source_digest
    ent = rec.get(kernel_name)
    if not ent or ent.get("source_digest") != source_digest():
        return None
    return ent.get("dram_bytes_per_launch_full_size")


# ---------------------------------------------------------------------------------------
_C5 = None


def c5_inputs():
    global _C5
    if _C5 is None:
        import nvfp4_workloads as W
        _C5 = W.C5()
    return _C5


def _oracle_step(oracle, W1, W2, A):
    """Every call of the step on the oracle; returns the outputs."""
    r1 = np.zeros(W1.shape, np.float32)
    r2 = np.zeros(W2.shape, np.float32)
    out = [oracle.quantize(W1, rounding=oracle.SR, residual=r1, seed=0, step=7),
           oracle.quantize(W2, block=oracle.BLOCK_16X16, rounding=oracle.SR, residual=r2, seed=0, step=7)]
    qa = oracle.quantize(A, gamax_mode=oracle.GAMAX_TENSOR, err_mode=oracle.ERR_MAE, scale_bound=256.0)
    out.append(qa)
    out.append(oracle.quantize(W1, block=oracle.BLOCK_16X16, gamax_mode=oracle.GAMAX_TENSOR,
                               err_mode=oracle.ERR_MAE, scale_bound=256.0, colwise=True))
    out.append(oracle.quantize(W2, block=oracle.BLOCK_16X16, gamax_mode=oracle.GAMAX_TENSOR,
                               err_mode=oracle.ERR_MAE, scale_bound=256.0, colwise=True))
    out.append(oracle.quantize(A))
    out.append(oracle.quantize(W2, rounding=oracle.SR, seed=0, step=7))
    out.append({"dq": oracle.dequantize(qa["codes"], qa["scales"], *A.shape, gamax_mode=oracle.GAMAX_TENSOR_GIVEN,
                                        gamax=qa["gamax"], scale_bound=256.0), "r1": r1, "r2": r2})
    return out


def cpu_baseline(sample_rows=2048, threads=(1, 0)):
    """The oracle as it stands on a bounded sample of the step -- the first
    `sample_rows` rows of each tensor (16-row aligned), every call -- once per
    thread count in `threads` (0 = every host core); the runs must give the
    same bytes.  Returns the all-core figure with the single-thread one beside it."""
    import oracle
    c5 = c5_inputs()
    W1, W2, A = (np.ascontiguousarray(c5.W1[:sample_rows]), np.ascontiguousarray(c5.W2[:sample_rows]),
                 np.ascontiguousarray(c5.A[:sample_rows]))
    plan = step_plan(*W1.shape, *W2.shape, *A.shape)
    total_bytes = sum(b for _, _, _, b in plan)
    total_elems = sum(e for _, _, e, _ in plan)
    runs, ref = {}, None
    for t in threads:
        with oracle.using_threads(t) as n:
            t0 = time.perf_counter()
            out = _oracle_step(oracle, W1, W2, A)
            dt = time.perf_counter() - t0
        flat = [v for d in out for v in d.values() if v is not None]
        if ref is None:
            ref = flat
        elif not all(np.array_equal(a.view(np.uint8), b.view(np.uint8)) for a, b in zip(ref, flat)):
            raise AssertionError("oracle: thread counts gave different bytes")
        runs[n] = dt
    cores = max(runs)
    dt = runs[cores]
    return {"value": total_bytes / dt / GB, "unit": "GB/s", "gelem_per_s": total_elems / dt / GB,
            "cores": cores, "kind": "oracle", "seconds_per_sample_step": dt,
            "single_thread_value": total_bytes / runs[min(runs)] / GB,
            "sample": f"first {sample_rows} rows of W1, W2 and A (every call of the step), C++ oracle on "
                      f"{cores} threads (single-thread run beside it: bit-identical)"}


def run_reference(args, rank, world):
    """--impl reference: the CPU oracle as it stands, on a bounded sample."""
    if rank != 0:
        return
    if args.warmup > 0:
        cpu_baseline(sample_rows=16, threads=(0,))
    times = []
    res = None
    for _ in range(args.steps):
        res = cpu_baseline(sample_rows=256, threads=(0,))
        times.append(res["seconds_per_sample_step"])
    val = res["value"]
    line = {"impl": "reference", "metric": METRIC,
            "value": round(val, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * statistics.median(times), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "gelem_per_s": round(res["gelem_per_s"], 6),
            "config": {"workload": WORKLOAD, "sample": res["sample"]},
            "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": res["cores"], "kind": "oracle",
                             "sample": res["sample"]},
            "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def mm_measurement(nv, torch, out, Ma, Ka, M2, K2, peaks, iters=5):
    """The FP4 product consumer (not part of the step): C = A W2^T with the
    step's round-to-nearest A codes and stochastic-rounding W2 codes, timed with
    CUDA events; against the fp4 dense peak taken as the measured bf16 peak x
    the nominal fp4 / bf16 ratio (13.5 / 2.25)."""
    sa = nv.nvfp4_scales_to_mma(out["sar"])
    sb = nv.nvfp4_scales_to_mma(out["s2s"])
    M, N, K = Ma, M2, Ka
    y = torch.empty((M, N), dtype=torch.bfloat16, device=out["car"].device)
    run = lambda: nv.nvfp4_mm(out["car"], sa, out["c2s"], sb, M, N, K, out=y)   # noqa: E731
    for _ in range(2):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        run()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / iters
    flops = 2.0 * M * N * K
    peak = (peaks["bf16_tflops"] if peaks else 1900.0) * 13.5 / 2.25
    res = {"kernel": "k_mm<bf16 out>", "shape_mnk": [M, N, K], "ms": round(ms, 4),
           "tflops": round(flops / ms / 1e9, 1), "peak_tflops": round(peak, 1),
           "frac": round(flops / ms / 1e9 / peak, 4),
           "peak_source": ("measured" if peaks else "fallback") + " bf16 x nominal fp4/bf16 ratio 6"}
    try:
        from nvfp4_block_quantization_quantize_gb300.consumers import fp4_mm, to_fp4_operands
        qa, qb = to_fp4_operands({"codes": out["car"], "scales": out["sar"]}), \
            to_fp4_operands({"codes": out["c2s"], "scales": out["s2s"]})
        for _ in range(2):
            fp4_mm(qa, qb)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(iters):
            fp4_mm(qa, qb)
        e1.record()
        torch.cuda.synchronize()
        lms = e0.elapsed_time(e1) / iters
        res["library_scaled_mm_tflops"] = round(flops / lms / 1e9, 1)
    except Exception as e:                                    # noqa: BLE001
        res["library_scaled_mm_tflops"] = None
        res["library_note"] = str(e).splitlines()[0][:120]
    return res


def c4_measurement(nv, torch, dev, peaks, iters=10, bounds=(256.0, 448.0)):
    """The other large graded configuration, timed beside the step (not part of
    it): fp32 [8192,8192] Student-t(3) (seed 3), four-over-six 16x16 MSE with a
    given per-tensor amax, rowwise + columnwise outputs from one read, bounds
    256 and 448.  The input (256 MiB) is larger than L2."""
    import nvfp4_workloads as wl
    x = torch.from_numpy(wl.c4()).to(dev)
    M, K = x.shape
    g = nv.nvfp4_amax(x)
    outs = dict(codes=torch.empty((M, K // 2), dtype=torch.uint8, device=dev),
                scales=torch.empty((M, K // 16), dtype=torch.uint8, device=dev),
                codes_col=torch.empty((K, M // 2), dtype=torch.uint8, device=dev),
                scales_col=torch.empty((K, M // 16), dtype=torch.uint8, device=dev))
    q = 0.5 + 1 / 16
    nbytes = M * K * (4 + 2 * q)
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    res = []
    for bound in bounds:
        run = lambda: nv.nvfp4_quantize(x, block="16x16", err_mode="mse", gamax_mode="tensor_given",   # noqa: E731
                                        gamax=g, scale_bound=bound, colwise=True, **outs)
        for _ in range(3):
            run()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(iters):
            run()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / iters
        res.append({"bound": bound, "ms": round(ms, 4), "GB/s": round(nbytes / (ms * 1e-3) / GB, 1),
                    "frac_of_peak": round(nbytes / (ms * 1e-3) / GB / peak, 3)})
    del x, outs
    return {"workload": "c4: fp32 [8192,8192] Student-t(3) seed 3, four-over-six 16x16 MSE, "
                        "per-tensor amax given, rowwise + columnwise", "kernel": "k_tile_ts4<f32, MSE>",
            "algorithmic_bytes": int(nbytes), "runs": res}


def run_mm_only(args, local_rank):
    import torch
    import nvfp4_block_quantization_quantize_gb300 as nv
    torch.cuda.set_device(local_rank)
    nv.build()
    nv.load_library()
    c5 = c5_inputs()
    dev = torch.device("cuda", local_rank)
    up = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)   # noqa: E731
    A, W2 = up(c5.A), up(c5.W2)
    qa = nv.nvfp4_quantize(A)
    q2 = nv.nvfp4_quantize(W2, rounding="sr", seed=0, step=7)
    out = {"car": qa["codes"], "sar": qa["scales"], "c2s": q2["codes"], "s2s": q2["scales"]}
    mm = mm_measurement(nv, torch, out, A.shape[0], A.shape[1], W2.shape[0], W2.shape[1], measured_peaks(),
                        iters=args.steps)
    print(json.dumps({"metric": "fp4 GEMM TFLOP/s", "value": mm["tflops"], "unit": "TFLOP/s",
                      "higher_is_better": True, "fp4_mm": mm}), flush=True)


def rowcol_measurement(nv, torch, W1, peaks, iters=10, variants=None):
    """Plain quantization with rowwise AND columnwise outputs from one read
    (timed beside the step, not part of it), on the step's W1 [4096,14336]
    bf16: round-to-nearest and stochastic rounding, 1x16 and 16x16 (the
    stochastic draws keyed on x's index, shared by both outputs)."""
    M, K = W1.shape
    dev = W1.device
    outs = dict(codes=torch.empty((M, K // 2), dtype=torch.uint8, device=dev),
                scales=torch.empty((M, K // 16), dtype=torch.uint8, device=dev),
                codes_col=torch.empty((K, M // 2), dtype=torch.uint8, device=dev),
                scales_col=torch.empty((K, M // 16), dtype=torch.uint8, device=dev))
    nbytes = M * K * (2 + 2 * (0.5 + 1 / 16))
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    res = []
    for name, kw in (("RTN 1x16", dict(block="1x16")), ("RTN 16x16", dict(block="16x16")),
                     ("SR 1x16", dict(block="1x16", rounding="sr", seed=0, step=7)),
                     ("SR 16x16", dict(block="16x16", rounding="sr", seed=0, step=7))):
        if variants and name not in variants:
            continue
        run = lambda: nv.nvfp4_quantize(W1, colwise=True, **kw, **outs)   # noqa: E731
        for _ in range(3):
            run()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(iters):
            run()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / iters
        res.append({"variant": name, "ms": round(ms, 4), "GB/s": round(nbytes / (ms * 1e-3) / GB, 1),
                    "frac_of_peak": round(nbytes / (ms * 1e-3) / GB / peak, 3)})
    return {"workload": "W1 [4096,14336] bf16, rowwise + columnwise, no global scale",
            "algorithmic_bytes": int(nbytes), "runs": res}


def _time_calls(torch, run, iters, warm=3):
    for _ in range(warm):
        run(0)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(iters):
        run(i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def _time_graph(torch, run, calls, reps=10):
    """Mean time per call of `calls` calls captured in one CUDA graph and
    replayed `reps` times (for calls too short to time one launch at a time:
    the replay leaves out the host's per-call work)."""
    for i in range(3):
        run(i)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for i in range(calls):
                run(i)
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (reps * calls)


def variants_measurement(nv, torch, W1, W2, A, peaks, iters=10, only=None):
    """Graded variants outside the step, each timed alone with CUDA events
    (mean of `iters` back-to-back calls; algorithmic bytes as in the step):
    SR + error feedback on every c5 tensor in both block shapes, and the c3
    four-over-six 1x16 configuration (bf16 [2048,7168], 72 columns x50, seed
    2: MAE and MSE, bound 256, per-tensor and per-row amax given) over 8
    rotating copies (235 MB, larger than L2).  Also the c2 stored-weight step
    (qdq of a bf16 [1024,1024] weight with an fp32 residual), reported in
    microseconds.  The c3 and c2 calls are timed from a CUDA-graph replay of
    back-to-back calls: one call takes less device time than the host needs
    to issue it."""
    import nvfp4_workloads as wl
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    q = 0.5 + 1 / 16
    res = []

    def add(name, kernel, nbytes, ms, elems):
        res.append({"variant": name, "kernel": kernel, "ms": round(ms, 4),
                    "GB/s": round(nbytes / (ms * 1e-3) / GB, 1),
                    "frac_of_peak": round(nbytes / (ms * 1e-3) / GB / peak, 3),
                    "gelem_per_s": round(elems / (ms * 1e-3) / GB, 2)})

    for tname, x in (("W1", W1), ("W2", W2), ("A", A)):
        M, K = x.shape
        r = torch.zeros((M, K), dtype=torch.float32, device=x.device)
        c = torch.empty((M, K // 2), dtype=torch.uint8, device=x.device)
        s = torch.empty((M, K // 16), dtype=torch.uint8, device=x.device)
        for blk in ("1x16", "16x16"):
            name = f"{tname} SR+EF {blk}"
            if only and only not in name:
                continue
            ms = _time_calls(torch, lambda i: nv.nvfp4_quantize(x, block=blk, rounding="sr", residual=r, seed=0,
                                                                 step=i, codes=c, scales=s), iters)
            add(name, f"{'k_rows' if blk == '1x16' else 'k_band16'}<bf16, plain, SR, EF>",
                M * K * (2 + 4 + 4 + q), ms, M * K)
        del r, c, s
    dev = A.device
    c3 = wl.c3()
    copies = [torch.from_numpy(c3.view(np.int16)).view(torch.bfloat16).to(dev) for _ in range(8)]
    M, K = c3.shape
    amax_t = nv.nvfp4_amax(copies[0])
    amax_r = nv.nvfp4_amax(copies[0], per_row=True)
    c = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
    s = torch.empty((M, K // 16), dtype=torch.uint8, device=dev)
    for err in ("mae", "mse"):
        for gm, g in (("tensor_given", amax_t), ("row_given", amax_r)):
            name = f"c3 4o6 {err.upper()} 1x16 {'per-tensor' if gm == 'tensor_given' else 'per-row'}"
            if only and only not in name:
                continue
            ms = _time_graph(torch, lambda i: nv.nvfp4_quantize(copies[i % 8], gamax_mode=gm, gamax=g, err_mode=err,
                                                                 scale_bound=256.0, codes=c, scales=s), 16)
            add(name, f"k_rows<bf16, {err.upper()}>", M * K * (2 + q), ms, M * K)
    del copies
    if not only or "c2" in only:
        cfg = wl.C2()
        Wt = torch.from_numpy(cfg.W0.view(np.int16)).view(torch.bfloat16).to(dev)
        r = torch.zeros(cfg.shape, dtype=torch.float32, device=dev)
        o = torch.empty(cfg.shape, dtype=torch.bfloat16, device=dev)
        ms = _time_graph(torch, lambda i: nv.nvfp4_qdq(Wt, rounding="sr", residual=r, seed=0, step=i, out=o), 50)
        n = cfg.shape[0] * cfg.shape[1]
        add("c2 SR+EF qdq 1024x1024 (one stored-weight step)", "k_rows<bf16, plain, SR, EF, qdq>",
            n * (2 + 4 + 4 + 2), ms, n)
        res[-1]["us"] = round(ms * 1e3, 2)
    return {"note": "each variant alone, mean of back-to-back calls with CUDA events (c3, c2: CUDA-graph replay)",
            "runs": res}


def run_variants_only(args, local_rank):
    import torch
    import nvfp4_block_quantization_quantize_gb300 as nv
    torch.cuda.set_device(local_rank)
    nv.build()
    nv.load_library()
    dev = torch.device("cuda", local_rank)
    c5 = c5_inputs()
    up = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)   # noqa: E731
    v = variants_measurement(nv, torch, up(c5.W1), up(c5.W2), up(c5.A), measured_peaks(), iters=args.steps,
                             only=args.only)
    print(json.dumps({"metric": "NVFP4 quantize GB/s", "value": v["runs"][0]["GB/s"], "unit": "GB/s",
                      "higher_is_better": True, "variants": v}), flush=True)


# One call each, for profiling the kernel variants the step does not run
# (bench.py --single NAME: warm-up calls, then --steps calls, CUDA-event time).
SINGLE = {
    "f32 SR+EF 1x16": ("k_rows<f32, plain, SR, EF>", "W2f", dict(rounding="sr", seed=0, ef=True)),
    "4o6 MAE 1x16 per-row": ("k_rows<bf16, MAE> (per-row scale)", "A", dict(err_mode="mae", gamax_mode="row_given",
                                                                          scale_bound=256.0, amax="row")),
    "RTN 16x16": ("k_band16<bf16, plain, RTN>", "A", dict(block="16x16")),
    "4o6 MAE 16x16 rowwise": ("k_band16<bf16, MAE>", "W2", dict(block="16x16", err_mode="mae",
                                                                gamax_mode="tensor_given", scale_bound=256.0,
                                                                amax="tensor")),
    "RTN_STD 1x16 per-tensor": ("k_rows<bf16, plain, RTN_STD, GS>", "A", dict(rounding="rtn_std",
                                                                           gamax_mode="tensor_given",
                                                                           amax="tensor")),
    "amax per-row": ("k_amax_rows<bf16>", "A", dict(amax_only="row")),
    "qdq SR+EF 1x16": ("k_rows<bf16, plain, SR, EF, qdq>", "W2", dict(rounding="sr", seed=0, ef=True, qdq=True)),
}


def run_single(args, local_rank):
    import torch
    import nvfp4_block_quantization_quantize_gb300 as nv
    torch.cuda.set_device(local_rank)
    nv.build()
    nv.load_library()
    dev = torch.device("cuda", local_rank)
    kern, tname, kw = SINGLE[args.single]
    kw = dict(kw)
    c5 = c5_inputs()
    src = c5.W2 if tname in ("W2", "W2f") else getattr(c5, tname)
    x = torch.from_numpy(src.view(np.int16)).view(torch.bfloat16).to(dev)
    if tname == "W2f":
        x = x.float()
    M, K = x.shape
    amax = kw.pop("amax", None)
    if amax:
        kw["gamax"] = nv.nvfp4_amax(x, per_row=amax == "row")
    ef, qdq, amax_only = kw.pop("ef", False), kw.pop("qdq", False), kw.pop("amax_only", None)
    r = torch.zeros((M, K), dtype=torch.float32, device=dev) if ef else None
    c = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
    s = torch.empty((M, K // 16), dtype=torch.uint8, device=dev)
    o = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    g = torch.empty((M,), dtype=torch.float32, device=dev)
    q = 0.5 + 1 / 16
    eb = x.element_size()
    if amax_only:
        run = lambda i: nv.nvfp4_amax(x, per_row=True, out=g)   # noqa: E731
        nbytes = M * K * eb
    elif qdq:
        run = lambda i: nv.nvfp4_qdq(x, residual=r, step=i, out=o, **kw)   # noqa: E731
        nbytes = M * K * (eb + 4 + 4 + 2)
    else:
        run = lambda i: nv.nvfp4_quantize(x, residual=r, step=i, codes=c, scales=s, **kw)   # noqa: E731
        nbytes = M * K * (eb + (8 if ef else 0) + q)
    ms = _time_calls(torch, run, args.steps, warm=args.warmup)
    peak = (measured_peaks() or {}).get("hbm_gbs", 6800.0)
    print(json.dumps({"single": args.single, "kernel": kern, "tensor": tname, "ms": round(ms, 4),
                      "GB/s": round(nbytes / (ms * 1e-3) / GB, 1),
                      "frac_of_peak": round(nbytes / (ms * 1e-3) / GB / peak, 3)}), flush=True)


def run_c4_only(args, local_rank):
    import torch
    import nvfp4_block_quantization_quantize_gb300 as nv
    torch.cuda.set_device(local_rank)
    nv.build()
    nv.load_library()
    dev = torch.device("cuda", local_rank)
    c4 = c4_measurement(nv, torch, dev, measured_peaks(), iters=args.steps, bounds=(256.0,))
    run = c4["runs"][0]
    print(json.dumps({"metric": "NVFP4 quantize GB/s", "value": run["GB/s"], "unit": "GB/s",
                      "higher_is_better": True, "c4_rowcol": c4}), flush=True)


def run_rowcol_only(args, local_rank):
    import torch
    import nvfp4_block_quantization_quantize_gb300 as nv
    torch.cuda.set_device(local_rank)
    nv.build()
    nv.load_library()
    dev = torch.device("cuda", local_rank)
    W1 = torch.from_numpy(c5_inputs().W1.view(np.int16)).view(torch.bfloat16).to(dev)
    rc = rowcol_measurement(nv, torch, W1, measured_peaks(), iters=args.steps,
                            variants=(args.only,) if args.only else None)
    print(json.dumps({"metric": "NVFP4 quantize GB/s", "value": rc["runs"][0]["GB/s"], "unit": "GB/s",
                      "higher_is_better": True, "rowcol_plain": rc}), flush=True)


# ---------------------------------------------------------------------------------------
def run_gpu(args, rank, world, local_rank):
    import torch
    import nvfp4_block_quantization_quantize_gb300 as nv
    import nvfp4_workloads as W

    torch.cuda.set_device(local_rank)
    nv.build()
    nv.load_library()
    dev = torch.device("cuda", local_rank)

    c5 = c5_inputs()

    def up(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)

    W1, W2, A = up(c5.W1), up(c5.W2), up(c5.A)
    (M1, K1), (M2, K2), (Ma, Ka) = W1.shape, W2.shape, A.shape
    plan = step_plan(M1, K1, M2, K2, Ma, Ka)
    bytes_step = sum(b for _, _, _, b in plan)
    elems_step = sum(e for _, _, e, _ in plan)

    u8 = lambda *s: torch.empty(s, dtype=torch.uint8, device=dev)   # noqa: E731
    f32 = lambda *s: torch.empty(s, dtype=torch.float32, device=dev)  # noqa: E731
    R1 = torch.zeros((M1, K1), dtype=torch.float32, device=dev)
    R2 = torch.zeros((M2, K2), dtype=torch.float32, device=dev)
    out = {
        "c1": u8(M1, K1 // 2), "s1": u8(M1, K1 // 16),
        "c2": u8(M2, K2 // 2), "s2": u8(M2, K2 // 16),
        "ca": u8(Ma, Ka // 2), "sa": u8(Ma, Ka // 16), "ga": f32(1),
        "c1r": u8(M1, K1 // 2), "s1r": u8(M1, K1 // 16), "c1c": u8(K1, M1 // 2),
        "s1c": u8(K1, M1 // 16), "g1": f32(1),
        "c2r": u8(M2, K2 // 2), "s2r": u8(M2, K2 // 16), "c2c": u8(K2, M2 // 2),
        "s2c": u8(K2, M2 // 16), "g2": f32(1),
        "car": u8(Ma, Ka // 2), "sar": u8(Ma, Ka // 16),
        "c2s": u8(M2, K2 // 2), "s2s": u8(M2, K2 // 16),
        "da": torch.empty((Ma, Ka), dtype=torch.bfloat16, device=dev),
    }
    stream = torch.cuda.current_stream(dev)
    o = out

    def step(t, ev=None, only=args.only):
        calls = {
            "W1 SR+EF 1x16": lambda: nv.nvfp4_quantize(W1, rounding="sr", residual=R1, seed=0, step=t,
                                                       codes=o["c1"], scales=o["s1"]),
            "W2 SR+EF 16x16": lambda: nv.nvfp4_quantize(W2, block="16x16", rounding="sr", residual=R2, seed=0,
                                                        step=t, codes=o["c2"], scales=o["s2"]),
            "A amax": lambda: nv.nvfp4_amax(A, out=o["ga"]),
            "A 4o6 1x16": lambda: nv.nvfp4_quantize(A, gamax_mode="tensor_given", gamax=o["ga"], err_mode="mae",
                                                    scale_bound=256.0, codes=o["ca"], scales=o["sa"]),
            "W1 amax": lambda: nv.nvfp4_amax(W1, out=o["g1"]),
            "W1 4o6 16x16 row+col": lambda: nv.nvfp4_quantize(W1, block="16x16", gamax_mode="tensor_given",
                                                              gamax=o["g1"], err_mode="mae", scale_bound=256.0,
                                                              colwise=True, codes=o["c1r"], scales=o["s1r"],
                                                              codes_col=o["c1c"], scales_col=o["s1c"]),
            "W2 amax": lambda: nv.nvfp4_amax(W2, out=o["g2"]),
            "W2 4o6 16x16 row+col": lambda: nv.nvfp4_quantize(W2, block="16x16", gamax_mode="tensor_given",
                                                              gamax=o["g2"], err_mode="mae", scale_bound=256.0,
                                                              colwise=True, codes=o["c2r"], scales=o["s2r"],
                                                              codes_col=o["c2c"], scales_col=o["s2c"]),
            "A RTN 1x16": lambda: nv.nvfp4_quantize(A, codes=o["car"], scales=o["sar"]),
            "W2 SR 1x16": lambda: nv.nvfp4_quantize(W2, rounding="sr", seed=0, step=t, codes=o["c2s"],
                                                    scales=o["s2s"]),
            "A dequantize": lambda: nv.nvfp4_dequantize(o["ca"], o["sa"], Ma, Ka, gamax_mode="tensor_given",
                                                        gamax=o["ga"], scale_bound=256.0, out=o["da"]),
        }
        for i, (name, _, _, _) in enumerate(plan):
            c = calls[name]
            if only and only not in name:
                continue
            if ev is not None:
                ev[i][0].record(stream)
            c()
            if ev is not None:
                ev[i][1].record(stream)

    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()

    for t in range(args.warmup):             # every call, so the amaxes a selected call reads exist
        step(t, only=None)
    torch.cuda.synchronize()

    nsteps = args.steps
    # per-call events come from a separate set of steps: an event recorded
    # between two kernels keeps the second from starting while the first
    # finishes (programmatic dependent launch), so the timed steps carry none
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in plan] for _ in range(nsteps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk_path = os.path.join(tempfile.gettempdir(), f"nvfp4_bench_clocks_rank{rank}.csv")
    os.makedirs(os.path.dirname(clk_path), exist_ok=True)
    graph = None
    if args.graph:
        # the K timed steps (their own step indices) captured as one CUDA
        # graph: the same launches, issued without the host's per-call work
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                for k in range(nsteps):
                    step(args.warmup + k)
        stream.wait_stream(side)
        torch.cuda.synchronize()
    proc, fh = clocks_sampler_start(clk_path)
    time.sleep(0.5 if proc else 0)
    barrier()
    torch.cuda.synchronize()
    start.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for k in range(nsteps):
            step(args.warmup + k)
    stop.record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = clocks_sampler_stop(proc, fh, clk_path, local_rank)
    total_ms = start.elapsed_time(stop)
    # the per-call breakdown: each instrumented step starts behind a ~1 ms
    # device spin, so the host has issued every call (and its events) before
    # the first one runs and no call's time includes the host's issue latency
    spin = getattr(torch.cuda, "_sleep", None)
    for k in range(nsteps):
        if spin is not None:
            spin(2_000_000)
        step(args.warmup + nsteps + k, evs[k])
    torch.cuda.synchronize()
    ran = [not args.only or args.only in name for name, _, _, _ in plan]
    per_call_ms = [statistics.mean(evs[k][i][0].elapsed_time(evs[k][i][1]) for k in range(nsteps))
                   if ran[i] else 0.0 for i in range(len(plan))]
    if args.only:
        plan = [p if r else (p[0], p[1], 0, 0) for p, r in zip(plan, ran)]
        bytes_step = sum(b for _, _, _, b in plan)
        elems_step = sum(e for _, _, e, _ in plan)
    if dist is not None:
        tt = torch.tensor([total_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total_ms = float(tt.item())
    ms_per_step = total_ms / nsteps
    value = world * bytes_step / (ms_per_step * 1e-3) / GB
    gelem = world * elems_step / (ms_per_step * 1e-3) / GB

    # ---- end to end: host (pinned) buffers through the public API ----
    e2e = None
    if args.e2e_steps > 0:
        pin = lambda t: t.cpu().pin_memory()   # noqa: E731
        hW1, hW2, hA = pin(W1), pin(W2), pin(A)
        hR1, hR2 = pin(R1), pin(R2)
        nbytes = lambda *ts: sum(t.numel() * t.element_size() for t in ts)   # noqa: E731
        h2d, d2h = [0], [0]

        def e2e_step(t):
            # every call of the step on host buffers, non-blocking: each call's
            # inputs go in while the previous calls' results come back.  Steps
            # are issued back to back: a step's uploads of the residuals that
            # the previous step writes back wait for those writes (the
            # binding's pending-write table), and every result reaches host
            # memory before the timed region ends
            nb = dict(non_blocking=True)
            outs = []
            outs.append(nv.nvfp4_quantize(hW1, rounding="sr", residual=hR1, seed=0, step=t, **nb))
            outs.append(nv.nvfp4_quantize(hW2, block="16x16", rounding="sr", residual=hR2, seed=0,
                                          step=t, **nb))
            qa = nv.nvfp4_quantize(hA, gamax_mode="tensor", err_mode="mae", scale_bound=256.0, **nb)
            outs.append(qa)
            outs.append(nv.nvfp4_quantize(hW1, block="16x16", gamax_mode="tensor", err_mode="mae",
                                          scale_bound=256.0, colwise=True, **nb))
            outs.append(nv.nvfp4_quantize(hW2, block="16x16", gamax_mode="tensor", err_mode="mae",
                                          scale_bound=256.0, colwise=True, **nb))
            outs.append(nv.nvfp4_quantize(hA, **nb))
            outs.append(nv.nvfp4_quantize(hW2, rounding="sr", seed=0, step=t, **nb))
            dq = nv.nvfp4_dequantize(qa["codes"], qa["scales"], Ma, Ka, gamax_mode="tensor_given",
                                     gamax=qa["gamax"], scale_bound=256.0, **nb)
            # bytes copied in: each call's own inputs (W1 twice, W2 three
            # times, A twice, both residuals, A's codes and scales again)
            h2d[0] = (nbytes(hW1, hR1, hW2, hR2, hA, hW1, hW2, hA, hW2) + nbytes(qa["codes"], qa["scales"]))
            d2h[0] = (sum(nbytes(v) for d in outs for v in d.values()) + nbytes(dq, hR1, hR2))

        # untimed: the same back-to-back steps once, so that the pinned host
        # buffers of K steps in flight are allocated before the timed ones
        for k in range(args.e2e_steps):
            e2e_step(k)
        nv.nvfp4_synchronize()
        torch.cuda.synchronize()
        barrier()
        t0 = time.perf_counter()
        for k in range(args.e2e_steps):
            e2e_step(args.e2e_steps + k)
        nv.nvfp4_synchronize()
        torch.cuda.synchronize()
        barrier()
        dt = (time.perf_counter() - t0) / args.e2e_steps
        if dist is not None:
            tt = torch.tensor([dt], device=dev)
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            dt = float(tt.item())
        e2e = {"value": round(world * bytes_step / dt / GB, 3), "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d[0]), "d2h_bytes_per_step": int(d2h[0]),
               "ms_per_step": round(dt * 1e3, 3)}

    if rank != 0:
        return
    # ---- roofline of the dominant kernel: the largest total time per step ----
    per_kernel = {}
    for (_, kern, _, b), ms in zip(plan, per_call_ms):
        if ms > 0:
            tot = per_kernel.setdefault(kern, [0.0, 0.0, 0])
            tot[0] += ms
            tot[1] += b
            tot[2] += 1
    kern = max(per_kernel, key=lambda k: per_kernel[k][0])
    ms_k, bytes_k, launches_k = per_kernel[kern]
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    achieved = (bytes_k / launches_k) / (ms_k / launches_k * 1e-3) / GB
    roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": ncu_traffic(kern),
                "kernel": kern, "launches_per_step": launches_k,
                "peak_source": "measured" if peaks else "fallback",
                "algorithmic_bytes_per_launch": int(bytes_k / launches_k),
                "ms_per_launch": round(ms_k / launches_k, 4),
                "share_of_step": round(ms_k / sum(per_call_ms), 3)}
    calls = [{"call": n, "kernel": k, "ms": round(ms, 4), "GB/s": round(b / (ms * 1e-3) / GB, 1),
              "frac_of_peak": round(b / (ms * 1e-3) / GB / peak, 3)}
             for (n, k, _, b), ms in zip(plan, per_call_ms) if ms > 0]
    mm = c4 = rc = var = None
    if not args.only:
        mm = mm_measurement(nv, torch, o, Ma, Ka, M2, K2, peaks)
        c4 = c4_measurement(nv, torch, dev, peaks)
        rc = rowcol_measurement(nv, torch, W1, peaks)
        var = variants_measurement(nv, torch, W1, W2, A, peaks)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline()
        cpu = {"value": round(cb["value"], 4), "unit": "GB/s", "cores": cb["cores"],
               "kind": "oracle", "sample": cb["sample"],
               "single_thread_value": round(cb["single_thread_value"], 4)}
    line = {
        "metric": METRIC,
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": nsteps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded numpy generators; no dataset)",
        "gelem_per_s": round(gelem, 3),
        "config": {"workload": WORKLOAD, "bytes_per_step": int(bytes_step),
                   "elements_per_step": int(elems_step),
                   "l2": "inputs larger than L2: each step streams ~2.7 GB and the calls are ordered "
                         "so that at least 150 MB of other traffic separates two passes over the same "
                         "tensor (the quantize passes after the amax passes included), within a step "
                         "and across steps",
                   "parallelism": f"{world} independent replica(s), no data-path collective",
                   "launch": ("the K timed steps captured once as a CUDA graph and replayed (same kernels and "
                              "arguments, each step its own step index)" if args.graph else
                              "calls issued one by one from Python")},
        # a per-tensor amax call launches two kernels (the zero, then the amax)
        "gpu_launches": nsteps * sum(2 if kern.startswith("k_amax_tensor") else 1
                                     for name, kern, _, _ in plan if not args.only or args.only in name),
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks, "calls": calls,
        "fp4_mm": mm, "c4_rowcol": c4, "rowcol_plain": rc, "variants": var,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if world > 1 and rank != 0:
            return
        run_reference(args, rank, world)
        return
    if args.mm_only:
        if rank == 0:
            run_mm_only(args, local_rank)
        return
    if args.c4_only:
        if rank == 0:
            run_c4_only(args, local_rank)
        return
    if args.rowcol_only:
        if rank == 0:
            run_rowcol_only(args, local_rank)
        return
    if args.variants_only:
        if rank == 0:
            run_variants_only(args, local_rank)
        return
    if args.single:
        if rank == 0:
            run_single(args, local_rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    run_gpu(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
