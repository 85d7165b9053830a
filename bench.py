"""Benchmark of the MXFP8 / NVFP4 quantizer path on GB300.

One step = one pass of every operation of the path over one batch of the
activation workload X [8192 x 4096] bf16 (N(0,1) with 0.1% of entries x100):

  1. mxfp8_quantize_rowcol   rowwise 1x32 + columnwise 32x1 copies, one pass,
                             E8M0 scales in the swizzled tensor-core layout
  2. dequantize_mxfp8        of the rowwise copy and of the columnwise copy
  3. nvfp4_quantize_per_token X as 8192 tokens x 4096 hidden (FP32 scale per
                             token, E4M3 per 16, packed E2M1)
  4. dequantize_nvfp4        of (3), per-token scales
  5. nvfp4_quantize_weight_shared  X as 8 gate/up pairs of [1024 x 2048]
                             parts (the MoE layer's hidden size as K), each
                             pair under one FP32 scale
  6. dequantize_nvfp4        of (5), per-group scales

The rowcol kernel runs first and alone; then the MXFP8 dequantizations,
the per-token chain and the weight chain run concurrently on three
streams and join before the next step.

value = algorithmic bytes of the step (bf16 read + codes / scales written,
or codes / scales read + bf16 written) / device time, in GB/s.  Inputs are
resident in HBM; every kernel reads data last touched at least one full
step (~680 MB of traffic) earlier (three rotating input copies, two
rotating output sets), so nothing is served from the 126 MB L2.  The
roofline line is the kernel with the largest share of a serial per-kernel
pass, timed by events on its own stream inside the timed region.  The
`shapes` lines time every kernel alone at the full size of each workload
it is specified on, over rotating buffer sets, write-back included.

--profile NAME launches one workload's kernel alone (the ncu harness).
--impl reference times the CPU oracle on a bounded sample of the same
workload (the oracle is the reference implementation of this path).

--impl reference times the CPU oracle on a bounded sample of the same
workload (the oracle is the reference implementation of this path).
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import ctypes
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("quantize GB/s and % of GB300 HBM peak (bytes in + codes/scales "
          "out), bit-exact")
UNIT = "GB/s"
M, K = 8192, 4096
# For the weight quantizer X is viewed as [16384 x 2048] (the MoE layer's
# hidden size as K): 8 gate/up pairs of two [1024 x 2048] parts, each pair
# under one FP32 scale.
WK = 2048
PAIRS = 8
PART_ROWS = M * K // WK // (2 * PAIRS)    # 1024 rows per part
WORKLOAD = ("MXFP8 rowwise+columnwise quantize (one pass) + both MXFP8 "
            "dequantizes + NVFP4 per-token quantize/dequantize + NVFP4 "
            "shared-scale weight quantize/dequantize of an activation "
            "[8192 x 4096] bf16, N(0,1) with 0.1% entries x100 (as weights: "
            "8 gate/up pairs of [1024 x 2048] parts)")


# --------------------------------------------------------------------------
# Algorithmic bytes per operation.
# --------------------------------------------------------------------------
def op_bytes():
    """Algorithmic bytes of each of the step's operations, in the order the
    per-kernel pass runs them."""
    n = M * K
    return {
        "mxfp8_quantize_rowcol": n * 2 + 2 * (n + n // 32),
        "dequantize_mxfp8_row": n + n // 32 + n * 2,
        "dequantize_mxfp8_col": n + n // 32 + n * 2,
        "nvfp4_quantize_per_token": n * 2 + n // 2 + n // 16 + 4 * M,
        "dequantize_nvfp4_tokens": n // 2 + n // 16 + 4 * M + n * 2,
        "nvfp4_quantize_weight_shared": n * 2 + n // 2 + n // 16 + 4 * PAIRS,
        "dequantize_nvfp4_weights": n // 2 + n // 16 + 4 * PAIRS + n * 2,
    }


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# --------------------------------------------------------------------------
# Clock sampling during the timed region.
# --------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,"
         "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        load = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# GPU arm.
# --------------------------------------------------------------------------
def max_over_ranks(value, dist, device):
    """Max of a per-rank float over all ranks (the rank-local value when not
    distributed)."""
    import torch
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(step_bytes, steps, world, ms_max):
    """Whole-job GB/s: every rank processes `step_bytes` per step, and the
    job takes as long as its slowest rank."""
    return step_bytes * steps * world / (ms_max / 1e3) / 1e9


def dist_setup(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n_gpus and world > 1:
        raise SystemExit(f"--gpus {n_gpus} but WORLD_SIZE={world}")
    return rank, world, local


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import nvfp4_quantizers_gb300 as q
    import workloads as W
    from nvfp4_quantizers_gb300 import build
    build.build()

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    x_bits = W.mxfp8_random(M, K, seed=rank)
    x_host = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16)
    X = [x_host.to(dev) for _ in range(3)]          # rotating input copies
    stream = torch.cuda.Stream(dev)
    lay = q.SCALE_SWIZZLED

    def new_outputs():
        return {
            "rc": torch.empty((M, K), dtype=torch.uint8, device=dev),
            "rs": torch.empty(q.scale_bytes(M, K // 32), dtype=torch.uint8, device=dev),
            "cc": torch.empty((K, M), dtype=torch.uint8, device=dev),
            "cs": torch.empty(q.scale_bytes(K, M // 32), dtype=torch.uint8, device=dev),
            "tc": torch.empty((M, K // 2), dtype=torch.uint8, device=dev),
            "ts": torch.empty(q.scale_bytes(M, K // 16), dtype=torch.uint8, device=dev),
            "tS": torch.empty(M, dtype=torch.float32, device=dev),
            "wc": torch.empty((PAIRS, 2 * PART_ROWS, WK // 2), dtype=torch.uint8, device=dev),
            "ws": torch.empty((PAIRS, q.scale_bytes(2 * PART_ROWS, WK // 16)), dtype=torch.uint8, device=dev),
            "wS": torch.empty(PAIRS, dtype=torch.float32, device=dev),
        }

    outs = [new_outputs(), new_outputs()]
    y_row = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    y_col = torch.empty((K, M), dtype=torch.bfloat16, device=dev)
    y_tok = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    y_w = torch.empty((PAIRS, 2 * PART_ROWS, WK), dtype=torch.bfloat16, device=dev)
    L = q.lib()
    ws_bytes = int(L.nvfp4_quantize_weight_shared_workspace_size(PAIRS))
    wsp = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    parts_tabs = []
    for xi in X:
        flat = xi.view(2 * PAIRS, PART_ROWS, WK)
        parts_tabs.append((ctypes.c_void_p * (2 * PAIRS))(
            *[flat[i].data_ptr() for i in range(2 * PAIRS)]))
    rows_tab = (ctypes.c_int64 * 2)(PART_ROWS, PART_ROWS)
    s = ctypes.c_void_p(stream.cuda_stream)
    # The step's three chains (MXFP8 quantize -> both dequantizations;
    # per-token quantize -> dequantize; weights -> dequantize) touch
    # different buffers: after the rowcol kernel (timed alone for the
    # roofline line), the other two chains fork onto their own streams and
    # join before the next step.
    # The weight chain's stream has the higher priority: its quantizer is
    # latency-bound and the longest chain, and the dequantizers (eight CTAs
    # on every SM) would otherwise hold the SMs while its CTAs wait to be
    # scheduled (5087 -> 5600 GB/s).
    side = [torch.cuda.Stream(dev), torch.cuda.Stream(dev, priority=-1)]
    s_side = [ctypes.c_void_p(x.cuda_stream) for x in side]
    ev_fork = torch.cuda.Event()
    ev_join = [torch.cuda.Event(), torch.cuda.Event()]

    def chk(st, what):
        if st != 0:
            raise RuntimeError(f"{what}: {q.status_string(st)}")

    names = list(op_bytes().keys())
    SIDE = {"nvfp4_quantize_per_token": 0, "dequantize_nvfp4_tokens": 0,
            "nvfp4_quantize_weight_shared": 1, "dequantize_nvfp4_weights": 1}

    def phase_table(ph):
        """The step's operations for buffer phase ph (outputs alternate over
        2 sets, inputs over 3): name -> (C function, arguments on the main
        stream, arguments on the operation's side stream).  Built once, so
        that a step costs the host only its launches."""
        o_new, o_old = outs[ph % 2], outs[(ph + 1) % 2]
        x0, x1 = X[ph % 3], X[(ph + 1) % 3]
        tab = parts_tabs[(ph + 2) % 3]
        t = {}

        def add(nm, fn, mk):
            side_s = s_side[SIDE[nm]] if nm in SIDE else s
            t[nm] = (fn, mk(s), mk(side_s))
        add("mxfp8_quantize_rowcol", L.mxfp8_quantize_rowcol, lambda st: (
            x0.data_ptr(), M, K, K, o_new["rc"].data_ptr(),
            o_new["rs"].data_ptr(), o_new["cc"].data_ptr(),
            o_new["cs"].data_ptr(), lay, st))
        add("dequantize_mxfp8_row", L.dequantize_mxfp8, lambda st: (
            o_old["rc"].data_ptr(), o_old["rs"].data_ptr(), M, K, lay,
            y_row.data_ptr(), st))
        add("dequantize_mxfp8_col", L.dequantize_mxfp8, lambda st: (
            o_old["cc"].data_ptr(), o_old["cs"].data_ptr(), K, M, lay,
            y_col.data_ptr(), st))
        add("nvfp4_quantize_per_token", L.nvfp4_quantize_per_token,
            lambda st: (x1.data_ptr(), M, K, K, o_new["tc"].data_ptr(),
                        o_new["ts"].data_ptr(), o_new["tS"].data_ptr(), lay,
                        st))
        add("dequantize_nvfp4_tokens", L.dequantize_nvfp4, lambda st: (
            o_old["tc"].data_ptr(), o_old["ts"].data_ptr(),
            o_old["tS"].data_ptr(), q.S_PER_ROW, 1, M, K, lay,
            y_tok.data_ptr(), st))
        add("nvfp4_quantize_weight_shared", L.nvfp4_quantize_weight_shared,
            lambda st: (PAIRS, 2, ctypes.cast(tab, ctypes.c_void_p),
                        ctypes.cast(rows_tab, ctypes.c_void_p), WK,
                        o_new["wc"].data_ptr(), o_new["ws"].data_ptr(),
                        o_new["wS"].data_ptr(), None, lay, wsp.data_ptr(),
                        wsp.numel(), st))
        add("dequantize_nvfp4_weights", L.dequantize_nvfp4, lambda st: (
            o_old["wc"].data_ptr(), o_old["ws"].data_ptr(),
            o_old["wS"].data_ptr(), q.S_PER_BATCH, PAIRS, 2 * PART_ROWS, WK,
            lay, y_w.data_ptr(), st))
        return t

    tables = [phase_table(ph) for ph in range(6)]

    def launch(fn, a, nm):
        st = fn(*a)
        if st != 0:
            raise RuntimeError(f"{nm}: {q.status_string(st)}")

    def step_serial(i, record):
        """All operations on the main stream; record[j] .. record[j + 1]
        brackets operation j (the per-kernel pass)."""
        t = tables[i % 6]
        for j, nm in enumerate(names):
            record[j].record(stream)
            fn, a, _ = t[nm]
            launch(fn, a, nm)
        record[len(names)].record(stream)

    # Concurrent order after the first operation: the MXFP8 dequantizations
    # (main stream), then each side chain dequantizing the previous step's
    # codes before quantizing this step's input, so that the step ends on
    # the kernels that leave the least dirty data in L2 for the next step.
    ORDER = ("dequantize_mxfp8_row", "dequantize_mxfp8_col",
             "mxfp8_quantize_rowcol", "dequantize_nvfp4_tokens",
             "nvfp4_quantize_per_token", "dequantize_nvfp4_weights",
             "nvfp4_quantize_weight_shared")

    FIRST = "mxfp8_quantize_rowcol"

    def step(i, bracket=None, bracketed=None):
        """One step: the rowcol kernel alone on the main stream, then the
        rest as three concurrent chains (the MXFP8 dequantizations on the
        main stream, the per-token and the weight chain on side streams)
        that join before the next step.  `bracket` (two events) is recorded
        around operation `bracketed` on the stream it runs on."""
        t = tables[i % 6]

        def run(nm, fn, a, st):
            if bracket is not None and nm == bracketed:
                bracket[0].record(st)
                launch(fn, a, nm)
                bracket[1].record(st)
            else:
                launch(fn, a, nm)
        fn, a, _ = t[FIRST]
        run(FIRST, fn, a, stream)
        ev_fork.record(stream)
        side[0].wait_event(ev_fork)
        side[1].wait_event(ev_fork)
        for nm in ORDER:
            if nm != FIRST:
                fn, _, a = t[nm]
                run(nm, fn, a, side[SIDE[nm]] if nm in SIDE else stream)
        ev_join[0].record(side[0])
        ev_join[1].record(side[1])
        stream.wait_event(ev_join[0])
        stream.wait_event(ev_join[1])

    # Our kernels per step: rowcol 1, dequant 2 + 1 + 1, per-token 1,
    # weights 1 (one kernel per call of up to 256 groups).
    launches_per_step = 1 + 2 + 1 + 1 + 1 + 1

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            if args.serial:
                step_serial(i, [torch.cuda.Event() for _ in range(8)])
            else:
                step(i)
    torch.cuda.synchronize(dev)

    # Per-kernel breakdown: a pass with events between all kernels, one
    # stream (events between kernels cost the launch overlap, so this pass
    # is not used for the headline number).  The kernel with the largest
    # share is the roofline line's kernel.
    nb = min(args.steps, 200)
    recs8 = [[torch.cuda.Event(enable_timing=True) for _ in range(8)]
             for _ in range(nb)]
    th0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(nb):
            step_serial(args.warmup + i, recs8[i])
    host_serial_ms = (time.perf_counter() - th0) * 1e3 / nb
    torch.cuda.synchronize(dev)
    per_kernel_ms = {}
    for j, nm in enumerate(names):
        per_kernel_ms[nm] = statistics.mean(
            recs8[i][j].elapsed_time(recs8[i][j + 1]) for i in range(nb))
    dom = max(names, key=lambda nm: per_kernel_ms[nm])
    if world > 1:
        dist.barrier()

    # Timed region: K steps.  The dominant kernel is bracketed by two events
    # on the stream it runs on (in the concurrent step it may share the GPU
    # with the other chains); the other kernels keep their
    # programmatic-dependent-launch overlap.  Running the rowcol kernel
    # first and alone measured best for the step (5294 GB/s against 4705
    # with the weight kernel first).
    recs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
            for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    i0 = args.warmup + nb
    with ClockSampler(local) as clk:
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            start.record(stream)
            for i in range(args.steps):
                if args.serial:
                    step_serial(i0 + i, [recs[i][0]] + [torch.cuda.Event()
                                                        for _ in range(7)])
                else:
                    step(i0 + i, recs[i], dom)
            end.record(stream)
        host_ms = (time.perf_counter() - t0) * 1e3 / args.steps
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        wall = time.perf_counter() - t0
    ms = start.elapsed_time(end)
    ms_max = max_over_ranks(ms, dist if world > 1 else None, dev)
    ob = op_bytes()
    step_bytes = sum(ob.values())
    if args.serial:
        dom_ms = per_kernel_ms[dom]
    else:
        dom_ms = statistics.mean(recs[i][0].elapsed_time(recs[i][1])
                                 for i in range(args.steps))
    peak, peak_kind = measured_peak()
    value = weak_scaling_value(step_bytes, args.steps, world, ms_max)

    # e2e through the public API: pinned host input -> device -> the step's
    # kernels -> quantized outputs back to pinned host memory.
    e2e = run_e2e(q, dev, x_bits, args) if rank == 0 else None

    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return

    total_ms = sum(per_kernel_ms.values())
    kernels = {}
    for nm in names:
        t = per_kernel_ms[nm]
        gbs = ob[nm] / (t / 1e3) / 1e9
        kernels[nm] = {"us": round(t * 1e3, 2), "GB/s": round(gbs, 1),
                       "frac": round(gbs / peak, 3),
                       "share": round(t / total_ms, 3),
                       "bytes": ob[nm]}
    traffic = load_traffic(dom)
    dom_gbs = ob[dom] / (dom_ms / 1e3) / 1e9
    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": step_config(world, args.serial),
        "pct_hbm_peak": round(100 * value / world / peak, 1),
        "roofline": {
            "kernel": dom,
            "chosen_by": "largest share of the per-kernel pass",
            "timed": "events around each launch on its own stream in the timed region",
            "bound": "hbm",
            "achieved": round(dom_gbs, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(dom_gbs / peak, 3),
            "traffic": traffic,
            "us_per_launch": round(dom_ms * 1e3, 2),
            "bytes_per_launch": ob[dom],
        },
        "kernels": kernels,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
        "e2e": e2e,
        "wall_s_timed_region": round(wall, 3),
        "host_enqueue_ms_per_step": {"timed": round(host_ms, 4),
                                     "per_kernel_pass": round(host_serial_ms, 4)},
    }
    out["gemm"] = run_gemm(q, W, dev, stream)
    if not args.no_shapes:
        out["shapes"] = run_shapes(q, W, dev, stream)
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args)
    print(json.dumps(out), flush=True)


def tensor_peaks():
    """fp8 and fp4 dense tensor peaks: the measured bf16 GEMM rate times the
    nominal fp8/bf16 (2x) and fp4/bf16 (6x) ratios."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16 = float(json.load(f)["bf16_tflops"])
        kind = "measured bf16 x nominal ratio"
    except Exception:
        bf16, kind = 1900.0, "fallback bf16 x nominal ratio"
    return {"bf16": bf16, "fp8": 2 * bf16, "fp4": 6 * bf16, "kind": kind}


def gemm_roofline(us, flops, nbytes, tensor_peak_tflops):
    """Both ceilings of a GEMM launch: tensor time at the dtype's peak and
    HBM time for its algorithmic bytes (operands, scales and fp32 C once).
    The larger one binds; frac = that time / the measured time."""
    hbm = measured_peak()[0]
    t_tensor = flops / (tensor_peak_tflops * 1e12) * 1e6
    t_hbm = nbytes / (hbm * 1e9) * 1e6
    bound = "tensor" if t_tensor >= t_hbm else "hbm"
    return {"us": round(us, 2), "TFLOP/s": round(flops / us / 1e6, 1),
            "GB/s": round(nbytes / us / 1e3, 1), "bytes": int(nbytes),
            "tensor_frac": round(t_tensor / us, 3),
            "hbm_frac": round(t_hbm / us, 3), "bound": bound,
            "frac": round(max(t_tensor, t_hbm) / us, 3)}


def run_gemm(q, W, dev, stream, reps=20):
    """The block-scaled GEMM consumers on the workloads they are specified
    for: MXFP8 A [2048 x 2048] x B [2048 x 8192]; NVFP4 4096 tokens routed
    top-8 over 128 experts against gate/up [1536 x 2048] weights."""
    import torch
    peaks = tensor_peaks()
    out = {}
    A, B = W.gemm_mxfp8_inputs(2048, 2048, 8192)
    qa = q.mxfp8_quantize_rowcol(torch.from_numpy(A.view(np.int16)).view(
        torch.bfloat16).to(dev), rowwise=True, colwise=False)
    qb = q.mxfp8_quantize_rowcol(torch.from_numpy(B.view(np.int16)).view(
        torch.bfloat16).to(dev), rowwise=False, colwise=True)

    def t_mx():
        return q.gemm_mxfp8(qa.row_codes, qa.row_scales, qb.col_codes_t,
                            qb.col_scales_t)
    ms = _time_fn(t_mx, stream, reps)
    fl = 2.0 * 2048 * 2048 * 8192
    # codes and E8M0 scales of A and B^T, fp32 C
    nb = 2048 * 2048 * (1 + 1 / 32) + 8192 * 2048 * (1 + 1 / 32) + \
        2048 * 8192 * 4
    out["mxfp8_2048x2048x8192"] = dict(
        gemm_roofline(ms * 1e3, fl, nb, peaks["fp8"]),
        peak_fp8=round(peaks["fp8"], 1))
    E, H, F = 128, 2048, 768
    tokens = W.gemm_tokens(4096, H)
    route = W.topk_routing(4096, E, 8)
    rows_by_e = [np.nonzero((route == e).any(axis=1))[0] for e in range(E)]
    padded = [((len(r) + 127) // 128) * 128 for r in rows_by_e]
    offs = np.concatenate([[0], np.cumsum(padded)])
    gathered = np.zeros((int(offs[-1]), H), np.uint16)
    for e in range(E):
        gathered[offs[e]:offs[e] + len(rows_by_e[e])] = tokens[rows_by_e[e]]
    ta = q.nvfp4_quantize_per_token(torch.from_numpy(gathered.view(np.int16))
                                    .view(torch.bfloat16).to(dev))
    wts = torch.from_numpy(np.stack(
        [np.concatenate(W.moe_expert(e, hidden=H, ffn=F)[:2])
         for e in range(E)]).view(np.int16)).view(torch.bfloat16).to(dev)
    tw = q.nvfp4_quantize_weight_shared([[wts[e]] for e in range(E)])
    del wts

    def t_nv():
        return q.gemm_nvfp4_grouped(ta.codes, ta.block_scales, ta.scales, offs,
                                    tw.codes, tw.block_scales, tw.scales)
    ms = _time_fn(t_nv, stream, reps)
    fl_routed = 2.0 * 32768 * 2 * F * H
    fl_padded = 2.0 * int(offs[-1]) * 2 * F * H
    Mp = int(offs[-1])
    # packed E2M1 + E4M3 scales of the gathered tokens and of all experts'
    # gate/up weights, per-token and per-expert FP32 scales, fp32 C
    nb = Mp * H * (0.5 + 1 / 16) + 4 * Mp + \
        E * 2 * F * H * (0.5 + 1 / 16) + 4 * E + Mp * 2 * F * 4
    out["nvfp4_grouped_4096tok_top8_128x1536x2048"] = dict(
        gemm_roofline(ms * 1e3, fl_padded, nb, peaks["fp4"]),
        **{"TFLOP/s_routed": round(fl_routed / ms / 1e9, 1),
           "padded_rows": Mp, "routed_rows": 32768,
           "peak_fp4": round(peaks["fp4"], 1)})
    # MoE expert forward up to the activation: routing gather fused into
    # the per-token quantizer, then the gate/up GEMM with SwiGLU (bf16 h).
    idx, offs2, _ = W.expert_gather_index(route, E)
    tok_dev = torch.from_numpy(tokens.view(np.int16)).view(
        torch.bfloat16).to(dev)
    idx_dev = torch.from_numpy(idx).to(dev)

    ops = _Ops(q, dev, stream)
    call_gq, _ = ops.gather_quantize(tok_dev, idx_dev)
    ms_gq = _time_fn(call_gq, stream, reps)
    tg = q.nvfp4_quantize_per_token_gather(tok_dev, idx_dev)

    def t_sw():
        return q.moe_gate_up_swiglu(tg.codes, tg.block_scales, tg.scales,
                                    offs2, tw.codes, tw.block_scales,
                                    tw.scales)
    ms_sw = _time_fn(t_sw, stream, reps)
    # the same forward with the gather in the GEMM's operand load: the
    # unique tokens quantized once (linear block scales), each routed row
    # gathered by the GEMM
    call_q1, _ = ops.per_token(tok_dev, lay=q.SCALE_LINEAR)
    ms_q1 = _time_fn(call_q1, stream, reps)
    xq = q.nvfp4_quantize_per_token(tok_dev, "linear")

    def t_swg():
        return q.moe_gate_up_swiglu_gather(xq, idx_dev, offs2, tw.codes,
                                           tw.block_scales, tw.scales)
    ms_swg = _time_fn(t_swg, stream, reps)
    Mp2 = int(offs2[-1])
    # gather-quantize: the unique tokens read once, gathered codes, block
    # scales and token scales written
    nb_gq = 4096 * H * 2 + Mp2 * H * (0.5 + 1 / 16) + 4 * Mp2
    # SwiGLU GEMM: operands as above, bf16 h [rows x F]
    nb_sw = Mp2 * H * (0.5 + 1 / 16) + 4 * Mp2 + \
        E * 2 * F * H * (0.5 + 1 / 16) + 4 * E + Mp2 * F * 2
    out["moe_gate_up_swiglu_4096tok_top8_128x768x2048"] = dict(
        gemm_roofline(ms_sw * 1e3, 2.0 * Mp2 * 2 * F * H, nb_sw,
                      peaks["fp4"]),
        **{"gather_quantize_us": round(ms_gq * 1e3, 2),
           "gather_quantize_GB/s": round(nb_gq / ms_gq / 1e6, 1),
           "gather_quantize_hbm_frac": round(
               nb_gq / ms_gq / 1e6 / measured_peak()[0], 3),
           "forward_us_materialized": round((ms_gq + ms_sw) * 1e3, 2),
           "quantize_unique_tokens_us": round(ms_q1 * 1e3, 2),
           "gather_in_gemm_us": round(ms_swg * 1e3, 2),
           "forward_us": round((ms_q1 + ms_swg) * 1e3, 2),
           "forward": ("per-token quantize of the 4096 unique tokens, then the "
                       "gate/up GEMM gathering the routed rows in its operand "
                       "load (no routed copy in HBM)"),
           "padded_rows": Mp2, "output": "bf16 h [rows x 768]"})
    # Dequantized-backward data gradient of the linear layer (2048, 2048) ->
    # 8192: dX [2048 x 2048] = dY [2048 x 8192] x W, W's columnwise MXFP8
    # copy dequantized in shared memory; beside it the path that writes the
    # bf16 dequantization to HBM and runs cuBLAS on it.
    dY = torch.from_numpy(W.gemm_tokens(2048, 8192).view(np.int16)).view(
        torch.bfloat16).to(dev)
    wq = q.mxfp8_quantize_rowcol(torch.from_numpy(W.linear_weight().view(
        np.int16)).view(torch.bfloat16).to(dev), rowwise=False, colwise=True)

    def t_dq():
        return q.gemm_bf16_mxfp8(dY, wq.col_codes_t, wq.col_scales_t)

    def t_mat():
        wt = q.dequantize_mxfp8(wq.col_codes_t, wq.col_scales_t)
        return torch.matmul(dY, wt.t())
    ms_dq = _time_fn(t_dq, stream, reps)
    ms_mat = _time_fn(t_mat, stream, reps)
    fl = 2.0 * 2048 * 2048 * 8192
    nb = 2048 * 8192 * 2 + 2048 * 8192 * (1 + 1 / 32) + 2048 * 2048 * 4
    out["bf16_x_mxfp8_dgrad_2048x8192x2048"] = dict(
        gemm_roofline(ms_dq * 1e3, fl, nb, peaks["bf16"]),
        **{"materialized_us": round(ms_mat * 1e3, 2),
           "materialized": "dequantize to bf16 in HBM, then cuBLAS bf16",
           "peak_bf16": round(peaks["bf16"], 1)})
    out["peaks_kind"] = peaks["kind"]
    return out


def _sets_for(footprint, l2, lo=2, hi=32):
    """Rotation depth: enough buffer sets (inputs + outputs of one launch
    each) that a launch's data was last touched at least 4 x L2 bytes of
    traffic earlier."""
    n = -(-4 * l2 // max(int(footprint), 1))
    return int(max(lo, min(hi, n)))


def _time_rotating(calls, stream, rounds=9, min_launches=24, warmup=3):
    """Per-launch device times (ms) of back-to-back launches that cycle over
    `calls` (each launching the kernel on its own input and output buffers,
    all on `stream`): every launch finds its inputs out of L2 and, as in a
    steady stream of launches, absorbs the write-back of the dirty lines the
    launch before it left in L2, so a kernel's own write-back is inside the
    timed region.  Each round times n launches between two events (n a
    multiple of len(calls)); returns the per-launch mean of every round."""
    import torch
    per = len(calls)
    n = per * max(1, -(-min_launches // per))
    with torch.cuda.stream(stream):
        for i in range(max(warmup, per)):
            calls[i % per]()
    torch.cuda.synchronize()
    evs = []
    with torch.cuda.stream(stream):
        for _ in range(rounds):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(n):
                calls[i % per]()
            e1.record(stream)
            evs.append((e0, e1))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) / n for a, b in evs]


def _shape_line(ms_list, nbytes, elems, peak, sets):
    ms = sorted(ms_list)
    med = statistics.median(ms)
    p10 = ms[int(0.1 * (len(ms) - 1))]
    p90 = ms[int(round(0.9 * (len(ms) - 1)))]
    gbs = nbytes / med / 1e6
    return {"us": round(med * 1e3, 2), "us_p10": round(p10 * 1e3, 2),
            "us_p90": round(p90 * 1e3, 2), "GB/s": round(gbs, 1),
            "GB/s_p10_p90": [round(nbytes / p90 / 1e6, 1),
                             round(nbytes / p10 / 1e6, 1)],
            "Gelem/s": round(elems / med / 1e6, 2),
            "frac": round(gbs / peak, 3), "bytes": int(nbytes),
            "writeback_included": True, "rotating_sets": int(sets)}


class _Ops:
    """Launchers of single library calls on preallocated buffers, straight
    through the C ABI (no allocation or Python marshalling per launch), for
    back-to-back timing."""

    def __init__(self, q, dev, stream):
        import torch
        self.torch = torch
        self.q = q
        self.L = q.lib()
        self.dev = dev
        self.s = ctypes.c_void_p(stream.cuda_stream)
        self.lay = q.SCALE_SWIZZLED

    def u8(self, n):
        return self.torch.empty(int(n), dtype=self.torch.uint8, device=self.dev)

    def chk(self, st, what):
        if st != 0:
            raise RuntimeError(f"{what}: {self.q.status_string(st)}")

    def rowcol(self, x):
        M, K = x.shape
        q = self.q
        rc, cc = self.u8(M * K), self.u8(M * K)
        rs = self.u8(q.scale_bytes(M, K // 32))
        cs = self.u8(q.scale_bytes(K, M // 32))
        args = (x.data_ptr(), M, K, K, rc.data_ptr(), rs.data_ptr(),
                cc.data_ptr(), cs.data_ptr(), self.lay, self.s)
        keep = (x, rc, rs, cc, cs)

        def call(keep=keep):
            self.chk(self.L.mxfp8_quantize_rowcol(*args), "rowcol")
        return call, (rc, rs, cc, cs)

    def dq_mxfp8(self, codes, scales):
        rows, cols = codes.shape
        y = self.torch.empty((rows, cols), dtype=self.torch.bfloat16,
                             device=self.dev)
        args = (codes.data_ptr(), scales.data_ptr(), rows, cols, self.lay,
                y.data_ptr(), self.s)
        keep = (codes, scales, y)

        def call(keep=keep):
            self.chk(self.L.dequantize_mxfp8(*args), "dequantize_mxfp8")
        return call

    def per_token(self, x, rht_flags=None, seed=2026, lay=None):
        T, H = x.shape
        q = self.q
        lay = self.lay if lay is None else lay
        c = self.u8(T * H // 2)
        bs = self.u8(q.scale_bytes(T, H // 16, lay))
        S = self.torch.empty(T, dtype=self.torch.float32, device=self.dev)
        keep = (x, c, bs, S)
        if rht_flags is None:
            args = (x.data_ptr(), T, H, H, c.data_ptr(), bs.data_ptr(),
                    S.data_ptr(), lay, self.s)

            def call(keep=keep):
                self.chk(self.L.nvfp4_quantize_per_token(*args), "per-token")
        else:
            args = (x.data_ptr(), T, H, H, ctypes.c_uint64(seed), rht_flags,
                    c.data_ptr(), bs.data_ptr(), S.data_ptr(), self.lay,
                    self.s)

            def call(keep=keep):
                self.chk(self.L.nvfp4_quantize_per_token_rht_sr(*args),
                         "per-token rht/sr")
        return call, (c, bs, S)

    def gather_quantize(self, x, idx):
        """Per-token NVFP4 of the rows idx of x (the routed copy)."""
        T_src, H = x.shape
        T = idx.numel()
        q = self.q
        c = self.u8(T * H // 2)
        bs = self.u8(q.scale_bytes(T, H // 16))
        S = self.torch.empty(T, dtype=self.torch.float32, device=self.dev)
        args = (x.data_ptr(), T_src, H, H, idx.data_ptr(), T, c.data_ptr(),
                bs.data_ptr(), S.data_ptr(), self.lay, self.s)
        keep = (x, idx, c, bs, S)

        def call(keep=keep):
            self.chk(self.L.nvfp4_quantize_per_token_gather(*args), "gather")
        return call, (c, bs, S)

    def dq_nvfp4(self, codes, bs, S, mode, batch, rows, cols):
        y = self.torch.empty(batch * rows * cols, dtype=self.torch.bfloat16,
                             device=self.dev)
        args = (codes.data_ptr(), bs.data_ptr(), S.data_ptr(), mode, batch,
                rows, cols, self.lay, y.data_ptr(), self.s)
        keep = (codes, bs, S, y)

        def call(keep=keep):
            self.chk(self.L.dequantize_nvfp4(*args), "dequantize_nvfp4")
        return call

    def weights(self, parts, G, P, part_rows, K, S_in=None):
        """parts: G * P contiguous bf16 tensors (group-major); S_in: the
        group scales to use (float32 [G] on the device) or None."""
        q = self.q
        R = sum(part_rows)
        tab = (ctypes.c_void_p * (G * P))(*[t.data_ptr() for t in parts])
        rows = (ctypes.c_int64 * P)(*part_rows)
        c = self.u8(G * R * K // 2)
        sbytes = q.scale_bytes(R, K // 16)
        bs = self.u8(G * sbytes)
        S = self.torch.empty(G, dtype=self.torch.float32, device=self.dev)
        wsb = int(self.L.nvfp4_quantize_weight_shared_workspace_size(G))
        ws = self.u8(max(wsb, 256))
        args = (G, P, ctypes.cast(tab, ctypes.c_void_p),
                ctypes.cast(rows, ctypes.c_void_p), K, c.data_ptr(),
                bs.data_ptr(), S.data_ptr(),
                None if S_in is None else S_in.data_ptr(), self.lay,
                ws.data_ptr(), ws.numel(), self.s)
        keep = (parts, tab, rows, c, bs, S, ws, S_in)

        def call(keep=keep):
            self.chk(self.L.nvfp4_quantize_weight_shared(*args), "weights")
        return call, (c, bs, S)

    def fp8blk(self, x, block_rows):
        rows, cols = x.shape
        c = self.u8(rows * cols)
        sc = self.torch.empty((rows // block_rows) * (cols // 128),
                              dtype=self.torch.float32, device=self.dev)
        args = (x.data_ptr(), rows, cols, cols, block_rows, c.data_ptr(),
                sc.data_ptr(), self.s)
        keep = (x, c, sc)

        def call(keep=keep):
            self.chk(self.L.fp8_block_quantize(*args), "fp8 block")
        return call, (c, sc)

    def fp8blk_dq(self, codes, sc, rows, cols, block_rows):
        y = self.torch.empty(rows * cols, dtype=self.torch.bfloat16,
                             device=self.dev)
        args = (codes.data_ptr(), sc.data_ptr(), rows, cols, block_rows,
                y.data_ptr(), self.s)
        keep = (codes, sc, y)

        def call(keep=keep):
            self.chk(self.L.fp8_block_dequantize(*args), "fp8 block dequant")
        return call

    def fp8blk_rt(self, codes, sc, rows, cols):
        ct = self.u8(rows * cols)
        st = self.torch.empty(cols * (rows // 128), dtype=self.torch.float32,
                              device=self.dev)
        args = (codes.data_ptr(), sc.data_ptr(), rows, cols, ct.data_ptr(),
                st.data_ptr(), self.s)
        keep = (codes, sc, ct, st)

        def call(keep=keep):
            self.chk(self.L.fp8_block_requantize_transpose(*args),
                     "fp8 block requantize-transpose")
        return call


def run_shapes(q, W, dev, stream):
    """Each quantizer and dequantizer alone at the full sizes of the
    workloads it is specified on: MXFP8 rowwise + columnwise of the four
    8192 x 4096 input classes and of the linear layer's input [2048 x 2048]
    and weight [8192 x 2048]; NVFP4 per-token on the ragged batch of 64
    sequences (lengths in [128, 4096], hidden 2048), also with the
    pretraining recipe's Hadamard transform and stochastic rounding; NVFP4
    shared-scale weights of a 128-expert MoE layer (gate/up pairs
    [2 x 768 x 2048] and down [2048 x 768]); FP8 with FP32 block scales (1x128
    tiles of the activation, 128x128 blocks of the linear weight, the tiles'
    backward-orientation conversion); and the dequantizations of each.

    Every line times back-to-back launches cycling over several sets of
    input and output buffers (at least 4 x L2 of data per cycle), so each
    launch reads its inputs from HBM and pays for its own write-back."""
    import torch
    peak = measured_peak()[0]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    ops = _Ops(q, dev, stream)
    out = {}

    def dev16(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    def line(name, calls, nbytes, elems, **extra):
        out[name] = dict(_shape_line(_time_rotating(calls, stream), nbytes,
                                     elems, peak, len(calls)), **extra)

    # MXFP8 rowwise + columnwise, then both dequantizations
    def mx(name, bits, dequant=False):
        x = dev16(bits)
        m, k = x.shape
        n = m * k
        b = 2 * n + 2 * (n + n // 32)
        sets = _sets_for(b, l2)
        built = [ops.rowcol(x if i == 0 else x.clone()) for i in range(sets)]
        line(f"mxfp8_rowcol_{name}", [c for c, _ in built], b, n)
        if dequant:
            for nm, j in (("row", 0), ("col", 2)):
                calls = []
                for _, o in built:
                    rows, cols = (m, k) if nm == "row" else (k, m)
                    calls.append(ops.dq_mxfp8(o[j].view(rows, cols), o[j + 1]))
                line(f"dequantize_mxfp8_{nm}_{m}x{k}", calls,
                     n + n // 32 + 2 * n, n)
        del built, x
        torch.cuda.empty_cache()

    for cls, gen in (("random", W.mxfp8_random), ("boundary", W.mxfp8_boundary),
                     ("zeros", W.mxfp8_zeros), ("maxes", W.mxfp8_maxes)):
        mx(f"8192x4096_{cls}", gen(8192, 4096), dequant=(cls == "random"))
    mx("2048x2048_linear_input", W.linear_input())
    mx("8192x2048_linear_weight", W.linear_weight())

    # NVFP4 per-token, ragged batch flattened
    H = 2048
    lengths = W.ragged_lengths()
    x = dev16(W.ragged_tokens(lengths, H))
    T = x.shape[0]
    tb = T * (2 * H + H // 2 + H // 16 + 4)
    sets = _sets_for(tb, l2)
    xs = [x] + [x.clone() for _ in range(sets - 1)]
    built = [ops.per_token(xi) for xi in xs]
    line(f"nvfp4_per_token_ragged_{T}x{H}", [c for c, _ in built], tb, T * H,
         sequences=int(len(lengths)))
    line(f"dequantize_nvfp4_ragged_{T}x{H}",
         [ops.dq_nvfp4(c, bs, S, q.S_PER_ROW, 1, T, H)
          for _, (c, bs, S) in built], tb, T * H)
    del built
    # the pretraining recipe's stabilizers on the same batch
    for nm, fl in (("rht", q.NVFP4_RHT), ("rht_sr", q.NVFP4_RHT | q.NVFP4_SR)):
        built = [ops.per_token(xi, rht_flags=fl) for xi in xs]
        line(f"nvfp4_per_token_{nm}_ragged_{T}x{H}", [c for c, _ in built],
             tb, T * H)
        del built
    del x, xs
    torch.cuda.empty_cache()

    # NVFP4 weights of a 128-expert MoE layer
    E, F = 128, 768
    experts = W.moe_layer(E, H, F)
    for nm, rows_p, cols in (("gate_up", [F, F], H), ("down", [H], F)):
        if nm == "gate_up":
            host = [p for g, u, d in experts for p in (g, u)]
        else:
            host = [d for g, u, d in experts]
        P = len(rows_p)
        rows = sum(rows_p)
        ne = E * rows * cols
        wb = ne * 2 + ne // 2 + ne // 16 + 4 * E
        sets = _sets_for(wb, l2)
        base = [dev16(h) for h in host]
        del host
        built = []
        for i in range(sets):
            parts = base if i == 0 else [t.clone() for t in base]
            built.append(ops.weights(parts, E, P, rows_p, cols))
        line(f"nvfp4_weight_{nm}_{E}x{rows}x{cols}", [c for c, _ in built],
             wb, ne)
        line(f"dequantize_nvfp4_{nm}_{E}x{rows}x{cols}",
             [ops.dq_nvfp4(c, bs, S, q.S_PER_BATCH, E, rows, cols)
              for _, (c, bs, S) in built], wb, ne)
        del built, base
        torch.cuda.empty_cache()
    del experts

    # FP8 with FP32 block scales: 1x128 tiles of X [8192 x 4096], 128x128
    # blocks of the linear weight [8192 x 2048], the dequantizations and the
    # backward-orientation conversion of the tiles
    for nm, bits, br in (("1x128_8192x4096", W.mxfp8_random(8192, 4096), 1),
                         ("128x128_8192x2048", W.linear_weight(), 128)):
        x = dev16(bits)
        rows, cols = x.shape
        n = x.numel()
        b = 3 * n + 4 * (n // (128 * br))
        sets = _sets_for(b, l2)
        built = [ops.fp8blk(x if i == 0 else x.clone(), br) for i in range(sets)]
        line(f"fp8_block_{nm}", [c for c, _ in built], b, n)
        line(f"fp8_block_dequantize_{nm}",
             [ops.fp8blk_dq(c, sc, rows, cols, br) for _, (c, sc) in built],
             b, n)
        if br == 1:
            line("fp8_block_requantize_transpose_8192x4096",
                 [ops.fp8blk_rt(c, sc, rows, cols) for _, (c, sc) in built],
                 2 * n + 8 * (n // 128), n)
        del built, x
        torch.cuda.empty_cache()
    out["timing"] = ("median over 9 rounds of the per-launch mean of >= 24 "
                     "back-to-back launches cycling over `rotating_sets` "
                     "buffer sets (>= 4 x L2 of data per cycle): inputs come "
                     "from HBM and each launch absorbs the write-back of the "
                     "previous launch's dirty lines; p10/p90 over the rounds; "
                     "GB/s = algorithmic bytes / time")
    return out


def _time_fn(fn, stream, reps):
    import torch
    with torch.cuda.stream(stream):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def load_traffic(kernel_name):
    """DRAM bytes (read + write) per launch of the dominant kernel from the
    committed ncu summary (profiles/traffic.json), or None when no capture
    was taken for the kernel as it is now (its source hash differs)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)[kernel_name]
        for src, digest in d["sources_sha256"].items():
            with open(os.path.join(ROOT, src), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != digest:
                    return None
        return int(d["dram_bytes_per_launch"])
    except Exception:
        return None


def run_e2e(q, dev, x_bits, args):
    """The step through the C ABI with host buffers: every step copies X from
    pinned host memory to the device, runs the seven operations on it and
    reads every code, scale and FP32 scale back into pinned host memory
    (one copy each way: a step's outputs sit in one device buffer).  Steps
    rotate over three streams, each with its own device buffers, workspace
    and host result buffer, so one step's copies overlap the neighbouring
    steps' kernels and opposite-direction copies, as a pipelined producer
    would run them."""
    import torch
    L = q.lib()
    lay = q.SCALE_SWIZZLED
    NS = 3
    x_pin = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    n_e2e = max(6, min(30, args.steps // 50))
    streams = [torch.cuda.Stream(dev) for _ in range(NS)]
    # the outputs read back, in one device buffer (256-byte aligned views)
    sizes = [("rc", M * K), ("rs", q.scale_bytes(M, K // 32)), ("cc", K * M),
             ("cs", q.scale_bytes(K, M // 32)), ("tc", M * K // 2),
             ("ts", q.scale_bytes(M, K // 16)), ("tS", 4 * M),
             ("wc", PAIRS * 2 * PART_ROWS * WK // 2),
             ("ws", PAIRS * q.scale_bytes(2 * PART_ROWS, WK // 16)),
             ("wS", 4 * PAIRS)]
    offs, o = {}, 0
    for nm, n in sizes:
        offs[nm] = o
        o += (n + 255) // 256 * 256
    total_out = o
    d2h = sum(n for _, n in sizes)
    ws_bytes = int(L.nvfp4_quantize_weight_shared_workspace_size(PAIRS))
    rows_tab = (ctypes.c_int64 * 2)(PART_ROWS, PART_ROWS)
    sets = []
    for i in range(NS):
        x = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
        ob = torch.empty(total_out, dtype=torch.uint8, device=dev)
        hb = torch.empty(total_out, dtype=torch.uint8).pin_memory()
        y = [torch.empty(M * K, dtype=torch.bfloat16, device=dev) for _ in range(4)]
        wsp = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
        flat = x.view(2 * PAIRS, PART_ROWS, WK)
        tab = (ctypes.c_void_p * (2 * PAIRS))(
            *[flat[k].data_ptr() for k in range(2 * PAIRS)])
        a = {nm: ob.data_ptr() + offs[nm] for nm, _ in sizes}
        st = ctypes.c_void_p(streams[i].cuda_stream)
        calls = [
            (L.mxfp8_quantize_rowcol, (x.data_ptr(), M, K, K, a["rc"], a["rs"],
                                       a["cc"], a["cs"], lay, st)),
            (L.dequantize_mxfp8, (a["rc"], a["rs"], M, K, lay, y[0].data_ptr(), st)),
            (L.dequantize_mxfp8, (a["cc"], a["cs"], K, M, lay, y[1].data_ptr(), st)),
            (L.nvfp4_quantize_per_token, (x.data_ptr(), M, K, K, a["tc"], a["ts"],
                                          a["tS"], lay, st)),
            (L.dequantize_nvfp4, (a["tc"], a["ts"], a["tS"], q.S_PER_ROW, 1, M, K,
                                  lay, y[2].data_ptr(), st)),
            (L.nvfp4_quantize_weight_shared,
             (PAIRS, 2, ctypes.cast(tab, ctypes.c_void_p),
              ctypes.cast(rows_tab, ctypes.c_void_p), WK, a["wc"], a["ws"],
              a["wS"], None, lay, wsp.data_ptr(), wsp.numel(), st)),
            (L.dequantize_nvfp4, (a["wc"], a["ws"], a["wS"], q.S_PER_BATCH, PAIRS,
                                  2 * PART_ROWS, WK, lay, y[3].data_ptr(), st)),
        ]
        sets.append((x, ob, hb, y, wsp, tab, calls))

    def step(i):
        x, ob, hb, _, _, _, calls = sets[i % NS]
        with torch.cuda.stream(streams[i % NS]):
            x.copy_(x_pin, non_blocking=True)
            for fn, a in calls:
                st = fn(*a)
                if st != 0:
                    raise RuntimeError(f"e2e: {q.status_string(st)}")
            hb.copy_(ob, non_blocking=True)

    for i in range(2 * NS):
        step(i)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(n_e2e):
        step(i)
    torch.cuda.synchronize(dev)
    dt = (time.perf_counter() - t0) / n_e2e
    st = q.get_last_error()
    if st != 0:
        raise RuntimeError(f"e2e: {q.status_string(st)}")
    step_bytes = sum(op_bytes().values())
    return {"value": round(step_bytes / dt / 1e9, 1), "unit": UNIT,
            "h2d_bytes_per_step": int(x_bits.nbytes),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(dt * 1e3, 3),
            "steps": n_e2e, "streams": NS,
            "api": "C ABI (libmxq) with preallocated device buffers; one "
                   "H2D copy of X and one D2H copy of all codes and scales "
                   "per step"}


# --------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline).
# --------------------------------------------------------------------------
def oracle_sample_step(x_rows):
    """The step's operations run by the CPU oracle on a row slice of X."""
    import oracle as O
    rc, rs = O.mxfp8_quantize_rowwise(x_rows)
    cc, cs = O.mxfp8_quantize_colwise(x_rows)
    O.mxfp8_dequantize(rc, rs)
    O.mxfp8_dequantize(cc, cs)
    tc, ts, tS = O.nvfp4_quantize_per_token(x_rows)
    O.nvfp4_dequantize(tc, ts, tS)
    half = x_rows.shape[0] // 2
    wc, wsc, wS = O.nvfp4_quantize_group([x_rows[:half], x_rows[half:]])
    O.nvfp4_dequantize(wc, wsc, np.array([wS]))


def oracle_timed(rows_total, threads):
    """Time the oracle on `rows_total` rows of X split over `threads` threads
    (32-row slices; ctypes releases the GIL inside the C oracle)."""
    import oracle as O
    import workloads as W
    O.lib()
    x = W.mxfp8_random(rows_total, K, seed=11)
    slices = [x[i:i + 32] for i in range(0, rows_total, 32)]
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(oracle_sample_step, slices))
    dt = time.perf_counter() - t0
    frac = rows_total / M
    return sum(op_bytes().values()) * frac / dt / 1e9, dt


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


def cpu_baseline(args, min_s=10.0, max_passes=40, single_min_s=5.0):
    """The oracle over `cpu_rows` rows of X, repeated until at least min_s
    seconds of CPU work have run (at most max_passes passes), on all host
    cores; then on one thread, over 32-row slices until single_min_s
    seconds have run."""
    import oracle as O
    import workloads as W
    O.lib()
    cores = os.cpu_count() or 1
    rows = args.cpu_rows
    x = W.mxfp8_random(rows, K, seed=11)
    slices = [x[i:i + 32] for i in range(0, rows, 32)]
    passes, total = 0, 0.0
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        while passes < max_passes and (passes == 0 or total < min_s):
            t0 = time.perf_counter()
            list(ex.map(oracle_sample_step, slices))
            total += time.perf_counter() - t0
            passes += 1
    v = sum(op_bytes().values()) * (rows / M) * passes / total / 1e9
    # one thread: whole 32-row slices, as many as fit in single_min_s
    n1, t1 = 0, 0.0
    while n1 == 0 or (t1 < single_min_s and n1 < len(slices)):
        t0 = time.perf_counter()
        oracle_sample_step(slices[n1 % len(slices)])
        t1 += time.perf_counter() - t0
        n1 += 1
    v1 = sum(op_bytes().values()) * (32 * n1 / M) / t1 / 1e9
    return {"value": round(v, 4), "unit": UNIT, "cores": cores,
            "kind": "oracle", "cpu_model": cpu_model(),
            "sample": (f"{passes} passes of the step's 7 operations over "
                       f"{rows} of the 8192 rows of X ({rows * K} elements "
                       f"per pass), 32-row slices over {cores} threads, "
                       f"{total:.1f} s"),
            "single_thread": {
                "value": round(v1, 5), "unit": UNIT, "cores": 1,
                "sample": (f"{n1} slices of 32 rows of X through the step's "
                           f"7 operations on one thread, {t1:.1f} s")}}


def step_config(world, serial=False):
    """The workload's `config`, the same for both arms of the bench."""
    return {
        "workload": WORKLOAD,
        "M": M, "K": K, "scale_layout": "swizzled",
        "weight_pairs": f"{PAIRS} x 2 x [{PART_ROWS} x {WK}]",
        "l2": ("inputs larger than L2: 3 rotating input copies and 2 "
               "rotating output sets, every kernel reads data last "
               "touched >= one step (~680 MB) earlier"),
        "parallelism": f"weak: one independent replica per GPU x{world}",
        "streams": ("1 (serial)" if serial else
                    "3: the rowcol kernel alone, then the MXFP8 "
                    "dequantizations, the per-token chain and the weight "
                    "chain (higher stream priority) concurrently"),
    }


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    # Size each step so that the whole run stays near a minute of wall time.
    per_row = []
    for _ in range(args.warmup):
        v, dt = oracle_timed(32 * max(1, cores), cores)
        per_row.append(dt / (32 * max(1, cores)))
    rows = args.ref_rows
    if rows <= 0:
        budget_s = 60.0
        rows = int(budget_s / max(args.steps, 1) / max(min(per_row), 1e-9))
        rows = max(32, min(M, rows // 32 * 32))
    vals, dts = [], []
    for _ in range(args.steps):
        v, dt = oracle_timed(rows, cores)
        vals.append(v)
        dts.append(dt)
    value = statistics.mean(vals)
    out = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.mean(dts), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": step_config(world),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT,
                         "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model(),
                         "sample": (f"{rows} of the {M} rows of X through "
                                    "the step's 7 operations per step "
                                    "(32-row slices over all cores); value "
                                    "= the step's algorithmic bytes scaled "
                                    "to the sampled rows / time")},
        "e2e": {"value": round(value, 4), "unit": UNIT,
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


PROFILE_WORKLOADS = (
    "rowcol_8192x4096", "rowcol_8192x2048", "dequant_mxfp8_8192x4096",
    "per_token_ragged", "dequant_nvfp4_ragged", "rht_ragged",
    "rht_sr_ragged",
    "weight_gate_up_128", "weight_down_128", "weight_step_8pairs",
    "weight_gate_up_128_given_scale",
    "dequant_nvfp4_gate_up_128", "fp8_block_1x128", "fp8_block_128x128",
    "fp8_block_dequant_1x128", "fp8_block_requant_t", "gemm_mxfp8",
    "gemm_nvfp4_grouped",
    "moe_gate_up_swiglu", "moe_gate_up_swiglu_gather", "gemm_bf16_dq")


def run_profile(args):
    """One workload's kernel alone, launched `--launches` times after one
    warm-up launch, on one set of buffers (a few GB at most): the harness
    the ncu captures run, so that a capture holds no other workload."""
    import torch
    import nvfp4_quantizers_gb300 as q
    import workloads as W
    from nvfp4_quantizers_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    ops = _Ops(q, dev, stream)

    def dev16(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    name = args.profile
    H, E, F = 2048, 128, 768
    if name.startswith("rowcol"):
        x = dev16(W.mxfp8_random(8192, 4096) if name.endswith("4096")
                  else W.linear_weight())
        call, _ = ops.rowcol(x)
    elif name == "dequant_mxfp8_8192x4096":
        _, o = ops.rowcol(dev16(W.mxfp8_random(8192, 4096)))
        _()
        call = ops.dq_mxfp8(o[0].view(8192, 4096), o[1])
    elif name in ("per_token_ragged", "dequant_nvfp4_ragged", "rht_ragged",
                  "rht_sr_ragged"):
        x = dev16(W.ragged_tokens(W.ragged_lengths(), H))
        T = x.shape[0]
        flags = {"rht_ragged": q.NVFP4_RHT,
                 "rht_sr_ragged": q.NVFP4_RHT | q.NVFP4_SR}.get(name)
        call, o = ops.per_token(x, rht_flags=flags)
        if name == "dequant_nvfp4_ragged":
            call()
            call = ops.dq_nvfp4(o[0], o[1], o[2], q.S_PER_ROW, 1, T, H)
    elif name.startswith(("weight_", "dequant_nvfp4_gate_up")):
        if name == "weight_step_8pairs":
            xs = dev16(W.mxfp8_random(8192, 4096)).view(16, 1024, 2048)
            call, o = ops.weights([xs[i] for i in range(16)], 8, 2,
                                  [1024, 1024], 2048)
        else:
            experts = W.moe_layer(E, H, F)
            if "down" in name:
                parts, rows_p, K = [dev16(d) for g, u, d in experts], [H], F
            else:
                parts = [dev16(t) for g, u, d in experts for t in (g, u)]
                rows_p, K = [F, F], H
            del experts
            call, o = ops.weights(parts, E, len(rows_p), rows_p, K)
            if name.endswith("given_scale"):
                call()
                call, o = ops.weights(parts, E, len(rows_p), rows_p, K,
                                      S_in=o[2])
            if name.startswith("dequant"):
                call()
                call = ops.dq_nvfp4(o[0], o[1], o[2], q.S_PER_BATCH, E,
                                    sum(rows_p), K)
    elif name.startswith("fp8_block"):
        br = 128 if name == "fp8_block_128x128" else 1
        x = dev16(W.linear_weight() if br == 128 else
                  W.mxfp8_random(8192, 4096))
        call, o = ops.fp8blk(x, br)
        if name == "fp8_block_requant_t":
            call()
            call = ops.fp8blk_rt(o[0], o[1], 8192, 4096)
        elif name == "fp8_block_dequant_1x128":
            call()
            call = ops.fp8blk_dq(o[0], o[1], 8192, 4096, 1)
    elif name.startswith(("gemm", "moe")):
        gemm_calls = _gemm_workloads(q, W, dev)
        call = gemm_calls[name]
    else:
        raise SystemExit(f"unknown workload {name}; one of {PROFILE_WORKLOADS}")
    with torch.cuda.stream(stream):
        call()
        torch.cuda.synchronize()
        for _ in range(args.launches):
            call()
    torch.cuda.synchronize()
    st = q.get_last_error()
    print(json.dumps({"profile": name, "launches": args.launches,
                      "status": q.status_string(st)}))
    if st != 0:
        raise SystemExit(1)


def _gemm_workloads(q, W, dev):
    """Launchers of the GEMM consumers on their benchmark workloads (the
    Python API allocates C per call)."""
    import torch

    def dev16(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
    out = {}
    A, B = W.gemm_mxfp8_inputs(2048, 2048, 8192)
    qa = q.mxfp8_quantize_rowcol(dev16(A), rowwise=True, colwise=False)
    qb = q.mxfp8_quantize_rowcol(dev16(B), rowwise=False, colwise=True)
    out["gemm_mxfp8"] = lambda: q.gemm_mxfp8(qa.row_codes, qa.row_scales,
                                             qb.col_codes_t, qb.col_scales_t)
    E, H, F = 128, 2048, 768
    tokens = W.gemm_tokens(4096, H)
    route = W.topk_routing(4096, E, 8)
    idx, offs, _ = W.expert_gather_index(route, E)
    tg = q.nvfp4_quantize_per_token_gather(dev16(tokens),
                                           torch.from_numpy(idx).to(dev))
    wts = dev16(np.stack([np.concatenate(W.moe_expert(e, hidden=H, ffn=F)[:2])
                          for e in range(E)]))
    tw = q.nvfp4_quantize_weight_shared([[wts[e]] for e in range(E)])
    del wts
    out["gemm_nvfp4_grouped"] = lambda: q.gemm_nvfp4_grouped(
        tg.codes, tg.block_scales, tg.scales, offs, tw.codes, tw.block_scales,
        tw.scales)
    out["moe_gate_up_swiglu"] = lambda: q.moe_gate_up_swiglu(
        tg.codes, tg.block_scales, tg.scales, offs, tw.codes, tw.block_scales,
        tw.scales)
    xq = q.nvfp4_quantize_per_token(dev16(tokens), "linear")
    idx_dev = torch.from_numpy(idx).to(dev)
    out["moe_gate_up_swiglu_gather"] = lambda: q.moe_gate_up_swiglu_gather(
        xq, idx_dev, offs, tw.codes, tw.block_scales, tw.scales)
    dY = dev16(W.gemm_tokens(2048, 8192))
    wq = q.mxfp8_quantize_rowcol(dev16(W.linear_weight()), rowwise=False,
                                 colwise=True)
    out["gemm_bf16_dq"] = lambda: q.gemm_bf16_mxfp8(dY, wq.col_codes_t,
                                                    wq.col_scales_t)
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="libmxq", choices=["libmxq", "reference"])
    ap.add_argument("--cpu-rows", type=int, default=8192)
    ap.add_argument("--ref-rows", type=int, default=0,
                    help="rows of X per reference step (0: sized to ~1 min)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-shapes", action="store_true",
                    help="skip the per-kernel lines at every workload's size")
    ap.add_argument("--serial", action="store_true",
                    help="run the step's three chains on one stream")
    ap.add_argument("--profile", default=None, choices=PROFILE_WORKLOADS,
                    help="launch only this workload's kernel (for ncu)")
    ap.add_argument("--launches", type=int, default=3,
                    help="launches after one warm-up launch, with --profile")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile:
        run_profile(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
