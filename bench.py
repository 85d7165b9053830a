"""Benchmark of the MXFP8 / NVFP4 quantizer path on GB300.

One step = one pass of every operation of the path over one batch of the
activation workload X [8192 x 4096] bf16 (N(0,1) with 0.1% of entries x100):

  1. mxfp8_quantize_rowcol   rowwise 1x32 + columnwise 32x1 copies, one pass,
                             E8M0 scales in the swizzled tensor-core layout
  2. dequantize_mxfp8        of the rowwise copy and of the columnwise copy
  3. nvfp4_quantize_per_token X as 8192 tokens x 4096 hidden (FP32 scale per
                             token, E4M3 per 16, packed E2M1)
  4. dequantize_nvfp4        of (3), per-token scales
  5. nvfp4_quantize_weight_shared  X as 4 gate/up pairs of [1024 x 4096]
                             parts, each pair under one FP32 scale
  6. dequantize_nvfp4        of (5), per-group scales

value = algorithmic bytes of the step (bf16 read + codes / scales written,
or codes / scales read + bf16 written) / device time, in GB/s.  Inputs are
resident in HBM; every kernel reads data last touched at least one full
step (~680 MB of traffic) earlier (three rotating input copies, two
rotating output sets), so nothing is served from the 126 MB L2.

--impl reference times the CPU oracle on a bounded sample of the same
workload (the oracle is the reference implementation of this path).
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
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
PAIRS = 4                       # X viewed as 4 gate/up pairs
PART_ROWS = M // (2 * PAIRS)    # 1024 rows per part
WORKLOAD = ("MXFP8 rowwise+columnwise quantize (one pass) + both MXFP8 "
            "dequantizes + NVFP4 per-token quantize/dequantize + NVFP4 "
            "shared-scale weight quantize/dequantize of an activation "
            "[8192 x 4096] bf16, N(0,1) with 0.1% entries x100")


# --------------------------------------------------------------------------
# Algorithmic bytes per operation.
# --------------------------------------------------------------------------
def op_bytes():
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
            "wc": torch.empty((PAIRS, 2 * PART_ROWS, K // 2), dtype=torch.uint8, device=dev),
            "ws": torch.empty((PAIRS, q.scale_bytes(2 * PART_ROWS, K // 16)), dtype=torch.uint8, device=dev),
            "wS": torch.empty(PAIRS, dtype=torch.float32, device=dev),
        }

    outs = [new_outputs(), new_outputs()]
    y_row = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    y_col = torch.empty((K, M), dtype=torch.bfloat16, device=dev)
    y_tok = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    y_w = torch.empty((PAIRS, 2 * PART_ROWS, K), dtype=torch.bfloat16, device=dev)
    L = q.lib()
    ws_bytes = int(L.nvfp4_quantize_weight_shared_workspace_size(PAIRS))
    wsp = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    import ctypes
    parts_tabs = []
    for xi in X:
        flat = xi.view(2 * PAIRS, PART_ROWS, K)
        parts_tabs.append((ctypes.c_void_p * (2 * PAIRS))(
            *[flat[i].data_ptr() for i in range(2 * PAIRS)]))
    rows_tab = (ctypes.c_int64 * 2)(PART_ROWS, PART_ROWS)
    s = ctypes.c_void_p(stream.cuda_stream)
    # The step's three chains (MXFP8 quantize -> both dequantizations;
    # per-token quantize -> dequantize; weights -> dequantize) touch
    # different buffers: after the rowcol kernel (timed alone for the
    # roofline line), the other two chains fork onto their own streams and
    # join before the next step.
    side = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    s_side = [ctypes.c_void_p(x.cuda_stream) for x in side]
    ev_fork = torch.cuda.Event()
    ev_join = [torch.cuda.Event(), torch.cuda.Event()]

    def chk(st, what):
        if st != 0:
            raise RuntimeError(f"{what}: {q.status_string(st)}")

    names = list(op_bytes().keys())
    ev = None

    def step(i, record=None, only=None, concurrent=False):
        o_new, o_old = outs[i % 2], outs[(i + 1) % 2]
        s1, s2 = (s_side[0], s_side[1]) if concurrent else (s, s)
        x0, x1, x2 = X[i % 3], X[(i + 1) % 3], X[(i + 2) % 3]
        tab = parts_tabs[(i + 2) % 3]

        def mark(j):
            if record is None:
                return
            if only is None:
                record[j].record(stream)
            elif j in only:
                record[only.index(j)].record(stream)
        mark(0)
        chk(L.mxfp8_quantize_rowcol(x0.data_ptr(), M, K, K, o_new["rc"].data_ptr(),
                                    o_new["rs"].data_ptr(), o_new["cc"].data_ptr(),
                                    o_new["cs"].data_ptr(), lay, s), "rowcol")
        mark(1)
        if concurrent:
            ev_fork.record(stream)
            side[0].wait_event(ev_fork)
            side[1].wait_event(ev_fork)
        chk(L.dequantize_mxfp8(o_old["rc"].data_ptr(), o_old["rs"].data_ptr(), M, K,
                               lay, y_row.data_ptr(), s), "dq row")
        mark(2)
        chk(L.dequantize_mxfp8(o_old["cc"].data_ptr(), o_old["cs"].data_ptr(), K, M,
                               lay, y_col.data_ptr(), s), "dq col")
        mark(3)
        def token_q():
            chk(L.nvfp4_quantize_per_token(
                x1.data_ptr(), M, K, K, o_new["tc"].data_ptr(),
                o_new["ts"].data_ptr(), o_new["tS"].data_ptr(), lay, s1),
                "per-token")

        def token_dq():
            chk(L.dequantize_nvfp4(o_old["tc"].data_ptr(), o_old["ts"].data_ptr(),
                                   o_old["tS"].data_ptr(), q.S_PER_ROW, 1, M, K,
                                   lay, y_tok.data_ptr(), s1), "dq tokens")

        def weights_q():
            chk(L.nvfp4_quantize_weight_shared(
                PAIRS, 2, ctypes.cast(tab, ctypes.c_void_p),
                ctypes.cast(rows_tab, ctypes.c_void_p), K,
                o_new["wc"].data_ptr(), o_new["ws"].data_ptr(),
                o_new["wS"].data_ptr(), None, lay, wsp.data_ptr(), wsp.numel(),
                s2), "weights")

        def weights_dq():
            chk(L.dequantize_nvfp4(o_old["wc"].data_ptr(), o_old["ws"].data_ptr(),
                                   o_old["wS"].data_ptr(), q.S_PER_BATCH, PAIRS,
                                   2 * PART_ROWS, K, lay, y_w.data_ptr(), s2),
                "dq weights")
        if concurrent:
            # Each side chain dequantizes the previous step's codes first and
            # quantizes this step's input last, so the step ends on the
            # kernels that leave the least dirty data in L2 for the next
            # step's rowcol kernel.
            token_dq()
            token_q()
            weights_dq()
            weights_q()
        else:
            token_q()
            mark(4)
            token_dq()
            mark(5)
            weights_q()
            mark(6)
            weights_dq()
        if concurrent:
            ev_join[0].record(side[0])
            ev_join[1].record(side[1])
            stream.wait_event(ev_join[0])
            stream.wait_event(ev_join[1])
        mark(7)

    # Our kernels per step: rowcol 1, dequant 2 + 1 + 1, per-token 1,
    # weights 1 (one cooperative kernel per call of up to 256 groups).
    launches_per_step = 1 + 2 + 1 + 1 + 1 + 1

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i, concurrent=not args.serial)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()

    # Timed region: K steps.  Only the dominant quantizer kernel
    # (mxfp8_quantize_rowcol) is bracketed by events inside a step, so the
    # other kernels keep their programmatic-dependent-launch overlap.
    recs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
            for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            start.record(stream)
            for i in range(args.steps):
                step(args.warmup + i, recs[i], only=(0, 1),
                     concurrent=not args.serial)
            end.record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        wall = time.perf_counter() - t0
    ms = start.elapsed_time(end)
    ms_max = max_over_ranks(ms, dist if world > 1 else None, dev)
    ob = op_bytes()
    step_bytes = sum(ob.values())
    dom = "mxfp8_quantize_rowcol"
    dom_ms = statistics.mean(recs[i][0].elapsed_time(recs[i][1])
                             for i in range(args.steps))
    # Per-kernel breakdown: a separate pass with events between all kernels
    # (events between kernels cost the launch overlap, so this pass is not
    # used for the headline number).
    nb = min(args.steps, 200)
    recs8 = [[torch.cuda.Event(enable_timing=True) for _ in range(8)]
             for _ in range(nb)]
    with torch.cuda.stream(stream):
        for i in range(nb):
            step(args.warmup + args.steps + i, recs8[i])
    torch.cuda.synchronize(dev)
    per_kernel_ms = {}
    for j, nm in enumerate(names):
        per_kernel_ms[nm] = statistics.mean(
            recs8[i][j].elapsed_time(recs8[i][j + 1]) for i in range(nb))
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
        "config": {
            "workload": WORKLOAD,
            "M": M, "K": K, "scale_layout": "swizzled",
            "weight_pairs": f"{PAIRS} x 2 x [{PART_ROWS} x {K}]",
            "l2": ("inputs larger than L2: 3 rotating input copies and 2 "
                   "rotating output sets, every kernel reads data last "
                   "touched >= one step (~680 MB) earlier"),
            "parallelism": f"weak: one independent replica per GPU x{world}",
            "streams": ("1 (serial)" if args.serial else
                        "3: rowcol alone, then its dequantizations, the "
                        "per-token chain and the weight chain concurrently"),
        },
        "pct_hbm_peak": round(100 * value / world / peak, 1),
        "roofline": {
            "kernel": dom,
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

    def t_gq():
        return q.nvfp4_quantize_per_token_gather(tok_dev, idx_dev)
    ms_gq = _time_fn(t_gq, stream, reps)
    tg = t_gq()

    def t_sw():
        return q.moe_gate_up_swiglu(tg.codes, tg.block_scales, tg.scales,
                                    offs2, tw.codes, tw.block_scales,
                                    tw.scales)
    ms_sw = _time_fn(t_sw, stream, reps)
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
           "forward_us": round((ms_gq + ms_sw) * 1e3, 2),
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


def _time_reps(fn, stream, reps, flush_w, flush_r, warmup=3):
    """Per-launch device times (ms) of `fn` on `stream`: the L2 is flushed
    before every rep (a write of one buffer larger than L2, then a read of
    another, so the timed launch starts with clean lines that hold none of
    its data), outside the events that bracket the launch."""
    import torch
    evs = []
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn()
        for _ in range(reps):
            flush_w.fill_(1)
            flush_r.sum()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            evs.append((e0, e1))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def _shape_line(ms_list, nbytes, elems, peak):
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
            "frac": round(gbs / peak, 3), "bytes": int(nbytes)}


def run_shapes(q, W, dev, stream, reps=20):
    """Each quantizer and dequantizer alone at the full sizes of the
    workloads it is specified on, L2 flushed before every launch: MXFP8
    rowwise + columnwise of the four 8192 x 4096 input classes and of the
    linear layer's input [2048 x 2048] and weight [8192 x 2048]; NVFP4
    per-token on the ragged batch of 64 sequences (lengths in [128, 4096],
    hidden 2048), also with the pretraining recipe's Hadamard transform and
    stochastic rounding; NVFP4 shared-scale weights of a 128-expert MoE layer
    (gate/up pairs [2 x 768 x 2048] and down [2048 x 768]); FP8 with FP32
    block scales (1x128 tiles of the activation, 128x128 blocks of the
    linear weight, the tiles' backward-orientation conversion); and the
    dequantizations of each."""
    import torch
    peak = measured_peak()[0]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(2 * l2 // 4, dtype=torch.float32, device=dev)
    out = {}

    def dev16(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    def mx(name, bits):
        x = dev16(bits)
        m, k = x.shape
        n = m * k
        r = q.mxfp8_quantize_rowcol(x)
        out[f"mxfp8_rowcol_{name}"] = _shape_line(
            _time_reps(lambda: q.mxfp8_quantize_rowcol(x), stream, reps,
                       flush_w, flush_r),
            2 * n + 2 * (n + n // 32), n, peak)
        return r

    r = None
    for cls, gen in (("random", W.mxfp8_random), ("boundary", W.mxfp8_boundary),
                     ("zeros", W.mxfp8_zeros), ("maxes", W.mxfp8_maxes)):
        r = mx(f"8192x4096_{cls}", gen(8192, 4096))
    n = 8192 * 4096
    for nm, cod, sc in (("row", r.row_codes, r.row_scales),
                        ("col", r.col_codes_t, r.col_scales_t)):
        out[f"dequantize_mxfp8_{nm}_8192x4096"] = _shape_line(
            _time_reps(lambda: q.dequantize_mxfp8(cod, sc), stream, reps,
                       flush_w, flush_r),
            n + n // 32 + 2 * n, n, peak)
    del r
    mx("2048x2048_linear_input", W.linear_input())
    mx("8192x2048_linear_weight", W.linear_weight())

    # NVFP4 per-token, ragged batch flattened
    H = 2048
    lengths = W.ragged_lengths()
    x = dev16(W.ragged_tokens(lengths, H))
    T = x.shape[0]
    tq = q.nvfp4_quantize_per_token(x)
    tb = T * (2 * H + H // 2 + H // 16 + 4)
    out[f"nvfp4_per_token_ragged_{T}x{H}"] = dict(_shape_line(
        _time_reps(lambda: q.nvfp4_quantize_per_token(x), stream, reps,
                   flush_w, flush_r), tb, T * H, peak),
        sequences=int(len(lengths)))
    out[f"dequantize_nvfp4_ragged_{T}x{H}"] = _shape_line(
        _time_reps(lambda: q.dequantize_nvfp4(tq.codes, tq.block_scales,
                                              tq.scales),
                   stream, reps, flush_w, flush_r), tb, T * H, peak)
    # the pretraining recipe's stabilizers on the same batch
    for nm, fl in (("rht", q.NVFP4_RHT), ("rht_sr", q.NVFP4_RHT | q.NVFP4_SR)):
        out[f"nvfp4_per_token_{nm}_ragged_{T}x{H}"] = _shape_line(
            _time_reps(lambda: q.nvfp4_quantize_per_token_rht_sr(x, 2026, fl),
                       stream, reps, flush_w, flush_r), tb, T * H, peak)
    del x, tq

    # NVFP4 weights of a 128-expert MoE layer
    E, F = 128, 768
    experts = W.moe_layer(E, H, F)
    gate_up = [[dev16(g), dev16(u)] for g, u, d in experts]
    down = [[dev16(d)] for g, u, d in experts]
    del experts
    for nm, groups, rows, cols in (("gate_up", gate_up, 2 * F, H),
                                   ("down", down, H, F)):
        ws = torch.empty(max(int(q.lib().nvfp4_quantize_weight_shared_workspace_size(E)), 256),
                         dtype=torch.uint8, device=dev)
        wq = q.nvfp4_quantize_weight_shared(groups, workspace=ws)
        ne = E * rows * cols
        wb = ne * 2 + ne // 2 + ne // 16 + 4 * E
        out[f"nvfp4_weight_{nm}_{E}x{rows}x{cols}"] = _shape_line(
            _time_reps(lambda: q.nvfp4_quantize_weight_shared(groups,
                                                              workspace=ws),
                       stream, reps, flush_w, flush_r), wb, ne, peak)
        out[f"dequantize_nvfp4_{nm}_{E}x{rows}x{cols}"] = _shape_line(
            _time_reps(lambda: q.dequantize_nvfp4(wq.codes, wq.block_scales,
                                                  wq.scales),
                       stream, reps, flush_w, flush_r), wb, ne, peak)
        del wq
    del gate_up, down

    # FP8 with FP32 block scales: 1x128 tiles of X [8192 x 4096], 128x128
    # blocks of the linear weight [8192 x 2048], the dequantizations and the
    # backward-orientation conversion of the tiles
    x = dev16(W.mxfp8_random(8192, 4096))
    n = x.numel()
    fq = q.fp8_block_quantize(x, 1)
    out["fp8_block_1x128_8192x4096"] = _shape_line(
        _time_reps(lambda: q.fp8_block_quantize(x, 1), stream, reps,
                   flush_w, flush_r), 3 * n + 4 * (n // 128), n, peak)
    out["fp8_block_dequantize_1x128_8192x4096"] = _shape_line(
        _time_reps(lambda: q.fp8_block_dequantize(fq.codes, fq.scales, 1),
                   stream, reps, flush_w, flush_r), 3 * n + 4 * (n // 128), n,
        peak)
    out["fp8_block_requantize_transpose_8192x4096"] = _shape_line(
        _time_reps(lambda: q.fp8_block_requantize_transpose(fq.codes,
                                                            fq.scales),
                   stream, reps, flush_w, flush_r), 2 * n + 8 * (n // 128), n,
        peak)
    del x, fq
    w = dev16(W.linear_weight())
    n = w.numel()
    wq = q.fp8_block_quantize(w, 128)
    out["fp8_block_128x128_8192x2048"] = _shape_line(
        _time_reps(lambda: q.fp8_block_quantize(w, 128), stream, reps,
                   flush_w, flush_r), 3 * n + 4 * (n // 16384), n, peak)
    out["fp8_block_dequantize_128x128_8192x2048"] = _shape_line(
        _time_reps(lambda: q.fp8_block_dequantize(wq.codes, wq.scales, 128),
                   stream, reps, flush_w, flush_r), 3 * n + 4 * (n // 16384),
        n, peak)
    del w, wq, flush_w, flush_r
    torch.cuda.empty_cache()
    out["timing"] = (f"median of {reps} launches (p10/p90 beside it), each "
                     "after an L2 flush; GB/s = algorithmic bytes / time")
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
    """The step through the public API with host buffers: every step copies
    X from pinned host memory to the device, runs the seven operations and
    reads every code, scale and FP32 scale back into pinned host memory.
    Steps alternate between two streams (and two sets of host result
    buffers), so one step's copies overlap the neighbouring steps' kernels
    and opposite-direction copies, as a pipelined producer would run them."""
    import torch
    x_pin = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    n_e2e = max(4, min(20, args.steps // 50))
    streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]

    def once():
        x = x_pin.to(dev, non_blocking=True)
        r = q.mxfp8_quantize_rowcol(x)
        q.dequantize_mxfp8(r.row_codes, r.row_scales)
        q.dequantize_mxfp8(r.col_codes_t, r.col_scales_t)
        t = q.nvfp4_quantize_per_token(x)
        q.dequantize_nvfp4(t.codes, t.block_scales, t.scales)
        parts = x.view(2 * PAIRS, PART_ROWS, K)
        w = q.nvfp4_quantize_weight_shared(
            [[parts[2 * g], parts[2 * g + 1]] for g in range(PAIRS)])
        q.dequantize_nvfp4(w.codes, w.block_scales, w.scales)
        return [r.row_codes, r.row_scales, r.col_codes_t, r.col_scales_t,
                t.codes, t.block_scales, t.scales, w.codes, w.block_scales,
                w.scales]

    def step(i, hosts):
        s = streams[i % 2]
        with torch.cuda.stream(s):
            for h, a in zip(hosts[i % 2], once()):
                h.copy_(a, non_blocking=True)

    with torch.cuda.stream(streams[0]):
        res = once()
    torch.cuda.synchronize(dev)
    hosts = [[torch.empty(a.shape, dtype=a.dtype).pin_memory() for a in res]
             for _ in range(2)]
    for i in range(4):
        step(i, hosts)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(n_e2e):
        step(i, hosts)
    torch.cuda.synchronize(dev)
    dt = (time.perf_counter() - t0) / n_e2e
    step_bytes = sum(op_bytes().values())
    d2h = sum(a.numel() * a.element_size() for a in res)
    return {"value": round(step_bytes / dt / 1e9, 1), "unit": UNIT,
            "h2d_bytes_per_step": int(x_bits.nbytes),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(dt * 1e3, 3),
            "steps": n_e2e, "streams": 2}


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


def cpu_baseline(args, min_s=10.0, max_passes=40):
    """The oracle over `cpu_rows` rows of X, repeated until at least min_s
    seconds of CPU work have run (at most max_passes passes)."""
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
    return {"value": round(v, 4), "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": (f"{passes} passes of the step's 8 operations over "
                       f"{rows} of the 8192 rows of X ({rows * K} elements "
                       f"per pass), 32-row slices over {cores} threads, "
                       f"{total:.1f} s")}


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
        "config": {"workload": WORKLOAD, "M": M, "K": K,
                   "sample_rows": rows},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT,
                         "cores": cores, "kind": "oracle",
                         "sample": f"{rows} of 8192 rows per step"},
        "e2e": {"value": round(value, 4), "unit": UNIT,
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


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
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
