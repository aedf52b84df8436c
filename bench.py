#!/usr/bin/env python
"""Benchmark of the GPTQ per-layer path on GB300: ms per layer, weights quantized / s.

One step = the whole path on one layer: Hessian of the calibration activations
(gptq_hessian_accumulate), dead columns + damping + inverse-Hessian factor (gptq_prepare),
the blocked column sweep with lazy trailing updates and packing (gptq_quantize_layer).

Default workload: a 4096 x 4096 layer, 262144 fp16 calibration tokens (128 x 2048) with
8 outlier channels and 41 dead channels, bf16 weights, 4-bit per-row asymmetric grid,
B = 128, damping 1 % -- synthetic, seeded.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank quantizes its own copy of the layer (independent problems, no
collective on the data path): weak scaling, value = all ranks' weights / max time.
``--impl reference`` times the fp64 CPU oracle on the host cores instead, on a bounded
sample of the same workload scaled to the full layer.
"""

from __future__ import annotations

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

METRIC = "ms per layer & weights quantized/sec (4096×4096 int4 GPTQ), % roofline"
UNIT = "weights/s"


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="layer4096_n262144")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--n-tok", type=int, default=None, help="override token count (smaller runs)")
    p.add_argument("--recon", action="store_true",
                   help="time the consumer instead: per-row ||(W - W_hat) X^T||^2 from the "
                        "packed codes, on X (gptq_recon_error)")
    p.add_argument("--obq", action="store_true",
                   help="greedy-order OBQ against the fixed-order sweep on a 4096 x 128 layer "
                        "(OBQ keeps a per-row inverse Hessian on chip: d_in <= 128)")
    p.add_argument("--block", type=int, default=None,
                   help="lazy-batch width B (default: the workload's, 128); 1 = eager "
                        "column-at-a-time trailing updates")
    return p.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def reduce_max(value, device=None):
    """Max of a per-rank scalar over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(weights_per_rank, world, ms_step):
    """Weak scaling: every rank quantizes its own layer; all ranks' weights / max time."""
    return world * weights_per_rank / (ms_step / 1e3)


def profiled_traffic(n_tok):
    """DRAM bytes per Hessian launch from the committed ncu summary, or None when the
    kernel source changed since the capture or the token count differs."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", "hessian_tc_layer4096.md")
    src = os.path.join(ROOT, "post_weight_quantization_03_gb300", "csrc", "hessian.cu")
    try:
        text = open(prof).read()
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    fields = dict(line.split(": ", 1) for line in text.splitlines()
                  if line.startswith(("traffic_bytes_per_launch_262144:", "source_sha256_16:")))
    if fields.get("source_sha256_16:".rstrip(":"), "").strip() != digest or n_tok != 262144:
        return None
    return int(fields["traffic_bytes_per_launch_262144"])


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


# ---------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.th = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [t.strip() for t in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.th.join(timeout=2)
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        for r in self.rows:
            for name, v in zip(self.NAMES, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(self.rows)}


# ---------------------------------------------------------------------------------------
# CPU oracle timing (baseline / reference arm): bounded sample scaled to the full layer
# ---------------------------------------------------------------------------------------

def oracle_sample(X_host_f32_rows, W_host, layer, bits, block, damp, tok_sample, row_sample):
    """Times the oracle on a sample: Hessian over `tok_sample` tokens, the full prepare
    at this d_in, the sweep of `row_sample` rows.  Returns (est_seconds_full, detail)."""
    import numpy as np
    from oracle import gptq_oracle as O
    n_tok = layer.act.n_tok
    m = layer.d_out
    Xs = X_host_f32_rows[:tok_sample]
    t0 = time.perf_counter()
    H = O.hessian(Xs)
    t1 = time.perf_counter()
    Hd, dead, _ = O.damp_hessian(H, damp)
    U = O.inverse_cholesky_upper(Hd)
    t2 = time.perf_counter()
    Ws = W_host[:row_sample]
    scale, zero = O.row_grid(Ws, bits)
    codes, _ = O.gptq_quantize(Ws, U, scale, zero, bits, block=block, dead=dead)
    O.pack_codes(codes, bits)
    t3 = time.perf_counter()
    est = (t1 - t0) * n_tok / tok_sample + (t2 - t1) + (t3 - t2) * m / row_sample
    detail = {"hessian_s": t1 - t0, "prepare_s": t2 - t1, "sweep_s": t3 - t2,
              "tok_sample": tok_sample, "row_sample": row_sample}
    _ = np
    return est, detail


def host_cores():
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(k, "").isdigit():
            n = min(n, int(os.environ[k]))
    return n


# ---------------------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------------------

def main():
    args = parse_args()
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    import torch.distributed as dist

    from post_weight_quantization_03_gb300 import build_lib, gptq
    from post_weight_quantization_03_gb300 import synthetic as S

    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank if world > 1 else 0)
    build_lib.build()
    gptq.load()

    wl = S.WORKLOADS[args.workload]
    if args.obq:
        return run_obq(args, dev, rank, world)
    if len(wl.layers) > 1:
        return run_block(args, wl, dev, rank, world)
    layer = wl.layers[0]
    bits, block, damp = wl.bits[-1], args.block or wl.block, wl.damp
    act = layer.act
    if args.n_tok:
        from dataclasses import replace
        act = replace(act, n_tok=args.n_tok)
        layer = replace(layer, act=act)
    m, d, n = layer.d_out, act.d_in, act.n_tok

    # inputs resident in HBM (drawn on the device, seeded; untimed)
    A = S.mixing_matrix(d, act.seed, dev)
    X = S.activations(act, device=dev, A=A)
    del A
    W = S.layer_weights(layer, dev)
    torch.cuda.synchronize()

    # outputs and workspaces (allocated once, outside the timed region)
    H = torch.empty(d, d, dtype=torch.float32, device=dev)
    U = torch.empty(d, d, dtype=torch.float32, device=dev)
    dm = torch.empty(d, dtype=torch.uint8, device=dev)
    qp = torch.empty(m, gptq.packed_words(d, bits), dtype=torch.int32, device=dev)
    sc = torch.empty(m, dtype=torch.float32, device=dev)
    zr = torch.empty(m, dtype=torch.int32, device=dev)
    ws_p = gptq.workspace(gptq.gptq_prepare_workspace_bytes(d), dev)
    ws_q = gptq.workspace(gptq.gptq_quantize_workspace_bytes(m, d, bits, block), dev)
    stream = torch.cuda.current_stream(dev)

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    if args.recon:
        return run_recon(args, wl, layer, X, W, H, U, dm, qp, sc, zr, ws_p, ws_q, bits, block,
                         damp, stream, dev, rank, world)

    def step(record=None):
        e = [ev() for _ in range(4)] if record is not None else None
        if e: e[0].record(stream)
        gptq.hessian(X, H, accumulate=False, stream=stream)
        if e: e[1].record(stream)
        gptq.prepare(H, damp, U=U, dead_mask=dm, ws=ws_p, stream=stream)
        if e: e[2].record(stream)
        gptq.quantize(W, U, bits, block, dm, ws=ws_q, stream=stream, out=(qp, sc, zr, None))
        if e:
            e[3].record(stream)
            record.append(e)

    args.warmup = max(3, args.warmup)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- timed region (device-resident inputs) -----------------------------------------
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    time.sleep(0.4)  # let the sampler produce a first row
    launches0 = gptq.gptq_kernel_launches()
    stage_events = []
    t_start, t_end = ev(), ev()
    t_start.record(stream)
    for _ in range(args.steps):
        step(stage_events)
    t_end.record(stream)
    torch.cuda.synchronize()
    launches = gptq.gptq_kernel_launches() - launches0
    clk = clocks.stop()
    ms_total = t_start.elapsed_time(t_end)
    if world > 1:
        dist.barrier()
    ms_total = reduce_max(ms_total, dev)
    ms_step = ms_total / args.steps
    st_h = statistics.mean(e[0].elapsed_time(e[1]) for e in stage_events)
    st_p = statistics.mean(e[1].elapsed_time(e[2]) for e in stage_events)
    st_q = statistics.mean(e[2].elapsed_time(e[3]) for e in stage_events)
    weights = m * d
    value = whole_job_value(weights, world, ms_step)

    peaks, peak_src = measured_peaks()
    # trailing-update traffic of the sweep: each block reads and writes the fp32 working copy
    # of every later column once (the per-block rank-B update); other traffic not counted
    q_bytes = float(sum(m * (d - min(b0 + block, d)) * 8 for b0 in range(0, d, block)))
    h_flops = float(d) * (d + 1) * n
    h_tflops = h_flops / (st_h / 1e3) / 1e12
    peak_t = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    roofline = {"kernel": "hessian (gptq_hessian_accumulate)", "bound": "tensor",
                "achieved": round(h_tflops, 3), "peak": peak_t, "unit": "TFLOP/s",
                "frac": round(h_tflops / peak_t, 4), "traffic": profiled_traffic(n),
                "traffic_unit": "bytes per launch (dram read + write, ncu, scaled from a "
                                "65536-token capture; profiles/hessian_tc_layer4096.md)",
                "algorithmic": f"d(d+1)N = {h_flops:.4e} flop per launch (lower triangle of "
                               f"2 X^T X incl. diagonal)",
                "peak_source": f"{peak_src} bf16 sustained (fp16 tensor rate = bf16)"}
    if st_q > st_h:
        # the sweep dominates (small B): report it against HBM, from its trailing-update bytes
        q_gbs = q_bytes / (st_q / 1e3) / 1e9
        roofline = {"kernel": "quantize stage (gptq_quantize_layer: sweeps + trailing updates)",
                    "bound": "hbm", "achieved": round(q_gbs, 1), "peak": float(peaks["hbm_gbs"]),
                    "unit": "GB/s", "frac": round(q_gbs / float(peaks["hbm_gbs"]), 4),
                    "traffic": None,
                    "algorithmic": f"sum over blocks of d_out*(d_in - block end)*8 bytes = "
                                   f"{q_bytes:.4e} per layer (fp32 read + write of the later "
                                   f"columns per block)",
                    "peak_source": f"{peak_src} copy bandwidth"}

    # ---- end to end through the C ABI from host buffers --------------------------------
    e2e = None
    if not args.no_e2e:
        Xh = torch.empty(X.shape, dtype=X.dtype, pin_memory=True)
        Xh.copy_(X)
        Wh = torch.empty(W.shape, dtype=W.dtype, pin_memory=True)
        Wh.copy_(W)
        qh = torch.empty(qp.shape, dtype=qp.dtype, pin_memory=True)
        sh = torch.empty(sc.shape, dtype=sc.dtype, pin_memory=True)
        zh = torch.empty(zr.shape, dtype=zr.dtype, pin_memory=True)
        Wd = torch.empty_like(W)
        # X streams from host memory in chunks whose copies overlap the Gram products
        ws_h = gptq.workspace(gptq.gptq_hessian_host_workspace_bytes(
            gptq._dtype_code(X), X.shape[1], 0), dev)
        w_stream = torch.cuda.Stream(dev)
        w_ready = torch.cuda.Event()

        def e2e_step():
            w_stream.wait_stream(stream)        # the previous step is done with Wd
            with torch.cuda.stream(w_stream):
                Wd.copy_(Wh, non_blocking=True)
                w_ready.record(w_stream)
            gptq.hessian_host(Xh, H, accumulate=False, ws=ws_h, stream=stream)
            gptq.prepare(H, damp, U=U, dead_mask=dm, ws=ws_p, stream=stream)
            stream.wait_event(w_ready)
            gptq.quantize(Wd, U, bits, block, dm, ws=ws_q, stream=stream,
                          out=(qp, sc, zr, None))
            qh.copy_(qp, non_blocking=True)
            sh.copy_(sc, non_blocking=True)
            zh.copy_(zr, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        a, b = ev(), ev()
        a.record(stream)
        for _ in range(args.steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        ms_e2e = reduce_max(a.elapsed_time(b) / args.steps, dev)
        h2d = X.numel() * X.element_size() + W.numel() * W.element_size()
        d2h = qp.numel() * 4 + sc.numel() * 4 + zr.numel() * 4
        e2e = {"value": whole_job_value(weights, world, ms_e2e), "unit": UNIT, "ms_per_step": ms_e2e,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "path": "X from pinned host memory through gptq_hessian_accumulate_host "
                       "(chunked copies overlapping the Gram products), W copied beside it, "
                       "codes/scales/zeros read back"}
        del Xh, ws_h

    # ---- CPU oracle baseline (rank 0, N = 1 only) ---------------------------------------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        Xs = X[:2048].float().cpu().numpy()
        Wn = W.float().cpu().numpy()
        est, det = oracle_sample(Xs, Wn, layer, bits, block, damp, tok_sample=2048,
                                 row_sample=64)
        cpu = {"value": weights / est, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
               "sample": (f"fp64 NumPy oracle: Hessian over the first {det['tok_sample']} "
                          f"tokens scaled x{n / det['tok_sample']:.0f}, full prepare at "
                          f"d_in={d}, sweep of {det['row_sample']} rows scaled "
                          f"x{m / det['row_sample']:.0f}"),
               "est_seconds_per_layer": est, "detail": det}

    if rank == 0:
        out = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded correlated activations and N(0, 0.02^2) weights)",
            "config": {"workload": wl.name, "d_out": m, "d_in": d, "n_tok": n, "bits": bits,
                       "block": block, "damp": damp, "x_dtype": act.dtype,
                       "w_dtype": layer.w_dtype,
                       "arith": "fp16 products exact, fp32 accumulation (Hessian); fp32 "
                                "elsewhere; 3xTF32-split operands for rank-K updates",
                       "l2": f"inputs exceed L2: X is {X.numel() * X.element_size() / 1e9:.2f}"
                             f" GB per step",
                       "parallelism": f"replicas x{world} (independent layers)"},
            "stages_ms": {"hessian": st_h, "prepare": st_p, "quantize": st_q},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": int(launches), "clocks": clk,
        }
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_recon(args, wl, layer, X, W, H, U, dm, qp, sc, zr, ws_p, ws_q, bits, block, damp,
              stream, dev, rank, world):
    """The consumer of the quantized layer, timed alone: per-row output error on X from the
    packed codes (one dequant-difference pass, one tcgen05 product, one reduction)."""
    import torch
    from post_weight_quantization_03_gb300 import gptq
    gptq.hessian(X, H, stream=stream)
    gptq.prepare(H, damp, U=U, dead_mask=dm, ws=ws_p, stream=stream)
    gptq.quantize(W, U, bits, block, dm, ws=ws_q, stream=stream, out=(qp, sc, zr, None))
    m, d, n = W.shape[0], W.shape[1], X.shape[0]
    ws_r = gptq.workspace(gptq.gptq_recon_error_workspace_bytes(gptq._dtype_code(X), m, d, n),
                          dev)
    for _ in range(max(3, args.warmup)):
        err = gptq.recon_error(X, W, qp, bits, sc, zr, ws=ws_r, stream=stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    time.sleep(0.4)
    launches0 = gptq.gptq_kernel_launches()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        err = gptq.recon_error(X, W, qp, bits, sc, zr, ws=ws_r, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    launches = gptq.gptq_kernel_launches() - launches0
    clk = clocks.stop()
    ms = a.elapsed_time(b) / args.steps
    flops = 2.0 * m * d * n
    peaks, peak_src = measured_peaks()
    peak_t = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    tf = flops / (ms / 1e3) / 1e12
    out = {
        "metric": "ms per layer & tokens/sec evaluating ||(W - W_hat) X^T||^2 per row from the "
                  "packed codes (4096x4096 int4)",
        "value": n / (ms / 1e3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": wl.name, "d_out": m, "d_in": d, "n_tok": n, "bits": bits,
                   "x_dtype": layer.act.dtype,
                   "l2": f"inputs exceed L2: X is {X.numel() * X.element_size() / 1e9:.2f} GB"},
        "total_error": float(err.double().sum().item()),
        "roofline": {"kernel": "recon_tc_kernel (tcgen05 kind::f16, (W - W_hat) X^T with the "
                               "row sums of squares in the epilogue)",
                     "bound": "tensor", "achieved": round(tf, 3), "peak": peak_t,
                     "unit": "TFLOP/s", "frac": round(tf / peak_t, 4), "traffic": None,
                     "algorithmic": f"2 d_out d_in N = {flops:.4e} flop per call (the whole "
                                    f"call timed: difference pass + product + reduction)",
                     "peak_source": f"{peak_src} bf16 sustained (fp16 tensor rate = bf16)"},
        "gpu_launches": int(launches), "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_obq(args, dev, rank, world):
    """OBQ (greedy order, per-row Schur downdates) and the fixed-order sweep on one narrow
    layer: time per call, and the output error of each (and of round-to-nearest) on X
    through the packed codes."""
    import torch
    from post_weight_quantization_03_gb300 import gptq
    from post_weight_quantization_03_gb300 import synthetic as S
    m, d, n, bits = 4096, 128, args.n_tok or 65536, 4
    act = S.ActivationSpec(d_in=d, n_tok=n, dtype="f16", n_dead=2, n_outlier=2, seed=77)
    X = S.activations(act, device=dev)
    W = S.weights(m, d, 0.02, "bf16", 78).to(dev)
    U, dm, _ = gptq.prepare(gptq.hessian(X), 0.01)
    ws_o = gptq.workspace(gptq.gptq_quantize_obq_workspace_bytes(m, d), dev)
    ws_g = gptq.workspace(gptq.gptq_quantize_workspace_bytes(m, d, bits, 128), dev)

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            out = fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            out = fn()
        b.record()
        torch.cuda.synchronize()
        return out, a.elapsed_time(b) / args.steps

    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    time.sleep(0.4)
    launches0 = gptq.gptq_kernel_launches()
    obq, ms_obq = timed(lambda: gptq.quantize_obq(W, U, bits, dm, ws=ws_o))
    launches = (gptq.gptq_kernel_launches() - launches0) // (args.steps + max(3, args.warmup))
    clk = clocks.stop()
    gq, ms_gptq = timed(lambda: gptq.quantize(W, U, bits, 128, dm, ws=ws_g))

    def errors(X, U, dm):
        outs = (("obq", gptq.quantize_obq(W, U, bits, dm)),
                ("gptq", gptq.quantize(W, U, bits, 128, dm)),
                ("rtn", gptq.quantize(W, torch.eye(d, device=dev), bits, 128, dm)))
        return {k: float(gptq.recon_error(X, W, o[0], bits, o[1], o[2]).double().sum().item())
                for k, o in outs}

    errs = {"2_outlier_channels": errors(X, U, dm)}
    # the same layer on inputs without outlier channels
    X0 = S.activations(S.ActivationSpec(d_in=d, n_tok=n, dtype="f16", n_dead=2, n_outlier=0,
                                        seed=77), device=dev)
    U0, dm0, _ = gptq.prepare(gptq.hessian(X0), 0.01)
    errs["no_outlier_channels"] = errors(X0, U0, dm0)
    peaks, _ = measured_peaks()
    sm_mhz = float(peaks.get("sm_max_mhz", 2070.0))
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    peak_alu = nsm * 128 * 2 * sm_mhz * 1e6 / 1e12      # fp32 FMA lanes x 2 flop x clock
    flops = 2.0 * m * sum(f * f for f in range(1, d + 1))  # Schur downdates of the free block
    tf = flops / (ms_obq / 1e3) / 1e12
    out = {
        "metric": "ms per layer: OBQ greedy order vs fixed-order GPTQ (4096 x 128 int4)",
        "value": m * d / (ms_obq / 1e3), "unit": "weights/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_obq,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "obq4096x128", "d_out": m, "d_in": d, "n_tok": n, "bits": bits,
                   "x_dtype": "f16", "w_dtype": "bf16"},
        "gptq_fixed_order_ms": ms_gptq,
        "output_error_on_X": errs,
        "roofline": {"kernel": "obq_kernel (one CTA per row, per-row inverse Hessian in shared "
                               "memory)", "bound": "alu", "achieved": round(tf, 4),
                     "peak": round(peak_alu, 2), "unit": "TFLOP/s",
                     "frac": round(tf / peak_alu, 4), "traffic": None,
                     "algorithmic": f"2 d_out sum_f f^2 = {flops:.4e} flop (rank-one downdates "
                                    f"of the shrinking free block)",
                     "peak_source": f"derived: {nsm} SMs x 128 fp32 lanes x 2 flop x "
                                    f"{sm_mhz:.0f} MHz"},
        "gpu_launches": int(launches), "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_block(args, wl, dev, rank, world):
    """A block of layers grouped by shared inputs (one Hessian and one prepare per group,
    one shared sweep per group and bit width): overlapped producer/consumer schedule timed
    over K steps, then the same work serialized with per-stage events."""
    import torch
    from post_weight_quantization_03_gb300 import gptq
    from post_weight_quantization_03_gb300 import synthetic as S
    from dataclasses import replace

    groups = {}
    for layer in wl.layers:
        groups.setdefault(layer.act, []).append(layer)
    G = []
    for act, layers in groups.items():
        a = replace(act, n_tok=args.n_tok) if args.n_tok else act
        G.append((S.activations(a, device=dev), [S.layer_weights(l, dev) for l in layers]))
    torch.cuda.synchronize()
    block = args.block or wl.block
    weights = sum(l.d_out * l.act.d_in for l in wl.layers) * len(wl.bits)

    def step(overlap, ev=None):
        return gptq.quantize_block(G, bits=wl.bits, block=block, damp=wl.damp, overlap=overlap,
                                   stage_events=ev)

    for _ in range(max(3, args.warmup)):
        step(True)
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    time.sleep(0.4)
    launches0 = gptq.gptq_kernel_launches()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        step(True)
    b.record()
    torch.cuda.synchronize()
    launches = gptq.gptq_kernel_launches() - launches0
    clk = clocks.stop()
    ms_step = a.elapsed_time(b) / args.steps
    # the same work serialized on one stream, per stage
    evs = []
    a.record()
    step(False, evs)
    b.record()
    torch.cuda.synchronize()
    ms_serial = a.elapsed_time(b)
    stages = {}
    for name, e0, e1 in evs:
        stages[name] = stages.get(name, 0.0) + e0.elapsed_time(e1)
    peaks, peak_src = measured_peaks()
    h_flops = float(sum(x.shape[1] * (x.shape[1] + 1) * x.shape[0] for x, _ in G))
    h_tf = h_flops / (stages["hessian"] / 1e3) / 1e12
    peak_t = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    out = {
        "metric": "ms per block & weights quantized/sec (7B-shaped block, 3- and 4-bit GPTQ)",
        "value": weights / (ms_step / 1e3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "groups": [[l.name for l in ls] for ls in groups.values()],
                   "d_in": [x.shape[1] for x, _ in G], "n_tok": [x.shape[0] for x, _ in G],
                   "bits": list(wl.bits), "block": block, "damp": wl.damp,
                   "schedule": "each group's Hessian (one call) on a low-priority producer "
                               "stream ahead of prepare + shared sweeps on a high-priority "
                               "consumer stream"},
        "serial_ms": ms_serial, "stages_ms_serial": stages,
        "roofline": {"kernel": "hessian (all groups, serialized pass)", "bound": "tensor",
                     "achieved": round(h_tf, 3), "peak": peak_t, "unit": "TFLOP/s",
                     "frac": round(h_tf / peak_t, 4), "traffic": None,
                     "algorithmic": f"sum d(d+1)N = {h_flops:.4e} flop",
                     "peak_source": f"{peak_src} bf16 sustained"},
        "gpu_launches": int(launches), "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_reference(args, rank, world):
    """The oracle on the host cores, each step a bounded sample scaled to the full layer."""
    if rank != 0:
        return
    import numpy as np
    import torch

    from post_weight_quantization_03_gb300 import synthetic as S

    wl = S.WORKLOADS[args.workload]
    if args.obq:
        return run_obq(args, dev, rank, world)
    if len(wl.layers) > 1:
        return run_block(args, wl, dev, rank, world)
    layer = wl.layers[0]
    bits, block, damp = wl.bits[-1], args.block or wl.block, wl.damp
    m, d, n = layer.d_out, layer.act.d_in, layer.act.n_tok
    X = S.activations(layer.act, device="cpu", n_tok=2048).float().numpy()
    W = S.layer_weights(layer).float().numpy()
    total = args.steps + args.warmup
    rows = 64 if total <= 15 else 32
    times = []
    det = None
    for i in range(total):
        est, det = oracle_sample(X, W, layer, bits, block, damp, tok_sample=2048,
                                 row_sample=rows)
        if i >= args.warmup:
            times.append(est)
    sec = statistics.mean(times)
    value = m * d / sec
    sample = (f"fp64 NumPy oracle per step: Hessian over 2048 tokens scaled x{n // 2048}, "
              f"full prepare at d_in={d}, sweep of {rows} rows scaled x{m // rows}")
    out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "impl": "reference",
           "config": {"workload": wl.name, "d_out": m, "d_in": d, "n_tok": n, "bits": bits,
                      "block": block, "damp": damp},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": host_cores(),
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0},
           "detail": det}
    _ = (np, torch)
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
